// decode.cuh -- paged decode attention kernels (sm_103a).
//
// What is computed ("04 - Hacia PagedAttention (vista previa)", section "La idea de
// PagedAttention", step 5; "Lo que deberias llevarte de la Fase 22 sobre la Fase 27", item 2):
// for each sequence s and query head h (KV head g = h / G), softmax attention of the single
// query row over the first ctx_s logical positions, whose K/V rows are gathered through the
// sequence's block table. Paging only changes where rows live, so the result is dense
// attention; the extra cost is the table walk, a few bytes per 16-token block.
//
// How (GB300 design; the pages give no kernel):
//  * grid = (partition p, KV head g, sequence s). A partition is `bpp` consecutive table
//    entries; CTAs whose partition starts past the sequence's last block exit at once, so the
//    grid can be sized from the host-known table width without reading lengths on the host.
//  * The G query heads sharing KV head g are packed into one CTA: each K/V block is read from
//    HBM once and used for all G rows.
//  * Every warp streams its own share of the partition's blocks (interleaved) through a private
//    ring of ST shared-memory stages. One lane issues two 1-D bulk TMA copies per block (the K
//    and V chunks, each 16*D contiguous elements thanks to the [block][head][16][D] pool layout)
//    that complete on the stage's mbarrier; the warp waits on the barrier (bounded), computes,
//    and refills the stage. No CTA-wide barrier sits in the streaming loop.
//  * Lanes own 16-byte column chunks of a row (conflict-free shared-memory reads). QK^T partial
//    dot products are summed across the lanes of a row with a halving transpose-reduce; the
//    per-block softmax runs on 16 logits per row; PV accumulates in fp32 registers.
//  * Online softmax in base 2 (scale*log2(e) folded into q, exp2f), running max and sum per
//    row; masked positions are removed by selection, never by multiplying with zero, so NaN
//    in unused rows cannot leak into the result.
//  * At the end the warps' states are merged in shared memory. A sequence with a single
//    partition writes its final row directly; otherwise the CTA writes an unnormalised partial
//    (o, max, sum) to the workspace, and the CTA that finishes last among the sequence's
//    partitions (an arrival counter per sequence and KV head) merges them (log-sum-exp combine)
//    inside the same kernel -- no second launch.
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {

template <typename T, int D>
struct RowGeom {
    static constexpr int VEC = Vec16<T>::N;          // elements per 16-byte chunk
    static constexpr int NCH = D / VEC;              // chunks per row
    static constexpr int LPR = NCH < 32 ? NCH : 32;  // lanes per row
    static constexpr int RPP = 32 / LPR;             // rows a warp covers per pass
    static constexpr int CPL = NCH / LPR;            // chunks per lane per row
    static constexpr int TPL = kBlock / RPP;         // tokens per lane per block
    static constexpr int CHUNK = kBlock * D;         // elements of one K (or V) block chunk
    static_assert(NCH >= 2 && (NCH & (NCH - 1)) == 0, "head_dim must give a power-of-two chunk count");
    static_assert(TPL >= 4 && TPL % 4 == 0, "tokens per lane must be a multiple of 4");
};

// Warps per CTA and pipeline stages per warp for one instantiation.
template <typename T, int D, int G>
struct DecodeTuning {
    static constexpr int NW = 4;
    static constexpr int STAGE_BYTES = 2 * kBlock * D * (int)sizeof(T);
    static constexpr int ST_RAW = (96 * 1024) / (NW * STAGE_BYTES);
    static constexpr int ST = NW * 2 * STAGE_BYTES > 200 * 1024 ? 1 : (ST_RAW < 2 ? 2 : (ST_RAW > 4 ? 4 : ST_RAW));
};

// The walk of step a1: the physical block holding logical block `blk` of sequence s (the table entry;
// a dense cache's identity walk returns blk itself) ...
__device__ __forceinline__ int walk_entry(const DecodeArgs& a, int s, int blk) {
    return a.dense ? blk : a.tables[(size_t)s * a.max_blocks + blk];
}
// ... and the index of its 16-row chunk of KV head g in the layer seen as [chunks][16][D]: a paged
// pool stores [block][head], a dense cache [sequence][head][block].
__device__ __forceinline__ long long chunk_index(const DecodeArgs& a, int s, int g, int phys) {
    return a.dense ? ((long long)s * a.n_kv + g) * a.max_blocks + phys : (long long)phys * a.n_kv + g;
}

constexpr int kMergeChunk = 32;  // partitions whose weights are staged in shared memory at a time
constexpr int kMergeLoads = 64;  // partial-output loads a merging thread keeps in flight at once

// Shared-memory floats the split-K merge needs (flag, row maxima, row sums, one chunk of weights).
template <int G>
struct MergeScratch {
    static constexpr size_t BYTES = (4 + 2 * G + G * kMergeChunk) * sizeof(float);
};

template <typename T, int D, int G, int NW, int ST>
struct DecodeSmem {
    using Geo = RowGeom<T, D>;
    static constexpr size_t STAGES = (size_t)NW * ST * 2 * Geo::CHUNK * sizeof(T);
    static constexpr size_t BARS = STAGES;                                 // uint64 [NW][ST]
    static constexpr size_t PHYS = BARS + (size_t)NW * ST * 8;             // int [NW][ST]
    static constexpr size_t TAB = PHYS + (size_t)NW * ST * 4;              // int [NW][kMaxBpp/NW]: block ids
    static constexpr size_t ZBUF = (TAB + (size_t)kMaxBpp * 4 + 15) / 16 * 16;  // float [NW][G*16]
    static constexpr size_t PBUF = ZBUF + (size_t)NW * G * kBlock * 4;    // float [NW][G*16]
    static constexpr size_t ML = PBUF + (size_t)NW * G * kBlock * 4;      // float [NW][G][2]
    static constexpr size_t TOTAL = ML + (size_t)NW * G * 2 * 4;
    static constexpr size_t MERGE = ((size_t)NW * G * D * 4 + 15) / 16 * 16;  // merge scratch, after the combine buffer
    static_assert(MERGE + MergeScratch<G>::BYTES <= STAGES, "combine buffer and merge scratch must fit in the stage area");
};

// Split-K epilogue of the CTA (s, g, p) of a sequence with np > 1 partitions, after the CTA has
// stored its unnormalised partial (o, max, sum) for its G query rows. The CTA that arrives last at
// the (s, g) counter merges the np partials of every row -- o = sum_p o_p 2^(m_p - M) / sum_p l_p
// 2^(m_p - M), M = max_p m_p -- and writes the output rows.
// The counter holds (call tag << 24) | arrivals. A value carrying another tag (a finished call,
// a zeroed or never-initialised buffer, another geometry's partials) counts as zero arrivals, so
// the workspace needs no clearing; the merging CTA resets the counter to 0, so a replay of an
// identical launch also starts from zero. One thread per CTA publishes the CTA's writes (barrier,
// then fence, then the atomic) and the merging CTA reads the partials from L2 after a fence. The
// merge order is fixed, so the result does not depend on which CTA happens to finish last.
template <typename T, int D, int G, int NT>
__device__ __forceinline__ void splitk_merge_if_last(const DecodeArgs& a, int s, int g, int np, float* scratch) {
    static_assert(NT % 32 == 0, "whole warps");
    constexpr int NWARP = NT / 32;
    constexpr int PER = (G * D + NT - 1) / NT;
    constexpr int MQ = kMergeLoads / PER < 2 ? 2 : (kMergeLoads / PER > 16 ? 16 : kMergeLoads / PER);
    int* flag = reinterpret_cast<int*>(scratch);
    float* sM = scratch + 4;  // [G]
    float* sL = sM + G;       // [G]
    float* sW = sL + G;       // [G][kMergeChunk]
    unsigned long long* cnt = a.counters + (size_t)s * a.n_kv + g;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(cnt);
        unsigned long long next;
        while (true) {
            next = ((cur >> 24) == a.call_tag) ? cur + 1 : ((a.call_tag << 24) | 1ull);
            const unsigned long long prev = atomicCAS(cnt, cur, next);
            if (prev == cur) break;
            cur = prev;
        }
        *flag = (next & 0xffffffull) == (unsigned long long)np;
        __threadfence();
    }
    __syncthreads();
    if (!*flag) return;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const size_t row0 = (size_t)s * a.n_q + (size_t)g * G;
    for (int r = warp; r < G; r += NWARP) {
        const float* ml = a.part_ml + (row0 + r) * a.n_parts * 2;
        float m = -INFINITY;
        for (int q = lane; q < np; q += 32) m = fmaxf(m, __ldcg(ml + 2 * q));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) {
            sM[r] = m;
            sL[r] = 0.f;
        }
    }
    float O[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) O[k] = 0.f;
    for (int c0 = 0; c0 < np; c0 += kMergeChunk) {
        __syncthreads();  // maxima visible; the previous chunk's weights consumed
        for (int r = warp; r < G; r += NWARP) {
            const float* ml = a.part_ml + (row0 + r) * a.n_parts * 2;
            const int q = c0 + lane;
            float w = 0.f, lw = 0.f;
            if (q < np) {
                const float m = __ldcg(ml + 2 * q);
                if (m != -INFINITY) {
                    w = exp2f(m - sM[r]);
                    lw = __ldcg(ml + 2 * q + 1) * w;
                }
            }
            sW[r * kMergeChunk + lane] = w;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
            if (lane == 0) sL[r] += lw;
        }
        __syncthreads();
        const int nq = min(kMergeChunk, np - c0);
        // The partials are read in groups of MQ: every thread first issues the MQ x PER loads of a
        // group (all independent, all in flight at once), then folds them in partition order. The
        // merging CTA ends the (sequence, KV head) -- often the whole launch -- so its reads must
        // not wait on each other one L2 round trip at a time. Same FMA order as a plain loop.
        for (int q0 = 0; q0 < nq; q0 += MQ) {
            const int mq = min(MQ, nq - q0);
            float v[PER][MQ];
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int idx = threadIdx.x + k * NT;
                const int r = idx / D;
                const float* po = a.part_o + ((row0 + r) * a.n_parts + c0 + q0) * D + idx % D;
#pragma unroll
                for (int u = 0; u < MQ; ++u)
                    v[k][u] = (idx < G * D && u < mq) ? __ldcg(po + (size_t)u * D) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int idx = threadIdx.x + k * NT;
                if (idx < G * D) {
                    const float* w = sW + (idx / D) * kMergeChunk + q0;
#pragma unroll
                    for (int u = 0; u < MQ; ++u)
                        if (u < mq) O[k] = fmaf(w[u], v[k][u], O[k]);
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int idx = threadIdx.x + k * NT;
        if (idx < G * D) {
            const int r = idx / D;
            const int d = idx % D;
            const float L = sL[r];
            reinterpret_cast<T*>(a.out)[(row0 + r) * D + d] = from_float<T>(L > 0.f ? O[k] / L : 0.f);
        }
    }
    if (threadIdx.x == 0) *cnt = 0ull;
}

// Fused KV append (decode step): the CTA whose partition holds the sequence's last block writes the
// new token's K and V rows of its KV head g at position ctx-1 -- slot table[nb-1]*16 + (ctx-1)%16,
// the slot the block manager reserved -- before any of its TMA loads, then fences the generic
// writes against the asynchronous proxy. No other CTA reads that block. An out-of-range block id
// writes nothing (the attention path skips and flags that block).
template <typename T, int D, int NT>
__device__ __forceinline__ void fused_append(const DecodeArgs& a, int s, int g, int p, int ctx, int nb) {
    if (a.k_new == nullptr || p != (nb - 1) / a.bpp) return;
    const int phys = walk_entry(a, s, nb - 1);
    if ((unsigned)phys >= (unsigned)a.num_blocks) return;
    constexpr int NCH = D * (int)sizeof(T) / 16;  // 16-byte chunks per row
    const size_t src_row = ((size_t)s * a.n_kv + g) * D;
    const size_t dst_row = ((size_t)chunk_index(a, s, g, phys) * kBlock + (ctx - 1) % kBlock) * D;
    for (int i = threadIdx.x; i < 2 * NCH; i += NT) {
        const bool is_v = i >= NCH;
        const int c = is_v ? i - NCH : i;
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(is_v ? a.v_new : a.k_new) + src_row) + c;
        uint4* dst = reinterpret_cast<uint4*>(const_cast<T*>(reinterpret_cast<const T*>(is_v ? a.v_layer : a.k_layer)) + dst_row) + c;
        *dst = __ldg(src);
    }
    fence_proxy_async_global();
}

template <typename T, int D, int G, int NW, int ST>
__global__ void __launch_bounds__(NW * 32) paged_decode_kernel(const DecodeArgs a) {
    using Geo = RowGeom<T, D>;
    using V = Vec16<T>;
    using S = DecodeSmem<T, D, G, NW, ST>;
    constexpr int VEC = Geo::VEC, LPR = Geo::LPR, RPP = Geo::RPP, CPL = Geo::CPL, TPL = Geo::TPL;
    constexpr int CHUNK = Geo::CHUNK;
    constexpr int TB = (G * TPL <= 32) ? TPL : 32 / G;  // tokens per QK sub-batch
    constexpr int NV = G * TB;                          // partial sums per lane per sub-batch
    constexpr int NF = NV >= LPR ? NV / LPR : 1;        // complete sums per lane after reduction
    constexpr int KS = (G * kBlock + 31) / 32;          // softmax entries per lane
    constexpr uint32_t CHUNK_BYTES = CHUNK * sizeof(T);

    extern __shared__ __align__(128) unsigned char smem[];
    T* stage = reinterpret_cast<T*>(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BARS);
    int* s_phys = reinterpret_cast<int*>(smem + S::PHYS);
    float* s_zall = reinterpret_cast<float*>(smem + S::ZBUF);
    float* s_pall = reinterpret_cast<float*>(smem + S::PBUF);
    float* s_ml = reinterpret_cast<float*>(smem + S::ML);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int p = blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;

    int ctx = a.lens[s];
    const int cap = a.max_blocks * kBlock;
    if (ctx < 0 || ctx > cap) {
        if (p == 0 && threadIdx.x == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_CONTEXT_LEN);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int nb = (ctx + kBlock - 1) / kBlock;
    const int b0 = p * a.bpp;
    if (b0 >= nb) {
        if (p == 0) {  // empty context: the attention sum is empty, the row is zero
            T* o = reinterpret_cast<T*>(a.out) + ((size_t)s * a.n_q + (size_t)g * G) * D;
            for (int i = threadIdx.x; i < G * D; i += NW * 32) o[i] = from_float<T>(0.f);
        }
        return;
    }
    const int nblk = min(a.bpp, nb - b0);
    const bool single = nb <= a.bpp;
    fused_append<T, D, NW * 32>(a, s, g, p, ctx, nb);

    if (threadIdx.x < NW * ST) mbar_init(&bars[threadIdx.x], 1);
    fence_mbar_init();
    __syncthreads();

    uint64_t* wbars = bars + warp * ST;
    int* wphys = s_phys + warp * ST;
    T* wstage = stage + (size_t)warp * ST * 2 * CHUNK;
    float* s_z = s_zall + warp * G * kBlock;
    float* s_p = s_pall + warp * G * kBlock;

    static_assert(kMaxBpp % NW == 0, "each warp stages kMaxBpp / NW table entries");
    int* wtab = reinterpret_cast<int*>(smem + S::TAB) + warp * (kMaxBpp / NW);
    const T* kbase = reinterpret_cast<const T*>(a.k_layer);
    const T* vbase = reinterpret_cast<const T*>(a.v_layer);
    const int nk = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;  // blocks of this warp
    const uint64_t policy = l2_evict_first_policy();

    // lane 0: start the copies of this warp's k-th block into stage k % ST
    auto issue = [&](int k) {
        const int st = k % ST;
        const int phys = wtab[k];
        const bool ok = (unsigned)phys < (unsigned)a.num_blocks;
        wphys[st] = ok ? phys : -1;
        if (ok) {
            const size_t off = (size_t)chunk_index(a, s, g, phys) * CHUNK;
            T* dst = wstage + (size_t)st * 2 * CHUNK;
            mbar_arrive_expect_tx(&wbars[st], 2 * CHUNK_BYTES);
            bulk_copy_g2s(dst, kbase + off, CHUNK_BYTES, &wbars[st], policy);
            bulk_copy_g2s(dst + CHUNK, vbase + off, CHUNK_BYTES, &wbars[st], policy);
        } else {
            atomicOr(a.status, (unsigned)PKV_DEV_BAD_BLOCK_ID);
            mbar_arrive(&wbars[st]);  // completes the phase with nothing copied: rows are masked
        }
    };
    // this warp's table entries (blocks warp, warp+NW, ...) staged once, so issuing a copy never
    // waits on a global read of the table
    for (int k = lane; k < nk; k += 32) wtab[k] = walk_entry(a, s, b0 + warp + k * NW);
    __syncwarp();
    if (lane == 0) {
        for (int k = 0; k < ST && k < nk; ++k) issue(k);
    }

    // this lane's place in a row: row group rg (tokens rg, rg+RPP, ...), column chunk cl
    const int rg = lane / LPR;
    const int cl = lane % LPR;

    float qr[G][CPL][VEC];
#pragma unroll
    for (int r = 0; r < G; ++r) {
        const T* qrow = reinterpret_cast<const T*>(a.q) + ((size_t)s * a.n_q + (size_t)g * G + r) * D;
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) {
            const uint4 u = *reinterpret_cast<const uint4*>(qrow + (cl + cc * LPR) * VEC);
            V::to_float(u, qr[r][cc]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qr[r][cc][e] *= a.scale_log2;
        }
    }

    float acc[G][CPL][VEC];
#pragma unroll
    for (int r = 0; r < G; ++r)
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[r][cc][e] = 0.f;
    float m_run[G];
#pragma unroll
    for (int r = 0; r < G; ++r) m_run[r] = -INFINITY;
    float lsum[KS];
#pragma unroll
    for (int x = 0; x < KS; ++x) lsum[x] = 0.f;

    for (int k = 0; k < nk; ++k) {
        const int st = k % ST;
        if (!mbar_wait_bounded(&wbars[st], (uint32_t)(k / ST) & 1u)) {
            if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
            for (int kk = k + 1; kk < k + ST && kk < nk; ++kk)  // let in-flight copies land
                mbar_wait_bounded(&wbars[kk % ST], (uint32_t)(kk / ST) & 1u);
            break;
        }
        const int jb = (b0 + warp + k * NW) * kBlock;  // logical position of the block's row 0
        const int nvalid = wphys[st] >= 0 ? min(kBlock, ctx - jb) : 0;
        const T* sK = wstage + (size_t)st * 2 * CHUNK;
        const T* sV = sK + CHUNK;

        // ---- logits z[r][j] = q_r . K_j (base-2 scaled), masked to -inf past the context ----
#pragma unroll
        for (int t0 = 0; t0 < TPL; t0 += TB) {
            float part[NV];
#pragma unroll
            for (int x = 0; x < NV; ++x) part[x] = 0.f;
#pragma unroll
            for (int tb = 0; tb < TB; ++tb) {
                const int j = rg + RPP * (t0 + tb);
#pragma unroll
                for (int cc = 0; cc < CPL; ++cc) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sK + j * D + (cl + cc * LPR) * VEC);
                    float kf[VEC];
                    V::to_float(u, kf);
#pragma unroll
                    for (int r = 0; r < G; ++r)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) part[r * TB + tb] = fmaf(qr[r][cc][e], kf[e], part[r * TB + tb]);
                }
            }
            HalvingReduce<NV, LPR / 2>::run(part, lane);
            const int base = (cl * NV) / LPR;
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                const int v = base + f;
                const int r = v / TB;
                const int j = rg + RPP * (t0 + v % TB);
                s_z[r * kBlock + j] = (j < nvalid) ? part[f] : -INFINITY;
            }
        }
        __syncwarp();

        // ---- per-block softmax update: entry e = lane + 32*x is (row e/16, token e%16) ----
        float zz[KS], mx[KS];
#pragma unroll
        for (int x = 0; x < KS; ++x) {
            const int e = lane + 32 * x;
            zz[x] = (e < G * kBlock) ? s_z[e] : -INFINITY;
            mx[x] = zz[x];
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) mx[x] = fmaxf(mx[x], __shfl_xor_sync(0xffffffffu, mx[x], o));
        }
        float alpha[G];
#pragma unroll
        for (int r = 0; r < G; ++r) {
            const float mb = __shfl_sync(0xffffffffu, mx[r / 2], (r % 2) * 16);
            const float mnew = fmaxf(m_run[r], mb);
            alpha[r] = (m_run[r] == -INFINITY) ? 0.f : exp2f(m_run[r] - mnew);
            m_run[r] = mnew;
        }
#pragma unroll
        for (int x = 0; x < KS; ++x) {
            const int e = lane + 32 * x;
            const int row = e / kBlock;
            float mr = -INFINITY, al = 0.f;
#pragma unroll
            for (int r = 0; r < G; ++r) {
                if (r == row) {
                    mr = m_run[r];
                    al = alpha[r];
                }
            }
            const float pz = (zz[x] == -INFINITY) ? 0.f : exp2f(zz[x] - mr);
            lsum[x] = lsum[x] * al + pz;
            if (e < G * kBlock) {
                const int j = e % kBlock;
                s_p[row * kBlock + (j % RPP) * TPL + j / RPP] = pz;
            }
        }
        __syncwarp();

        // ---- acc_r = alpha_r * acc_r + sum_j p_rj V_j over this lane's tokens ----
#pragma unroll
        for (int r = 0; r < G; ++r)
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[r][cc][e] *= alpha[r];
        const bool full = nvalid == kBlock;
#pragma unroll
        for (int t4 = 0; t4 < TPL; t4 += 4) {
            float4 pr[G];
#pragma unroll
            for (int r = 0; r < G; ++r) pr[r] = *reinterpret_cast<const float4*>(s_p + r * kBlock + rg * TPL + t4);
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                const int j = rg + RPP * (t4 + tt);
                const bool keep = full || j < nvalid;
#pragma unroll
                for (int cc = 0; cc < CPL; ++cc) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sV + j * D + (cl + cc * LPR) * VEC);
                    float vf[VEC];
                    V::to_float(u, vf);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) vf[e] = keep ? vf[e] : 0.f;
#pragma unroll
                    for (int r = 0; r < G; ++r) {
                        const float pj = tt == 0 ? pr[r].x : tt == 1 ? pr[r].y : tt == 2 ? pr[r].z : pr[r].w;
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[r][cc][e] = fmaf(pj, vf[e], acc[r][cc][e]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && k + ST < nk) {
            fence_proxy_async_smem();
            issue(k + ST);
        }
    }

    // ---- finish this warp: row sums, then fold the row groups' partial accumulators ----
#pragma unroll
    for (int x = 0; x < KS; ++x)
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) lsum[x] += __shfl_xor_sync(0xffffffffu, lsum[x], o);
    float l_run[G];
#pragma unroll
    for (int r = 0; r < G; ++r) l_run[r] = __shfl_sync(0xffffffffu, lsum[r / 2], (r % 2) * 16);
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
        for (int r = 0; r < G; ++r)
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[r][cc][e] += __shfl_xor_sync(0xffffffffu, acc[r][cc][e], o);

    // ---- merge the warps (the stage area is free once every warp has left its loop) ----
    __syncthreads();
    float* s_acc = reinterpret_cast<float*>(smem);  // [NW][G][D]
    if (lane < LPR) {
#pragma unroll
        for (int r = 0; r < G; ++r)
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) {
                float* dst = s_acc + ((size_t)warp * G + r) * D + (cl + cc * LPR) * VEC;
#pragma unroll
                for (int e = 0; e < VEC; e += 4)
                    *reinterpret_cast<float4*>(dst + e) =
                        make_float4(acc[r][cc][e], acc[r][cc][e + 1], acc[r][cc][e + 2], acc[r][cc][e + 3]);
            }
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < G; ++r) {
            s_ml[(warp * G + r) * 2] = m_run[r];
            s_ml[(warp * G + r) * 2 + 1] = l_run[r];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int r = idx / D;
        const int d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, s_ml[(w * G + r) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float mw = s_ml[(w * G + r) * 2];
            if (mw != -INFINITY) {
                const float sc = exp2f(mw - M);
                L = fmaf(s_ml[(w * G + r) * 2 + 1], sc, L);
                O = fmaf(s_acc[((size_t)w * G + r) * D + d], sc, O);
            }
        }
        const size_t row = (size_t)s * a.n_q + (size_t)g * G + r;
        if (single) {
            reinterpret_cast<T*>(a.out)[row * D + d] = from_float<T>(L > 0.f ? O / L : 0.f);
        } else {
            const size_t prow = row * a.n_parts + p;
            a.part_o[prow * D + d] = O;
            if (d == 0) {
                a.part_ml[prow * 2] = M;
                a.part_ml[prow * 2 + 1] = L;
            }
        }
    }
    if (!single)
        splitk_merge_if_last<T, D, G, NW * 32>(a, s, g, (nb + a.bpp - 1) / a.bpp,
                                               reinterpret_cast<float*>(smem + S::MERGE));
}

// Lets `kern` use `smem` bytes of dynamic shared memory on the current device (once per device; a
// benign race, the call is idempotent).
template <typename K>
cudaError_t allow_dynamic_smem(K kern, size_t smem, unsigned long long* done) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && !(__atomic_load_n(done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        __atomic_fetch_or(done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    return cudaSuccess;
}

template <typename T, int D, int G>
struct DecodeKernel {
    static constexpr int NW = DecodeTuning<T, D, G>::NW;
    static constexpr int ST = DecodeTuning<T, D, G>::ST;
    static constexpr size_t smem = DecodeSmem<T, D, G, NW, ST>::TOTAL;
    static unsigned long long attr_done;
    static cudaError_t prepare() { return allow_dynamic_smem(paged_decode_kernel<T, D, G, NW, ST>, smem, &attr_done); }
    // CTAs of this kernel one SM holds at once (shared memory, registers, threads)
    static cudaError_t ctas_per_sm(int* out) {
        cudaError_t err = prepare();
        if (err != cudaSuccess) return err;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, paged_decode_kernel<T, D, G, NW, ST>, NW * 32, smem);
    }
};
template <typename T, int D, int G>
unsigned long long DecodeKernel<T, D, G>::attr_done = 0;

template <typename T, int D, int G>
cudaError_t launch_decode_tpl(const DecodeArgs& a, cudaStream_t stream, int* n_launches) {
    using K = DecodeKernel<T, D, G>;
    constexpr int NW = K::NW;
    constexpr size_t smem = K::smem;
    auto kern = paged_decode_kernel<T, D, G, NW, K::ST>;
    cudaError_t err = K::prepare();
    if (err != cudaSuccess) return err;
    dim3 grid(a.n_parts, a.n_kv, a.n_seqs);
    kern<<<grid, NW * 32, smem, stream>>>(a);
    if (n_launches) *n_launches = 1;
    return cudaGetLastError();
}

template <typename T>
cudaError_t decode_ctas_per_sm_dtype(int head_dim, int group, int* out) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return DecodeKernel<T, DD, GG>::ctas_per_sm(out);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_decode_dtype(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return launch_decode_tpl<T, DD, GG>(a, stream, n);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
