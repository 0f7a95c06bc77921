// prefill_umma.cuh -- paged prefill / chunked prefill attention on the tcgen05 tensor cores (fp16 /
// bf16), accumulators in tensor memory.
//
// Same operation and masking rules as prefill_mma.cuh ("PagedAttention e continuous batching",
// "01 - Conceito", paragraph 5; "La idea de PagedAttention", step 5): chunk token i of sequence s
// sits at position c - n + i and attends to keys 0 .. that position through the block table.
//
// CTA = (128 query rows, KV head, sequence); rows = token x head-in-group (GQA rows packed, so each
// K/V tile serves all G heads). Seven warps:
//   warps 0-3  softmax: thread t owns query row t, which is TMEM lane t (a warp reaches only its
//              own 32 lanes); it reads its row of S, masks by selection, keeps the running max
//              and sum in registers, writes its row of P (storage type) into shared memory;
//   warps 4, 6 producers: walk the block table and move 64-key K tiles (warp 4) and V tiles
//              (warp 6) of four 16-token blocks into a ring of ST stages with TMA tensor copies
//              (128-byte swizzle); a K stage is released when S_j is done, a V stage when PV_j is;
//              warp 6 zeroes the V rows of skipped blocks and of the positions past the context;
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM buffers (128 x 64 fp32),
//              then O += P_j V_j into a TMEM accumulator (128 x D fp32), each followed by a
//              tcgen05.commit onto an mbarrier.
// S is double-buffered, so S_{j+1} runs on the tensor pipe while the softmax warps work on S_j.
// O is rescaled (read, multiplied, written back in TMEM) only when a row's running maximum grows
// by more than 8 (a factor 2^8 in the weights): P <= 2^8 stays exact enough in the storage type
// and the final division by the same running sum keeps the result the softmax's. The weights are
// 2^(s * scale * log2 e - m) from one FFMA and one ex2.approx each; the running sum adds them in
// fp32 before they are rounded to the storage type for the PV product.
// Each mbarrier serves one buffer, and no thread waits on a phase two completions old, so phase
// parities never alias. Every wait is bounded (PKV_DEV_WAIT_TIMEOUT).
#pragma once

#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "decode_mma.cuh"
#include "internal.h"
#include "prefill_mma.cuh"
#include "umma.cuh"

namespace pkv {

// 2^x with the ex2.approx.ftz instruction (2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D>
struct UmmaTuning {
    static constexpr int ST = D == 256 ? 2 : (D == 128 ? 3 : 4);  // K/V stages
    static constexpr int NP = D == 256 ? 1 : 2;                   // P buffers
    static constexpr uint32_t TMEM_COLS = (128 + D) <= 256 ? 256u : 512u;
};

template <int D, int ST, int NP>
struct UmmaSmem {
    static constexpr size_t QB = (size_t)128 * D * 2;   // Q [D/64][128 rows][128 B]
    static constexpr size_t KT = (size_t)64 * D * 2;    // K or V tile [D/64][64 keys][128 B]
    static constexpr size_t PB = (size_t)128 * 128;     // P [128 rows][64 keys x 2 B]
    static constexpr size_t Q = 0;
    static constexpr size_t KV = QB;                      // [ST][K tile, V tile]
    static constexpr size_t P = KV + (size_t)ST * 2 * KT;
    static constexpr size_t BARS = P + (size_t)NP * PB;
    // full_k[ST] full_v[ST] k_empty[ST] v_empty[ST] s_full[2] s_free[2] p_full[NP] p_free[NP] vtail
    static constexpr int NBARS = 4 * ST + 4 + 2 * NP + 1;
    static constexpr size_t TADDR = BARS + (size_t)NBARS * 8;  // TMEM base address
    static constexpr size_t TOTAL = TADDR + 16;
    static constexpr size_t ALLOC = TOTAL + 1024;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(224, 1)
    paged_prefill_umma_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v) {
    static_assert(128 % G == 0, "whole tokens per tile");
    using Tu = UmmaTuning<D>;
    constexpr int ST = Tu::ST;
    constexpr int NP = Tu::NP;
    using S = UmmaSmem<D, ST, NP>;
    using M = MmaType<T>;
    constexpr int ROWS = 128;
    constexpr int QT = ROWS / G;
    constexpr int PANELS = D / 64;
    constexpr uint32_t KT = (uint32_t)S::KT;
    constexpr uint32_t PANEL = 64 * 128;                // one 64-key panel of a K/V tile
    constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
    constexpr int NPV = D > 128 ? 128 : D;             // N of one PV instruction
    constexpr uint32_t IDESC_S = umma_idesc_f16(BF, 128, 64, false);
    constexpr uint32_t IDESC_PV = umma_idesc_f16(BF, 128, NPV, true);
    constexpr uint32_t S_COL = 0;                       // S buffers: columns [0, 128)
    constexpr uint32_t O_COL = 128;                     // O: columns [128, 128 + D)

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BARS);
    uint64_t* full_k = bars;
    uint64_t* full_v = full_k + ST;
    uint64_t* k_empty = full_v + ST;
    uint64_t* v_empty = k_empty + ST;
    uint64_t* s_full = v_empty + ST;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* p_free = p_full + NP;
    uint64_t* vtail = p_free + NP;
    uint32_t* taddr_s = reinterpret_cast<uint32_t*>(smem + S::TADDR);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + (uint32_t)S::Q;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = a.q_tiles - 1 - (int)blockIdx.x;  // tiles with the most keys start first
    const int g = blockIdx.y;
    const int s = blockIdx.z;

    const int q0 = a.q_start[s];
    const int q1 = a.q_start[s + 1];
    const int n_new = q1 - q0;
    const int ctx = a.lens[s];
    if (q0 < 0 || q1 > a.n_tokens || n_new < 0 || n_new > a.q_tiles * QT || ctx < n_new ||
        ctx > a.max_blocks * kBlock) {
        if (blockIdx.x == 0 && g == 0 && threadIdx.x == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_QUERY_RANGE);
        return;
    }
    const int t0 = tile * QT;
    if (t0 >= n_new) return;
    const int t_end = min(t0 + QT, n_new);
    const int pos0 = ctx - n_new + t0;
    const int pos_last = ctx - n_new + t_end - 1;
    const int n_tiles = pos_last / 64 + 1;
    const int nb = (ctx + kBlock - 1) / kBlock;
    const bool tail_tile = n_tiles * 64 > ctx;

    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full_k[i], 1);
            mbar_init(&full_v[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 128);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(&p_full[i], 128);
            mbar_init(&p_free[i], 1);
        }
        mbar_init(vtail, 32);
        fence_mbar_init();
    }
    // Q tile -> shared memory (128-byte swizzle, the layout tcgen05 reads); rows past the chunk are 0
    {
        const T* qg = reinterpret_cast<const T*>(a.q);
        for (int i = threadIdx.x; i < ROWS * (D / 8); i += 224) {
            const int r = i / (D / 8);
            const int ch = i % (D / 8);
            const int tt = r / G;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t0 + tt < n_new)
                v = *reinterpret_cast<const uint4*>(qg + ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + r % G) * D +
                                                    ch * 8);
            *reinterpret_cast<uint4*>(smem + S::Q + swzq<ROWS>(r, ch)) = v;
        }
        fence_proxy_async_smem();  // generic writes, read by the tensor core
    }
    if (warp == 5) tmem_alloc(taddr_s, Tu::TMEM_COLS);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = *taddr_s;

    if (warp == 4 || warp == 6) {
        // ===================== producers: warp 4 moves K tiles, warp 6 moves V tiles =====================
        // A K stage is released once S_j has been computed, a V stage once O += P_j V_j has: the next
        // K tile can land while the softmax of this one runs.
        const bool is_v = warp == 6;
        uint64_t* full = is_v ? full_v : full_k;
        uint64_t* empty = is_v ? v_empty : k_empty;
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % ST;
            if (j >= ST && !mbar_wait_bounded(&empty[st], (uint32_t)((j / ST) - 1) & 1u)) {
                if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
                break;
            }
            const int blk = j * 4 + lane;
            const bool inb = lane < 4 && blk < nb;
            const int phys = inb ? trow[blk] : -1;
            const bool ok = inb && (unsigned)phys < (unsigned)a.num_blocks;
            const unsigned okm = __ballot_sync(0xffffffffu, ok);
            const unsigned badm = __ballot_sync(0xffffffffu, inb && !ok);
            unsigned char* vst = smem + S::KV + (size_t)st * 2 * KT + KT;
            if (badm) {
                // skipped blocks: keys masked by the softmax, V rows zeroed (P = 0 there, 0 * NaN is not)
                if (!is_v && lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_BLOCK_ID);
                if (is_v) {
                    for (int b = 0; b < 4; ++b) {
                        if (!((badm >> b) & 1u)) continue;
                        for (int i = lane; i < PANELS * 128; i += 32) {  // 2 KiB per panel = 128 x 16 B
                            const int pn = i / 128;
                            reinterpret_cast<uint4*>(vst + (size_t)pn * PANEL + (size_t)b * 2048)[i % 128] =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)__popc(okm) * (uint32_t)(kBlock * D * 2));
            __syncwarp();
            if (ok) {
                const int row0 = (phys * a.n_kv + g) * kBlock;
                const uint32_t dst = sbase + (uint32_t)S::KV + (uint32_t)st * 2 * KT + (is_v ? KT : 0u) +
                                     (uint32_t)lane * 2048;
#pragma unroll
                for (int pn = 0; pn < PANELS; ++pn) tma_load_2d_keep(dst + pn * PANEL, tm, pn * 64, row0, &full[st]);
            }
            issued = j + 1;
            if (is_v && j == n_tiles - 1 && tail_tile) {
                if (!mbar_wait_bounded(&full_v[st], (uint32_t)(j / ST) & 1u)) {
                    if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
                    break;
                }
                const int r0 = ctx - j * 64;  // first key row past the context, 1 .. 63
                for (int i = lane; i < PANELS * (64 - r0) * 8; i += 32) {
                    const int pn = i / ((64 - r0) * 8);
                    const int rem = i % ((64 - r0) * 8);
                    reinterpret_cast<uint4*>(vst + (size_t)pn * PANEL + (size_t)(r0 + rem / 8) * 128)[rem % 8] =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                mbar_arrive(vtail);
            }
        }
        for (int j = max(0, issued - ST); j < issued; ++j)  // the copies of the last stages have landed
            mbar_wait_bounded(&full[j % ST], (uint32_t)(j / ST) & 1u);
    } else if (warp == 5) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            bool ok = true;
            auto issue_s = [&](int j) -> bool {
                const int st = j % ST;
                const int b = j & 1;
                if (!mbar_wait_bounded(&full_k[st], (uint32_t)(j / ST) & 1u)) return false;
                if (j >= 2 && !mbar_wait_bounded(&s_free[b], (uint32_t)((j >> 1) - 1) & 1u)) return false;
                tcgen05_after_sync();
                const uint32_t sK = sbase + (uint32_t)S::KV + (uint32_t)st * 2 * KT;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t ad = umma_desc_sw128(sQ + (uint32_t)(ks >> 2) * (ROWS * 128) + (uint32_t)(ks & 3) * 32,
                                                        16, 1024);
                    const uint64_t bd = umma_desc_sw128(sK + (uint32_t)(ks >> 2) * PANEL + (uint32_t)(ks & 3) * 32, 16, 1024);
                    umma_f16(tmem + S_COL + (uint32_t)b * 64, ad, bd, IDESC_S, ks > 0);
                }
                umma_commit(&s_full[b]);
                umma_commit(&k_empty[st]);  // the K stage may take tile j + ST once S_j is done
                return true;
            };
            ok = issue_s(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles && !issue_s(j + 1)) {
                    ok = false;
                    break;
                }
                const int pb = j % NP;
                const int st = j % ST;
                if (!mbar_wait_bounded(&p_full[pb], (uint32_t)(j / NP) & 1u) ||
                    !mbar_wait_bounded(&full_v[st], (uint32_t)(j / ST) & 1u) ||
                    (j == n_tiles - 1 && tail_tile && !mbar_wait_bounded(vtail, 0u))) {
                    ok = false;
                    break;
                }
                tcgen05_after_sync();
                const uint32_t sP = sbase + (uint32_t)S::P + (uint32_t)pb * (uint32_t)S::PB;
                const uint32_t sV = sbase + (uint32_t)S::KV + (uint32_t)st * 2 * KT + KT;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = umma_desc_sw128(sP + (uint32_t)kk * 32, 16, 1024);
#pragma unroll
                    for (int h = 0; h < D / NPV; ++h) {
                        const uint64_t bd = umma_desc_sw128(sV + (uint32_t)kk * 2048 + (uint32_t)h * (NPV / 64) * PANEL,
                                                            PANEL, 1024);
                        umma_f16(tmem + O_COL + (uint32_t)(h * NPV), ad, bd, IDESC_PV, j > 0 || kk > 0);
                    }
                }
                umma_commit(&p_free[pb]);
                umma_commit(&v_empty[st]);
            }
            if (!ok) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
            // every issued MMA has completed before TMEM is released (the last commit covers them all)
            const int last = n_tiles - 1;
            mbar_wait_bounded(&p_free[last % NP], (uint32_t)(last / NP) & 1u);
        }
        __syncwarp();
    } else {
        // ===================== softmax (warps 0-3): thread = query row = TMEM lane =====================
        const int row = threadIdx.x;
        const int tt = row / G;
        const bool live = t0 + tt < n_new;
        const int lim = min(pos0 + tt, ctx - 1);
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float sl = a.scale_log2;
        float m_used = -INFINITY;
        float l = 0.f;
        bool ok = true;
        unsigned char* prow_base = smem + S::P + (size_t)row * 128;
        // which of a tile's four blocks were loaded (a table entry out of range is skipped): read from
        // the table itself one tile ahead, so that no wait on a producer's barrier is needed here
        const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
        auto tile_mask = [&](int j) -> int {
            int m = 0;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const int blk = j * 4 + bb;
                if (blk < nb && (unsigned)__ldg(trow + blk) < (unsigned)a.num_blocks) m |= 1 << bb;
            }
            return m;
        };
        int okm_next = tile_mask(0);
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;
            const int pb = j % NP;
            const int okm = okm_next;
            if (j + 1 < n_tiles) okm_next = tile_mask(j + 1);
            if (!mbar_wait_bounded(&s_full[b], (uint32_t)(j >> 1) & 1u)) {
                ok = false;
                break;
            }
            tcgen05_after_sync();
            uint32_t sv[64];
            tmem_ld32(tmem + lane_base + S_COL + (uint32_t)b * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(tmem + lane_base + S_COL + (uint32_t)b * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_wait_ld();
            tcgen05_before_sync();
            mbar_arrive(&s_free[b]);  // the S buffer may take S_{j+2}
            const int key0 = j * 64;
            float sc[64];
            float mx8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mx8[c] = -INFINITY;
            if (key0 + 63 <= lim && okm == 0xF) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    sc[c] = __uint_as_float(sv[c]);
                    mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) {  // masking by selection: a masked score is -inf
                    const bool v = key0 + c <= lim && ((okm >> (c >> 4)) & 1);
                    sc[c] = v ? __uint_as_float(sv[c]) : -INFINITY;
                    mx8[c & 7] = fmaxf(mx8[c & 7], sc[c]);
                }
            }
            const float smax = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float mt = smax * sl;  // the tile's row maximum in base 2 (scale > 0)
            // running maximum: move it (and rescale O, l) only when it grows by more than 8
            const bool grow = mt > m_used + 8.f;
            const float m_new = grow ? mt : m_used;
            const float alpha = grow ? exp2f(m_used - m_new) : 1.f;  // 0 when m_used is -inf
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                // O holds P_0..P_{j-1} V: wait for the last PV, then scale this warp's 32 rows in TMEM
                if (!mbar_wait_bounded(&p_free[(j - 1) % NP], (uint32_t)((j - 1) / NP) & 1u)) {
                    ok = false;
                    break;
                }
                tcgen05_after_sync();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_base + O_COL + (uint32_t)c0, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                    tmem_st32(tmem + lane_base + O_COL + (uint32_t)c0, ov);
                }
                tmem_wait_st();
            }
            l *= alpha;
            m_used = m_new;
            // p = 2^(s * scale_log2 - m): one FFMA and one ex2 per score; a masked score (-inf) gives
            // exactly 0. While every score so far is masked m_used is -inf: subtract 0 instead.
            const float msub = m_used == -INFINITY ? 0.f : m_used;
            uint32_t pw[32];
            float ls[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) ls[c] = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2_approx(fmaf(sc[2 * c], sl, -msub));
                const float p1 = ex2_approx(fmaf(sc[2 * c + 1], sl, -msub));
                pw[c] = M::pack(p0, p1);
                ls[c & 7] += p0 + p1;
            }
            l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
            // P buffer pb is free once PV_{j-NP} has completed
            if (j >= NP && !mbar_wait_bounded(&p_free[pb], (uint32_t)((j / NP) - 1) & 1u)) {
                ok = false;
                break;
            }
            unsigned char* prow = prow_base + (size_t)pb * S::PB;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
                    make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
            fence_proxy_async_smem();
            tcgen05_before_sync();
            mbar_arrive(&p_full[pb]);
        }
        if (ok) {
            const int last = n_tiles - 1;
            if (!mbar_wait_bounded(&p_free[last % NP], (uint32_t)(last / NP) & 1u)) ok = false;
        }
        if (!ok) {
            if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
        } else {
            tcgen05_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T* orow = reinterpret_cast<T*>(a.out) + ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + row % G) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32(tmem + lane_base + O_COL + (uint32_t)c0, ov);
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    w[c] = M::pack(__uint_as_float(ov[2 * c]) * inv, __uint_as_float(ov[2 * c + 1]) * inv);
                if (live) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(orow + c0 + 8 * c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2],
                                                                                  w[4 * c + 3]);
                }
            }
        }
    }
    tcgen05_before_sync();
    __syncthreads();
    if (warp == 5) {
        tcgen05_after_sync();
        tmem_dealloc(tmem, Tu::TMEM_COLS);
    }
}

template <typename T, int D, int G>
cudaError_t launch_prefill_umma_tpl(const PrefillArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                    cudaStream_t stream) {
    using Tu = UmmaTuning<D>;
    constexpr size_t smem = UmmaSmem<D, Tu::ST, Tu::NP>::ALLOC;
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    auto kern = paged_prefill_umma_kernel<T, D, G>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static unsigned long long attr_done = 0;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        __atomic_fetch_or(&attr_done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    dim3 grid(a.q_tiles, a.n_kv, a.n_seqs);
    kern<<<grid, 224, smem, stream>>>(a, tk, tv);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_umma_dtype(int head_dim, int group, const PrefillArgs& a, const CUtensorMap& tk,
                                      const CUtensorMap& tv, cudaStream_t stream) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return launch_prefill_umma_tpl<T, DD, GG>(a, tk, tv, stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
