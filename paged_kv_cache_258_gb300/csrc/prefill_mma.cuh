// prefill_mma.cuh -- paged prefill / chunked prefill attention on the tensor cores (fp16 / bf16).
//
// A chunk of n new tokens per sequence attends causally to the sequence's cache through its block
// table ("PagedAttention e continuous batching", "01 - Conceito", paragraph 5: long prompts are
// sliced into chunks; "04 - Hacia PagedAttention (vista previa)", "La idea de PagedAttention",
// step 5: the kernel gathers the rows itself). The chunk's tokens are the newest, already
// appended: with c = context_lens[s] they sit at positions c - n .. c - 1, and position p sees
// keys 0 .. p. Unlike decode this is a dense contraction (n query rows x c keys x head_dim), so
// the work is laid out for the tensor pipe:
//
//  * CTA = (tile of query rows, KV head, sequence). The G query heads sharing one KV head are
//    packed into the rows (row = token * G + head-in-group), so every K/V tile is read once for
//    all of them; a CTA holds 16 * NWC rows, one 16-row slice per consumer warp.
//  * One producer warp walks the block table and moves each 64-key tile (four 16-token blocks)
//    of K and of V into a ring of ST shared-memory stages with TMA tensor copies (64-column x
//    16-row boxes, 128-byte swizzle), on a "full" mbarrier per stage for K and one for V; the
//    consumer warps release a stage on its "empty" mbarrier.
//  * Consumer warps (flash-attention style, mma.sync m16n8k16, fp32 accumulate): S = Q K^T for
//    their 16 rows x 64 keys, causal/context masking by selection, online softmax in base 2 in
//    registers, P rounded to the storage type and fed straight from the S accumulators as the A
//    operand of O += P V (V through ldmatrix.trans).
//  * Rows past a sequence's context in its last tile: the producer zeroes those V rows once the
//    tile has landed (their P is exactly 0, but 0 * NaN would not be), then signals a one-shot
//    mbarrier the consumers wait on for that tile.
//  * Every wait is bounded (PKV_DEV_WAIT_TIMEOUT, then a bounded drain of copies in flight).
#pragma once

#include <math.h>

#include "common.cuh"
#include "decode_mma.cuh"
#include "internal.h"

namespace pkv {

// 2-D tensor copy of a 64-column x 16-row box with the default L2 policy (K/V tiles of a prefill
// are re-read by every query tile of the sequence, so they should stay in L2).
__device__ __forceinline__ void tma_load_2d_keep(uint32_t dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

template <int D, int NWC, int ST>
struct PrefillSmem {
    static constexpr int ROWS = 16 * NWC;                 // query rows per CTA
    static constexpr size_t BLK = 16 * D * 2;            // one (block, KV head) chunk
    static constexpr int BPT = 4;                         // blocks per 64-key tile
    static constexpr size_t KT = BPT * BLK;              // one K (or V) tile
    static constexpr size_t Q = (size_t)ST * 2 * KT;    // [D/64 panels][ROWS][128 B], swizzled
    static constexpr size_t BARS = Q + (size_t)ROWS * D * 2;  // full_k[ST], full_v[ST], empty[ST], vtail
    static constexpr size_t OKM = BARS + (size_t)(3 * ST + 1) * 8;  // int[ST]: loaded-block mask
    static constexpr size_t TOTAL = OKM + (size_t)ST * 4;
    static constexpr size_t ALLOC = TOTAL + 1024;         // room to align the base to 1024
};

// Byte offset of 16-byte chunk `ch` of query row `r` in the swizzled Q tile of `ROWS` rows.
template <int ROWS>
__device__ __forceinline__ uint32_t swzq(int r, int ch) {
    return (uint32_t)((ch >> 3) * ROWS * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

template <typename T, int D, int G, int NWC, int ST>
__global__ void __launch_bounds__((NWC + 1) * 32, 1)
    paged_prefill_mma_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v) {
    static_assert(16 % G == 0, "a warp's 16 rows hold whole tokens");
    using M = MmaType<T>;
    using S = PrefillSmem<D, NWC, ST>;
    constexpr int ROWS = S::ROWS;
    constexpr int QT = ROWS / G;      // query tokens per CTA
    constexpr int KSTEPS = D / 16;    // QK^T k-steps
    constexpr int PANELS = D / 64;
    constexpr int NT = D / 8;         // PV n-tiles (8 head dims each)
    constexpr uint32_t BLK = (uint32_t)S::BLK;
    constexpr uint32_t KT = (uint32_t)S::KT;
    constexpr bool QREG = D <= 128;   // Q fragments held in registers (else re-read per tile)
    constexpr int KC = D <= 128 ? 64 : 32;  // keys per compute sub-tile (register budget at D = 256)
    constexpr int NTHREADS = (NWC + 1) * 32;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* full_k = reinterpret_cast<uint64_t*>(smem + S::BARS);
    uint64_t* full_v = full_k + ST;
    uint64_t* empty = full_v + ST;
    uint64_t* vtail = empty + ST;
    int* s_ok = reinterpret_cast<int*>(smem + S::OKM);
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
    const int pos0 = ctx - n_new + t0;           // position of the CTA's first token
    const int pos_last = ctx - n_new + t_end - 1;
    const int n_tiles = pos_last / 64 + 1;       // 64-key tiles covering keys 0 .. pos_last
    const int nb = (ctx + kBlock - 1) / kBlock;
    const bool tail_tile = n_tiles * 64 > ctx;   // the last tile holds rows past the context

    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full_k[i], 1);
            mbar_init(&full_v[i], 1);
            mbar_init(&empty[i], NWC);
        }
        mbar_init(vtail, 32);
        fence_mbar_init();
    }
    // Q tile -> shared memory; rows of tokens past the chunk are zero
    {
        const T* qg = reinterpret_cast<const T*>(a.q);
        for (int i = threadIdx.x; i < ROWS * (D / 8); i += NTHREADS) {
            const int r = i / (D / 8);
            const int ch = i % (D / 8);
            const int tt = r / G;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t0 + tt < n_new)
                v = *reinterpret_cast<const uint4*>(qg + ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + r % G) * D +
                                                    ch * 8);
            *reinterpret_cast<uint4*>(smem + S::Q + swzq<ROWS>(r, ch)) = v;
        }
    }
    __syncthreads();

    if (warp == NWC) {
        // ===================== producer warp =====================
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
            if (badm) {
                // skipped blocks: their keys are masked, and their V rows are zeroed (P = 0 there,
                // but 0 * stale NaN would not be 0)
                if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_BLOCK_ID);
                for (int b = 0; b < 4; ++b) {
                    if (!((badm >> b) & 1u)) continue;
                    unsigned char* vb = smem + (size_t)st * 2 * KT + KT + (size_t)b * BLK;
                    for (int i = lane; i < (int)(BLK / 16); i += 32)
                        reinterpret_cast<uint4*>(vb)[i] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                s_ok[st] = (int)okm;
                const uint32_t bytes = (uint32_t)__popc(okm) * BLK;
                mbar_arrive_expect_tx(&full_k[st], bytes);
                mbar_arrive_expect_tx(&full_v[st], bytes);
            }
            __syncwarp();
            if (ok) {
                const int row0 = (phys * a.n_kv + g) * kBlock;
                const uint32_t dk = sbase + (uint32_t)st * 2 * KT + (uint32_t)lane * BLK;
#pragma unroll
                for (int pn = 0; pn < PANELS; ++pn) tma_load_2d_keep(dk + pn * 2048, &tm_k, pn * 64, row0, &full_k[st]);
#pragma unroll
                for (int pn = 0; pn < PANELS; ++pn)
                    tma_load_2d_keep(dk + KT + pn * 2048, &tm_v, pn * 64, row0, &full_v[st]);
            }
            issued = j + 1;
            if (j == n_tiles - 1 && tail_tile) {
                // zero the V rows at or past the context once the tile has landed, then release it
                if (!mbar_wait_bounded(&full_v[st], (uint32_t)(j / ST) & 1u)) {
                    if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
                    break;
                }
                const int r0 = ctx - j * 64;  // first row past the context, 1 .. 63
                unsigned char* vt = smem + (size_t)st * 2 * KT + KT;
                for (int i = lane; i < (64 - r0) * (D / 8); i += 32) {
                    const int r = r0 + i / (D / 8);
                    const int ch = i % (D / 8);
                    *reinterpret_cast<uint4*>(vt + (size_t)(r >> 4) * BLK + swz(r & 15, ch)) = make_uint4(0u, 0u, 0u, 0u);
                }
                mbar_arrive(vtail);
            }
        }
        // wait (bounded) for the copies of the last stages before the CTA may exit
        for (int j = max(0, issued - ST); j < issued; ++j) {
            mbar_wait_bounded(&full_k[j % ST], (uint32_t)(j / ST) & 1u);
            mbar_wait_bounded(&full_v[j % ST], (uint32_t)(j / ST) & 1u);
        }
        return;
    }

    // ===================== consumer warps =====================
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int mi = lane >> 3;
    const int lr = lane & 7;
    const int qa_row = warp * 16 + lr + 8 * (mi & 1);  // A (Q): (r0-7,c) (r8-15,c) (r0-7,c+1) (r8-15,c+1)
    const int qa_chk = mi >> 1;
    const int kb_row = lr + 8 * (mi >> 1);              // B (K): (k0-7,c) (k0-7,c+1) (k8-15,c) (k8-15,c+1)
    const int kb_chk = mi & 1;
    const int vb_row = lr + 8 * (mi & 1);               // B (V, trans): (k0-7,c) (k8-15,c) (k0-7,c+1) (k8-15,c+1)
    const int vb_chk = mi >> 1;

    uint32_t qf[QREG ? KSTEPS : 1][4];
    if constexpr (QREG) {
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) ldmatrix_x4(qf[ks], sQ + swzq<ROWS>(qa_row, 2 * ks + qa_chk));
    }

    const int r_lo = warp * 16 + gid;  // this lane's rows: r_lo and r_lo + 8
    const int lim0 = min(pos0 + r_lo / G, ctx - 1);
    const int lim1 = min(pos0 + (r_lo + 8) / G, ctx - 1);
    const int wmin = min(pos0 + (warp * 16) / G, ctx - 1);      // smallest limit among the warp's rows
    const int wmax = min(pos0 + (warp * 16 + 15) / G, ctx - 1);  // largest
    const float sl = a.scale_log2;

    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool timed_out = false;

    for (int j = 0; j < n_tiles; ++j) {
        const int st = j % ST;
        const uint32_t par = (uint32_t)(j / ST) & 1u;
        if (!mbar_wait_bounded(&full_k[st], par)) {
            timed_out = true;
            break;
        }
        const int key0 = j * 64;
        const uint32_t sK = sbase + (uint32_t)st * 2 * KT;
        const uint32_t sV = sK + KT;
        bool v_ready = false;
        // the 64-key tile is consumed in sub-tiles of KC keys (KC / 8 S n-tiles live at a time)
#pragma unroll
        for (int h = 0; h < 64 / KC; ++h) {
            const int kc0 = key0 + h * KC;
            const bool active = kc0 <= wmax;  // some key of the sub-tile is visible to some row of the warp
            uint32_t pk[KC / 8][2];
            if (active) {
                // ---- S = Q K^T: 16 rows x KC keys ----
                float sc[KC / 8][4];
#pragma unroll
                for (int n = 0; n < KC / 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    uint32_t qt[4];
                    const uint32_t* af;
                    if constexpr (QREG) {
                        af = qf[ks];
                    } else {
                        ldmatrix_x4(qt, sQ + swzq<ROWS>(qa_row, 2 * ks + qa_chk));
                        af = qt;
                    }
#pragma unroll
                    for (int np = 0; np < KC / 16; ++np) {
                        uint32_t b[4];
                        ldmatrix_x4(b, sK + (uint32_t)(h * (KC / 16) + np) * BLK + swz(kb_row, 2 * ks + kb_chk));
                        M::mma(sc[2 * np], af, b[0], b[1]);
                        M::mma(sc[2 * np + 1], af, b[2], b[3]);
                    }
                }
                // ---- masking by selection: key <= the row's position (and < context), block loaded ----
                const int okm = s_ok[st] >> (h * (KC / 16));
                constexpr int full = (1 << (KC / 16)) - 1;
                if (kc0 + KC - 1 > wmin || (okm & full) != full) {
#pragma unroll
                    for (int n = 0; n < KC / 8; ++n) {
                        const int key = kc0 + 8 * n + 2 * tig;
                        const bool bok = (okm >> (n >> 1)) & 1;
                        sc[n][0] = (bok && key <= lim0) ? sc[n][0] * sl : -INFINITY;
                        sc[n][1] = (bok && key + 1 <= lim0) ? sc[n][1] * sl : -INFINITY;
                        sc[n][2] = (bok && key <= lim1) ? sc[n][2] * sl : -INFINITY;
                        sc[n][3] = (bok && key + 1 <= lim1) ? sc[n][3] * sl : -INFINITY;
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < KC / 8; ++n) {
                        sc[n][0] *= sl;
                        sc[n][1] *= sl;
                        sc[n][2] *= sl;
                        sc[n][3] *= sl;
                    }
                }
                // ---- online softmax (base 2): rows r_lo (values 0,1) and r_lo + 8 (values 2,3) ----
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int n = 0; n < KC / 8; ++n) {
                    mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
                    mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0);
                const float mn1 = fmaxf(m1, mx1);
                const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
                const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
                m0 = mn0;
                m1 = mn1;
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int n = 0; n < KC / 8; ++n) {
                    const float p0 = sc[n][0] == -INFINITY ? 0.f : exp2f(sc[n][0] - mn0);
                    const float p1 = sc[n][1] == -INFINITY ? 0.f : exp2f(sc[n][1] - mn0);
                    const float p2 = sc[n][2] == -INFINITY ? 0.f : exp2f(sc[n][2] - mn1);
                    const float p3 = sc[n][3] == -INFINITY ? 0.f : exp2f(sc[n][3] - mn1);
                    pk[n][0] = M::pack(p0, p1);
                    pk[n][1] = M::pack(p2, p3);
                    const float2 ra = M::unpack(pk[n][0]);  // the rounded weights the MMA uses
                    const float2 rb = M::unpack(pk[n][1]);
                    ls0 += ra.x + ra.y;
                    ls1 += rb.x + rb.y;
                }
                l0 = l0 * al0 + ls0;
                l1 = l1 * al1 + ls1;
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        o[n][0] *= al0;
                        o[n][1] *= al0;
                        o[n][2] *= al1;
                        o[n][3] *= al1;
                    }
                }
            }
            if (!v_ready) {
                v_ready = mbar_wait_bounded(&full_v[st], par) &&
                          (j != n_tiles - 1 || !tail_tile || mbar_wait_bounded(vtail, 0u));
                if (!v_ready) {
                    timed_out = true;
                    break;
                }
            }
            if (active) {
                // ---- O += P V: A = P straight from the S accumulators, B = V^T via ldmatrix.trans ----
#pragma unroll
                for (int kk = 0; kk < KC / 16; ++kk) {
                    const uint32_t af[4] = {pk[2 * kk][0], pk[2 * kk][1], pk[2 * kk + 1][0], pk[2 * kk + 1][1]};
                    const uint32_t vblk = sV + (uint32_t)(h * (KC / 16) + kk) * BLK;
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        uint32_t b[4];
                        ldmatrix_x4_trans(b, vblk + swz(vb_row, 2 * dp + vb_chk));
                        M::mma(o[2 * dp], af, b[0], b[1]);
                        M::mma(o[2 * dp + 1], af, b[2], b[3]);
                    }
                }
            }
        }
        if (timed_out) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (timed_out) {
        if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
        return;
    }

    // ---- normalise, stage this warp's 16 rows in its own Q rows, store 16-byte chunks ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    __syncwarp();
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        *reinterpret_cast<uint32_t*>(smem + S::Q + swzq<ROWS>(r_lo, n) + 4 * tig) = M::pack(o[n][0] * inv0, o[n][1] * inv0);
        *reinterpret_cast<uint32_t*>(smem + S::Q + swzq<ROWS>(r_lo + 8, n) + 4 * tig) =
            M::pack(o[n][2] * inv1, o[n][3] * inv1);
    }
    __syncwarp();
    T* og = reinterpret_cast<T*>(a.out);
    for (int i = lane; i < 16 * (D / 8); i += 32) {
        const int r = warp * 16 + i / (D / 8);
        const int ch = i % (D / 8);
        const int tt = r / G;
        if (t0 + tt < n_new)
            *reinterpret_cast<uint4*>(og + ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + r % G) * D + ch * 8) =
                *reinterpret_cast<const uint4*>(smem + S::Q + swzq<ROWS>(r, ch));
    }
}

template <typename T, int D, int G>
struct PrefillTuning {
    static constexpr int NWC = prefill_mma_rows(D) / 16;  // one 16-row slice per consumer warp
    static constexpr int ST = D == 256 ? 2 : 4;        // stages of 64 keys (K + V)
    static constexpr int QT = 16 * NWC / G;            // query tokens per CTA
};

template <typename T, int D, int G>
cudaError_t launch_prefill_mma_tpl(const PrefillArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                   cudaStream_t stream) {
    constexpr int NWC = PrefillTuning<T, D, G>::NWC;
    constexpr int ST = PrefillTuning<T, D, G>::ST;
    constexpr size_t smem = PrefillSmem<D, NWC, ST>::ALLOC;
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    auto kern = paged_prefill_mma_kernel<T, D, G, NWC, ST>;
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
    kern<<<grid, (NWC + 1) * 32, smem, stream>>>(a, tk, tv);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_mma_dtype(int head_dim, int group, const PrefillArgs& a, const CUtensorMap& tk,
                                     const CUtensorMap& tv, cudaStream_t stream) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return launch_prefill_mma_tpl<T, DD, GG>(a, tk, tv, stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
