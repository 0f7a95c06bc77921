// decode_mma.cuh -- paged decode attention on the tensor cores, for fp16 / bf16 storage (sm_103a).
//
// Same method, partitions, split-K partials and in-kernel merge as decode.cuh ("04 - Hacia
// PagedAttention (vista previa)", "La idea de PagedAttention", step 5: the kernel walks the block
// table and gathers the rows itself). What changes is how one 16-token block is consumed:
//
//  * K and V chunks arrive by TMA tensor copies (cp.async.bulk.tensor, 2-D map over the layer's
//    rows) in 64-column panels with the 128-byte swizzle, so 8 consecutive token rows of the same
//    16-byte column land in 8 different bank groups and ldmatrix reads are conflict-free.
//  * QK^T runs as S = K . Q^T with mma.sync m16n8k16: M = the 16 tokens of the block, N = 8 query
//    rows (the G rows sharing this KV head, zero-padded), K = head_dim in steps of 16. The packed
//    GQA rows make this a real dense tile; one instruction covers 16 tokens x 8 rows x 16 dims.
//  * The fp32 S fragment feeds the online softmax in registers (each lane owns 2 query rows x 2
//    tokens; row max / sum reduce over the 8 lanes sharing a row). P is rounded to the storage
//    type and turned from the accumulator layout into the B-operand layout of the next MMA with
//    movmatrix.trans -- no shared-memory round trip.
//  * PV runs as O^T = V^T . P^T: M = 16 head dims per instruction (V^T from ldmatrix.trans),
//    N = 8 query rows, K = the 16 tokens. The fp32 accumulator is head_dim/4 registers per lane;
//    it is rescaled only when some row's running maximum moved.
//  * Masked positions: logits past the context are replaced by -inf (selection), and the V rows
//    past the context are zeroed in shared memory before the PV MMA, so NaN in unused rows can
//    never reach the result (0 * NaN would).
// Per 16-token block a warp issues head_dim/8 ldmatrix and head_dim/8 MMA instructions plus ~50
// for the softmax, against ~600-2,100 for the CUDA-core kernel: the kernel stays HBM-bound even
// with 4 query rows per KV head.
#pragma once

#include <math.h>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"

namespace pkv {

template <typename T>
struct MmaType;
template <>
struct MmaType<__half> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return __half22float2(*reinterpret_cast<__half2*>(&w));
    }
    __device__ __forceinline__ static void mma(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};
template <>
struct MmaType<__nv_bfloat16> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ __forceinline__ static void mma(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// 2-D tensor copy of a 64-column x 16-row box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Byte offset, inside a swizzled [panel][16 rows][128 B] tile, of 16-byte column chunk `ch`
// (of the whole row) of token row `r`: the 128-byte swizzle XORs the chunk index with r mod 8.
__device__ __forceinline__ uint32_t swz(int r, int ch) {
    return (uint32_t)((ch >> 3) * 2048 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

template <int D, int NW, int ST>
struct MmaSmem {
    static constexpr size_t TILE = 16 * D * 2;                       // one K or V tile (bytes)
    static constexpr size_t STAGES = (size_t)NW * ST * 2 * TILE;     // 1024-aligned base
    static constexpr size_t BARS = STAGES;                           // uint64 [NW][ST][K, V]
    static constexpr size_t PHYS = BARS + (size_t)NW * ST * 16;     // int [NW][ST]
    static constexpr size_t ML = (PHYS + (size_t)NW * ST * 4 + 15) / 16 * 16;  // float [NW][8][2]
    static constexpr size_t TOTAL = ML + (size_t)NW * 8 * 2 * 4;
    static constexpr size_t ALLOC = TOTAL + 1024;                     // room to align the base
    static constexpr size_t MERGE = (size_t)NW * 8 * D * 4;          // merge scratch, after the combine buffer
    static_assert(MERGE + MergeScratch<8>::BYTES <= STAGES, "combine buffer and merge scratch must fit");
};

template <typename T, int D, int G, int NW, int ST>
__global__ void __launch_bounds__(NW * 32) paged_decode_mma_kernel(const DecodeArgs a,
                                                                    const __grid_constant__ CUtensorMap tm_k,
                                                                    const __grid_constant__ CUtensorMap tm_v) {
    static_assert(G <= 8, "at most 8 query rows per KV head");
    using M = MmaType<T>;
    using S = MmaSmem<D, NW, ST>;
    constexpr int KSTEPS = D / 16;  // QK k-steps = PV m-tiles
    constexpr int PANELS = D / 64;
    constexpr uint32_t TILE = (uint32_t)S::TILE;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BARS);
    int* s_phys = reinterpret_cast<int*>(smem + S::PHYS);
    float* s_ml = reinterpret_cast<float*>(smem + S::ML);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;  // MMA group id: token (QK C rows) / dim (PV C rows)
    const int tig = lane & 3;   // thread in group: owns query rows 2*tig, 2*tig+1
    const int p = blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    // A launch that follows this one as a programmatic dependent (the next layer of the same
    // decode step) may start once every CTA of this grid has passed here: its CTAs then fill the
    // SMs this grid's tail leaves idle. Without such a launch this is a no-op.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // This warp's blocks of the partition are p*bpp + warp + k*NW (k < nk). Their table entries live
    // in registers, 32 per chunk (lane l holds entry 32c + l of chunk c): chunk 0 is read before the
    // context length is known, so the two global reads overlap, and each later chunk one chunk ahead
    // of its first use. Entries past the sequence's last block are read (inside the table row) but
    // never used.
    auto load_chunk = [&](int c) -> int {
        const long long kk = (long long)c * 32 + lane;
        const long long idx = (long long)p * a.bpp + warp + kk * NW;
        return kk * NW + warp < a.bpp && idx < a.max_blocks ? walk_entry(a, s, (int)idx) : -1;
    };
    int tab_lo = load_chunk(0);                        // entries of chunk c_lo
    int tab_hi = a.bpp > 32 * NW ? load_chunk(1) : -1;  // entries of chunk c_lo + 1
    int ctx = a.lens[s];
    const int cap = a.max_blocks * kBlock;
    if (ctx < 0 || ctx > cap) {
        if (p == 0 && threadIdx.x == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_CONTEXT_LEN);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int nb = (ctx + kBlock - 1) / kBlock;
    const int b0 = p * a.bpp;
    if (b0 >= nb) {
        if (p == 0) {
            grid_dependency_wait();
            T* o = reinterpret_cast<T*>(a.out) + ((size_t)s * a.n_q + (size_t)g * G) * D;
            for (int i = threadIdx.x; i < G * D; i += NW * 32) o[i] = from_float<T>(0.f);
        }
        return;
    }
    const int nblk = min(a.bpp, nb - b0);
    const bool single = nb <= a.bpp;
    fused_append<T, D, NW * 32>(a, s, g, p, ctx, nb);

    // Two mbarriers per stage: K tile (even) and V tile (odd), so QK^T starts as soon as K lands and
    // the next K copy is issued before PV runs.
    if (threadIdx.x < 2 * NW * ST) mbar_init(&bars[threadIdx.x], 1);
    fence_mbar_init();
    __syncthreads();

    uint64_t* wbars = bars + warp * ST * 2;  // [ST][K, V]
    int* wphys = s_phys + warp * ST;
    const uint32_t wstage = smem_addr(smem) + (uint32_t)(warp * ST) * 2 * TILE;
    unsigned char* wstage_ptr = smem + (size_t)warp * ST * 2 * TILE;
    const int nk = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;
    const uint64_t policy = l2_evict_first_policy();

    // Every lane: the physical block of this warp's k-th block, for k = 0, 1, 2, ... in order (each
    // exactly once); entering chunk c moves to it and starts the read of chunk c + 1.
    auto entry = [&](int k) -> int {
        if ((k & 31) == 0 && k > 0) {
            tab_lo = tab_hi;
            tab_hi = load_chunk((k >> 5) + 1);
        }
        return __shfl_sync(0xffffffffu, tab_lo, k & 31);
    };
    // lane 0: start the copy of the K (v = 0) or V (v = 1) tile of this warp's k-th block
    auto issue = [&](int k, int v, int phys) {
        const int st = k % ST;
        const bool ok = (unsigned)phys < (unsigned)a.num_blocks;
        uint64_t* bar = &wbars[st * 2 + v];
        if (v == 0) wphys[st] = ok ? phys : -1;
        if (ok) {
            const int row0 = (int)(chunk_index(a, s, g, phys) * kBlock);
            const uint32_t dst = wstage + (uint32_t)st * 2 * TILE + (uint32_t)v * TILE;
            mbar_arrive_expect_tx(bar, TILE);
#pragma unroll
            for (int pn = 0; pn < PANELS; ++pn) tma_load_2d(dst + pn * 2048, v ? &tm_v : &tm_k, pn * 64, row0, bar, policy);
        } else {
            if (v == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_BLOCK_ID);
            mbar_arrive(bar);  // completes the phase with nothing copied: the block is masked
        }
    };
    // after a timed-out wait: wait (bounded) for the tiles of blocks [k0, k1) of kind v still in flight
    auto drain = [&](int k0, int k1, int v) {
        for (int kk = k0; kk < k1 && kk < nk; ++kk) mbar_wait_bounded(&wbars[(kk % ST) * 2 + v], (uint32_t)(kk / ST) & 1u);
    };
    for (int k = 0; k < ST && k < nk; ++k) {
        const int phys = entry(k);
        if (lane == 0) {
            issue(k, 0, phys);
            issue(k, 1, phys);
        }
    }

    // Q^T fragments (B operand of S = K Q^T): row gid, dims 16ks + 2tig (+1) and +8; rows >= G are 0.
    uint32_t qb[KSTEPS][2];
    {
        const T* qrow = reinterpret_cast<const T*>(a.q) + ((size_t)s * a.n_q + (size_t)g * G + gid) * D;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            if (gid < G) {
                qb[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * tig);
                qb[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * tig);
            } else {
                qb[ks][0] = 0u;
                qb[ks][1] = 0u;
            }
        }
    }

    float acc[KSTEPS][4];  // O^T: m-tile mt, (dim 16mt+gid | +8) x (row 2tig | 2tig+1)
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const float sl = a.scale_log2;

    // ldmatrix row addresses: matrix mi = lane / 8, row lane % 8
    const int mi = lane >> 3;
    const int lr = lane & 7;
    const int k_tok = lr + 8 * (mi & 1);  // K (A of QK): matrices (t0-7,c0) (t8-15,c0) (t0-7,c1) (t8-15,c1)
    const int k_chk = mi >> 1;
    const int v_tok = lr + 8 * (mi >> 1);  // V (A of PV, transposed): (t0-7,c0) (t0-7,c1) (t8-15,c0) (t8-15,c1)
    const int v_chk = mi & 1;

    for (int k = 0; k < nk; ++k) {
        const int st = k % ST;
        const uint32_t par = (uint32_t)(k / ST) & 1u;
        const int phys_next = k + ST < nk ? entry(k + ST) : -1;  // the block whose copies go next
        if (!mbar_wait_bounded(&wbars[st * 2], par)) {
            if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
            drain(k, k + ST, 0);  // K tiles of blocks k .. k+ST-1 may be in flight
            drain(k, k + ST, 1);  // and their V tiles
            break;
        }
        const int jb = (b0 + warp + k * NW) * kBlock;
        const int nvalid = wphys[st] >= 0 ? min(kBlock, ctx - jb) : 0;
        const uint32_t sK = wstage + (uint32_t)st * 2 * TILE;
        const uint32_t sV = sK + TILE;
        uint32_t b0f = 0u, b1f = 0u;
        if (nvalid > 0) {
            // ---- S = K Q^T (16 tokens x 8 rows), fp32 ----
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                uint32_t af[4];
                ldmatrix_x4(af, sK + swz(k_tok, 2 * ks + k_chk));
                M::mma(sc, af, qb[ks][0], qb[ks][1]);
            }
            // ---- online softmax: lane holds tokens gid, gid+8 of rows 2tig, 2tig+1 ----
            const bool v0 = gid < nvalid, v1 = gid + 8 < nvalid;
            const float z0 = v0 ? sc[0] * sl : -INFINITY;  // token gid,   row 2tig
            const float z1 = v0 ? sc[1] * sl : -INFINITY;  // token gid,   row 2tig+1
            const float z2 = v1 ? sc[2] * sl : -INFINITY;  // token gid+8, row 2tig
            const float z3 = v1 ? sc[3] * sl : -INFINITY;  // token gid+8, row 2tig+1
            float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
            const float al0 = (m_run[0] == -INFINITY) ? 0.f : exp2f(m_run[0] - mn0);
            const float al1 = (m_run[1] == -INFINITY) ? 0.f : exp2f(m_run[1] - mn1);
            m_run[0] = mn0;
            m_run[1] = mn1;
            const float p0 = (z0 == -INFINITY) ? 0.f : exp2f(z0 - mn0);
            const float p1 = (z1 == -INFINITY) ? 0.f : exp2f(z1 - mn1);
            const float p2 = (z2 == -INFINITY) ? 0.f : exp2f(z2 - mn0);
            const float p3 = (z3 == -INFINITY) ? 0.f : exp2f(z3 - mn1);
            const uint32_t pa = M::pack(p0, p1);  // token gid:   rows 2tig, 2tig+1
            const uint32_t pb = M::pack(p2, p3);  // token gid+8
            const float2 ra = M::unpack(pa), rb = M::unpack(pb);  // the rounded weights the MMA uses
            l_run[0] = l_run[0] * al0 + ra.x + rb.x;
            l_run[1] = l_run[1] * al1 + ra.y + rb.y;
            b0f = movmatrix_trans(pa);  // P^T: tokens 2tig, 2tig+1 of row gid
            b1f = movmatrix_trans(pb);  // tokens 8+2tig, 9+2tig of row gid
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    acc[mt][0] *= al0;
                    acc[mt][1] *= al1;
                    acc[mt][2] *= al0;
                    acc[mt][3] *= al1;
                }
            }
        }
        __syncwarp();  // the K tile has been read by every lane
        if (lane == 0 && k + ST < nk) {
            fence_proxy_async_smem();
            issue(k + ST, 0, phys_next);
        }
        if (!mbar_wait_bounded(&wbars[st * 2 + 1], par)) {
            if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
            drain(k + 1, k + ST + 1, 0);  // K tiles of blocks k+1 .. k+ST may be in flight
            drain(k, k + ST, 1);          // V tiles of blocks k .. k+ST-1
            break;
        }
        if (nvalid > 0) {
            if (nvalid < kBlock) {  // zero the V rows past the context (they may hold anything)
                unsigned char* vt = wstage_ptr + (size_t)st * 2 * TILE + TILE;
                const int nch = (kBlock - nvalid) * (D / 8);
                for (int i = lane; i < nch; i += 32) {
                    const int r = nvalid + i / (D / 8);
                    const int ch = i % (D / 8);
                    *reinterpret_cast<uint4*>(vt + swz(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // ---- O^T += V^T P^T (16 dims x 8 rows per instruction) ----
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
                uint32_t af[4];
                ldmatrix_x4_trans(af, sV + swz(v_tok, 2 * mt + v_chk));
                M::mma(acc[mt], af, b0f, b1f);
            }
        }
        __syncwarp();  // the V tile has been read by every lane
        if (lane == 0 && k + ST < nk) {
            fence_proxy_async_smem();
            issue(k + ST, 1, phys_next);
        }
    }

    // ---- row sums over the 8 lanes sharing a row ----
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], o);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], o);
    }

    // ---- merge the warps ----
    // Launched as a programmatic dependent, this grid may have streamed its keys while the previous
    // kernel was finishing; the split-K workspace and the outputs are touched only once that kernel
    // has completed and its writes are visible. Otherwise the wait returns at once.
    grid_dependency_wait();
    __syncthreads();
    float* s_acc = reinterpret_cast<float*>(smem);  // [NW][8][D]
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
        const int d0 = 16 * mt + gid;
        const int r0 = 2 * tig;
        float* base = s_acc + (size_t)warp * 8 * D;
        if (r0 < G) {
            base[r0 * D + d0] = acc[mt][0];
            base[r0 * D + d0 + 8] = acc[mt][2];
        }
        if (r0 + 1 < G) {
            base[(r0 + 1) * D + d0] = acc[mt][1];
            base[(r0 + 1) * D + d0 + 8] = acc[mt][3];
        }
    }
    if (gid == 0) {
        const int r0 = 2 * tig;
        s_ml[(warp * 8 + r0) * 2] = m_run[0];
        s_ml[(warp * 8 + r0) * 2 + 1] = l_run[0];
        s_ml[(warp * 8 + r0 + 1) * 2] = m_run[1];
        s_ml[(warp * 8 + r0 + 1) * 2 + 1] = l_run[1];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int r = idx / D;
        const int d = idx % D;
        float Mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) Mx = fmaxf(Mx, s_ml[(w * 8 + r) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float mw = s_ml[(w * 8 + r) * 2];
            if (mw != -INFINITY) {
                const float sc = exp2f(mw - Mx);
                L = fmaf(s_ml[(w * 8 + r) * 2 + 1], sc, L);
                O = fmaf(s_acc[((size_t)w * 8 + r) * D + d], sc, O);
            }
        }
        const size_t row = (size_t)s * a.n_q + (size_t)g * G + r;
        if (single) {
            reinterpret_cast<T*>(a.out)[row * D + d] = from_float<T>(L > 0.f ? O / L : 0.f);
        } else {
            const size_t prow = row * a.n_parts + p;
            a.part_o[prow * D + d] = O;
            if (d == 0) {
                a.part_ml[prow * 2] = Mx;
                a.part_ml[prow * 2 + 1] = L;
            }
        }
    }
    if (!single)
        splitk_merge_if_last<T, D, G, NW * 32>(a, s, g, (nb + a.bpp - 1) / a.bpp,
                                               reinterpret_cast<float*>(smem + S::MERGE));
}

template <typename T, int D, int G>
struct MmaTuning {
    // A stage holds one K + V tile pair (32*D bytes). 64 KiB per CTA (3 CTAs per SM) measured best
    // for D=128 (2 stages per warp) and D=256 (1 stage per warp, latency covered by 12 warps/SM).
    static constexpr int NW = 4;
    static constexpr int ST = D == 256 ? 1 : (D == 128 ? 2 : 4);
};

template <typename T, int D, int G>
struct DecodeMmaKernel {
    static constexpr int NW = MmaTuning<T, D, G>::NW;
    static constexpr int ST = MmaTuning<T, D, G>::ST;
    static constexpr size_t smem = MmaSmem<D, NW, ST>::ALLOC;
    static unsigned long long attr_done;
    static cudaError_t prepare() {
        return allow_dynamic_smem(paged_decode_mma_kernel<T, D, G, NW, ST>, smem, &attr_done);
    }
    // CTAs of this kernel one SM holds at once (shared memory, registers, threads)
    static cudaError_t ctas_per_sm(int* out) {
        cudaError_t err = prepare();
        if (err != cudaSuccess) return err;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, paged_decode_mma_kernel<T, D, G, NW, ST>, NW * 32,
                                                             smem);
    }
};
template <typename T, int D, int G>
unsigned long long DecodeMmaKernel<T, D, G>::attr_done = 0;

template <typename T, int D, int G>
cudaError_t launch_decode_mma_tpl(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream, int* n_launches) {
    using K = DecodeMmaKernel<T, D, G>;
    constexpr int NW = K::NW;
    constexpr size_t smem = K::smem;
    auto kern = paged_decode_mma_kernel<T, D, G, NW, K::ST>;
    cudaError_t err = K::prepare();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_parts, a.n_kv, a.n_seqs);
    cfg.blockDim = dim3(NW * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.overlap_previous ? 1 : 0;
    err = cudaLaunchKernelEx(&cfg, kern, a, tk, tv);
    if (err != cudaSuccess) return err;
    if (n_launches) *n_launches = 1;
    return cudaGetLastError();
}

template <typename T>
cudaError_t decode_mma_ctas_per_sm_dtype(int head_dim, int group, int* out) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return DecodeMmaKernel<T, DD, GG>::ctas_per_sm(out);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_decode_mma_dtype(int head_dim, int group, const DecodeArgs& a, const CUtensorMap& tk,
                                    const CUtensorMap& tv, cudaStream_t stream, int* n) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return launch_decode_mma_tpl<T, DD, GG>(a, tk, tv, stream, n);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
