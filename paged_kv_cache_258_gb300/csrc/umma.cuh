// umma.cuh -- thin wrappers over the sm_100-family tensor-core instructions (tcgen05) and tensor
// memory (TMEM), as used by the prefill kernel. Encodings follow the PTX ISA:
//   * shared-memory matrix descriptor (64-bit): start address >> 4 in bits [0,14), leading byte
//     offset >> 4 in [16,30), stride byte offset >> 4 in [32,46), descriptor version 1 in [46,48),
//     layout (2 = 128-byte swizzle) in [61,64);
//   * instruction descriptor of .kind::f16 (32-bit): D format in [4,6) (1 = f32), A and B formats in
//     [7,10) and [10,13) (0 = f16, 1 = bf16), A / B major-ness in bits 15 / 16 (1 = MN-major),
//     N >> 3 in [17,23), M >> 4 in [24,29).
// With the 128-byte swizzle every operand tile is stored as 64-element (128-byte) panels of rows,
// eight rows forming one 1024-byte swizzle atom:
//   K-major operand (rows = M or N, 16-element k-steps): stride byte offset 1024 (next 8 rows);
//     a k-step inside a panel moves the start address by 32 bytes, the next panel by its size;
//   MN-major operand (rows = K, 64 contiguous M/N elements per row per panel): leading byte
//     offset = panel size (next 64 M/N elements), stride byte offset 1024 (next 8 K rows).
#pragma once

#include <stdint.h>

namespace pkv {

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__host__ __device__ constexpr uint32_t umma_idesc_f16(bool bf16, int m, int n, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// The tcgen05 instructions come in two forms: .cta_group::1 (one SM) and .cta_group::2 (a pair of
// CTAs on two SMs of a cluster computing one M = 256 product: each holds half of the rows of A and
// D and half of the N columns of B, at the same shared-memory and tensor-memory offsets, and one
// thread of the even CTA issues). A kernel uses one form throughout; CG selects it.
// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
template <int CG>
__device__ __forceinline__ void umma_f16_cg(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    if constexpr (CG == 2) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
            : "memory");
    }
}

// D[tmem] (+)= A[tmem] * B[smem]: A's row i in TMEM lane i, two 16-bit elements per 32-bit column
// (a 16-element k-step is 8 columns).
template <int CG>
__device__ __forceinline__ void umma_f16_tmem_a_cg(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                   bool accumulate) {
    if constexpr (CG == 2) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
            : "memory");
    }
}

// One arrival on this CTA's mbarrier `bar` once every tcgen05.mma this thread issued so far has
// completed (for .cta_group::2, on both SMs of the pair).
template <int CG>
__device__ __forceinline__ void umma_commit_cg(uint64_t* bar) {
    if constexpr (CG == 2) {
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                     : "memory");
    } else {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                     : "memory");
    }
}

// Whole-warp TMEM allocation of `ncols` columns; for .cta_group::2 one warp of each CTA of the pair
// executes it and both receive the same columns.
template <int CG>
__device__ __forceinline__ void tmem_alloc_cg(uint32_t* dst, uint32_t ncols) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    if constexpr (CG == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(a), "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(a), "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc_cg(uint32_t taddr, uint32_t ncols) {
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- CTA pairs: cluster rank, remote mbarrier arrivals, cluster-scope waits ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the cluster's shared-memory window, of this CTA's shared variable `p` as it sits in
// the CTA of cluster rank `rank` (the same offset there).
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
    return r;
}

// One arrival on an mbarrier of another CTA of the cluster (address from cluster_addr), with the
// instruction's default semantics (release at CTA scope). A release at cluster scope would fence
// the thread's outstanding memory operations first; measured on paired prefill, that put ~0.5-1.5
// us on every hand-off between the two CTAs (a tile took 3.1 us instead of ~1.1). What the hand-offs
// order is physical completion that the arriving thread has already observed (an MMA completion
// seen on its own barrier, or its own shared-memory writes, fenced for the asynchronous proxy).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// `count` arrivals at once on an mbarrier of another CTA of the cluster (default semantics).
__device__ __forceinline__ void mbar_arrive_remote_count(uint32_t cluster_bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar), "r"(count) : "memory");
}

// One arrival per calling thread on an mbarrier of another CTA, sent as a single remote operation
// per group of converged lanes (the lowest lane carries the group's count after a warp sync that
// orders the others' earlier memory operations before its release). Remote arrivals are
// serialised at the receiving CTA, so 32 of them cost far more than one that counts 32.
__device__ __forceinline__ void mbar_arrive_remote_warp(uint32_t cluster_bar) {
    const unsigned m = __activemask();
    __syncwarp(m);
    if ((threadIdx.x & 31) == (unsigned)(__ffs(m) - 1)) mbar_arrive_remote_count(cluster_bar, (uint32_t)__popc(m));
}

// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tcgen05_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tcgen05_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane (the warp covers 32 lanes).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace pkv
