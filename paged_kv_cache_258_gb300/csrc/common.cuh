// common.cuh -- device helpers: 16-byte vector conversions, mbarriers, bulk TMA copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// ---- element types --------------------------------------------------------------------------
// One 16-byte vector (uint4) of T, widened to fp32.
template <typename T>
struct Vec16;

template <>
struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
};

template <>
struct Vec16<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void word(uint32_t w, float* f) {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        float2 x = __half22float2(h);
        f[0] = x.x;
        f[1] = x.y;
    }
    __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
        word(u.x, f);
        word(u.y, f + 2);
        word(u.z, f + 4);
        word(u.w, f + 6);
    }
};

template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    // bf16 is the top half of an fp32: widening is a shift (low element) or a mask (high).
    __device__ __forceinline__ static void word(uint32_t w, float* f) {
        f[0] = __uint_as_float(w << 16);
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
        word(u.x, f);
        word(u.y, f + 2);
        word(u.z, f + 4);
        word(u.w, f + 6);
    }
};

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---- shared-memory addressing, mbarriers, bulk copies ----------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Upper bound of one wait on an asynchronous copy. A healthy copy completes in microseconds;
// past this the caller records PKV_DEV_WAIT_TIMEOUT and stops waiting instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Wait for the phase of `bar` with the given parity; false if it did not complete in time.
// Wait until the grid this one was launched as a programmatic dependent of has completed and its
// memory operations are visible (returns at once for an ordinary launch).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// L2 policy for data read exactly once (the KV stream): evict it first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One-dimensional bulk copy global -> shared through the TMA engine, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (TMA) accesses to the same memory: required before refilling a buffer that was just read.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy global writes before later async-proxy (TMA) reads
// of the same global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- warp reductions -------------------------------------------------------------------------
// Sum N values per lane across aligned groups of 2*O lanes, halving the values kept per lane at
// each step (a transpose-reduce): after the call, lane L of its group holds the complete sums of
// value indices [(L % (2*O)) * N / (2*O), +max(1, N / (2*O))) in v[0..]. N and O powers of two.
template <int N, int O>
struct HalvingReduce {
    __device__ __forceinline__ static void run(float* v, int lane) {
        if constexpr (O == 0) {
            return;
        } else if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = upper ? v[i] : v[i + H];
                const float keep = upper ? v[i + H] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            HalvingReduce<H, O / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            HalvingReduce<1, O / 2>::run(v, lane);
        }
    }
};

}  // namespace pkv
