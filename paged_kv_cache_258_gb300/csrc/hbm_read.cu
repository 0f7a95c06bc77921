// hbm_read.cu -- a plain streaming read of a device buffer (sm_103a): the read-only ceiling of HBM on
// the part the library runs on. The decode kernels only read KV (a few bytes of outputs per
// kilobyte read), so their bandwidth is best judged against a read-only stream measured the same
// way, beside the read + write copy bandwidth. A measurement helper, not part of the method.
#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kReadThreads = 256;
constexpr int kReadCtasPerSm = 8;  // 2,048 threads per SM, eight 16-byte loads in flight each
constexpr int kReadUnroll = 8;

// Every 16-byte word of src is loaded exactly once (streaming, evict-first) and folded by XOR into
// one 32-bit word per thread; a warp folds its lanes and one lane XORs the result into *fold.
__global__ void __launch_bounds__(kReadThreads) hbm_read_kernel(const uint4* __restrict__ src, size_t n16,
                                                               unsigned int* __restrict__ fold) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned int acc = 0u;
    for (; i + (kReadUnroll - 1) * stride < n16; i += kReadUnroll * stride) {
        uint4 v[kReadUnroll];
#pragma unroll
        for (int k = 0; k < kReadUnroll; ++k) v[k] = __ldcs(src + i + k * stride);
#pragma unroll
        for (int k = 0; k < kReadUnroll; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcs(src + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0 && acc != 0u) atomicXor(fold, acc);
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_hbm_read_probe(const void* buf, size_t bytes, uint32_t* fold, void* stream) {
    if (bytes == 0) return PKV_OK;
    if (!buf || !fold || bytes % 16 != 0) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(buf) & 15u) != 0 || (reinterpret_cast<uintptr_t>(fold) & 3u) != 0)
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    if (pkv::current_sm_count(&sms) != cudaSuccess) return PKV_ERR_CUDA;
    const size_t n16 = bytes / 16;
    const size_t want = (n16 + pkv::kReadThreads - 1) / pkv::kReadThreads;
    const unsigned ctas = (unsigned)(want < (size_t)sms * pkv::kReadCtasPerSm ? want : (size_t)sms * pkv::kReadCtasPerSm);
    pkv::hbm_read_kernel<<<ctas, pkv::kReadThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(buf), n16, fold);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    pkv::count_launches(1);
    return PKV_OK;
}
