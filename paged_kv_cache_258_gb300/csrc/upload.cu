// upload.cu -- a step's metadata, pinned host memory -> device, through the SMs (sm_103a).
//
// The block tables the attention kernels walk ("04 - Hacia PagedAttention (vista previa)", "La idea
// de PagedAttention", steps 2 and 5), with the step's lengths, slots, query starts and copy pairs,
// are written by the host block manager into a page-locked image. A copy-engine copy of that image
// would queue behind bulk host-to-device copies other streams have in flight; this kernel's threads
// read the image directly over the host link instead. A pure byte move, bit-exact by construction.
#include "common.cuh"
#include "internal.h"

namespace pkv {

// One 16-byte word per thread (.cv loads: never served from a cache line fetched before the host
// rewrote the image); a ragged tail of 4-byte words goes to the threads after the last 16-byte word.
__global__ void __launch_bounds__(256) upload_metadata_kernel(uint4* __restrict__ dst,
                                                              const uint4* __restrict__ src, size_t n16,
                                                              uint32_t* __restrict__ dst_tail,
                                                              const uint32_t* __restrict__ src_tail, int n_tail) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n16) dst[i] = __ldcv(src + i);
    const size_t t = i - n16;
    if (i >= n16 && t < (size_t)n_tail) dst_tail[t] = __ldcv(src_tail + t);
}

cudaError_t launch_upload_metadata(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    const size_t n16 = bytes / 16;
    const int n_tail = (int)((bytes % 16) / 4);
    const size_t threads = n16 + (size_t)n_tail;
    const unsigned ctas = (unsigned)((threads + 255) / 256);
    upload_metadata_kernel<<<ctas, 256, 0, stream>>>(
        static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16,
        reinterpret_cast<uint32_t*>(static_cast<char*>(dst) + n16 * 16),
        reinterpret_cast<const uint32_t*>(static_cast<const char*>(src) + n16 * 16), n_tail);
    return cudaGetLastError();
}

}  // namespace pkv
