// decode_bf16.cu -- paged decode attention instantiations for __nv_bfloat16 storage.
#include "decode.cuh"

namespace pkv {

cudaError_t launch_decode_bf16(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches) {
    return launch_decode_dtype<__nv_bfloat16>(head_dim, group, a, stream, n_launches);
}

}  // namespace pkv
