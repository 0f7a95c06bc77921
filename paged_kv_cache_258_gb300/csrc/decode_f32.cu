// decode_f32.cu -- paged decode attention instantiations for float storage.
#include "decode.cuh"

namespace pkv {

cudaError_t launch_decode_f32(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches) {
    return launch_decode_dtype<float>(head_dim, group, a, stream, n_launches);
}

}  // namespace pkv
