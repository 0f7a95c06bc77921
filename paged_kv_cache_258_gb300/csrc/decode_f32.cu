// decode_f32.cu -- paged decode attention instantiations for float storage.
#include "decode.cuh"

namespace pkv {

cudaError_t launch_decode_f32(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches) {
    return launch_decode_dtype<float>(head_dim, group, a, stream, n_launches);
}

cudaError_t decode_ctas_per_sm_f32(int head_dim, int group, long long rows, int* out) {
    (void)rows;
    return decode_ctas_per_sm_dtype<float>(head_dim, group, out);
}

}  // namespace pkv
