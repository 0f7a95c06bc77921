// decode_f16.cu -- paged decode attention instantiations for __half storage.
#include "decode.cuh"
#include "decode_mma.cuh"

namespace pkv {

cudaError_t launch_decode_f16(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches) {
    const long long rows = (long long)a.num_blocks * a.n_kv * kBlock;
    if (decode_uses_mma(PKV_F16, group, rows)) {
        CUtensorMap tk, tv;
        cudaError_t err = kv_tensor_map(a.k_layer, rows, head_dim, PKV_F16, PKV_BOX_PANEL, &tk);
        if (err == cudaSuccess) err = kv_tensor_map(a.v_layer, rows, head_dim, PKV_F16, PKV_BOX_PANEL, &tv);
        if (err != cudaSuccess) return err;
        return launch_decode_mma_dtype<__half>(head_dim, group, a, tk, tv, stream, n_launches);
    }
    return launch_decode_dtype<__half>(head_dim, group, a, stream, n_launches);
}

cudaError_t decode_ctas_per_sm_f16(int head_dim, int group, long long rows, int* out) {
    if (decode_uses_mma(PKV_F16, group, rows)) return decode_mma_ctas_per_sm_dtype<__half>(head_dim, group, out);
    return decode_ctas_per_sm_dtype<__half>(head_dim, group, out);
}

}  // namespace pkv
