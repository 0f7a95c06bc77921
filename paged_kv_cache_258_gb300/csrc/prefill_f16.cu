// prefill_f16.cu -- paged prefill attention instantiations (tcgen05 tensor cores) for __half storage.
#include "prefill_umma.cuh"

namespace pkv {

cudaError_t launch_prefill_f16(int head_dim, int group, const PrefillArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.num_blocks * a.n_kv * kBlock;
    if (rows >= (1LL << 31)) return cudaErrorInvalidValue;  // TMA row coordinates are 32-bit
    CUtensorMap tk, tv;
    cudaError_t err = kv_tensor_map(a.k_layer, rows, head_dim, PKV_F16, PKV_BOX_PANEL, &tk);
    // head_dim 256 runs as CTA pairs, each CTA copying half of every V block's columns
    const int vbox = UmmaTuning<256>::PAIR && head_dim == 256 ? PKV_BOX_BLOCK_HALF : PKV_BOX_BLOCK;
    if (err == cudaSuccess) err = kv_tensor_map(a.v_layer, rows, head_dim, PKV_F16, vbox, &tv);
    if (err != cudaSuccess) return err;
    return launch_prefill_umma_dtype<__half>(head_dim, group, a, tk, tv, stream);
}

cudaError_t prefill_wave_ctas_f16(int head_dim, int group, int sms, int* out) {
    return prefill_umma_wave_ctas_dtype<__half>(head_dim, group, sms, out);
}

}  // namespace pkv
