// decode_static.cu -- paged decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run decode
// attention: code running while a CUDA stream is being captured into a graph, a real-time
// serving loop that forbids allocation after start-up, or a host that embeds this library
// under a fixed device-memory budget with no allocator of its own. pkv_paged_decode_attention
// needs a caller-provided workspace for its split-K partial results; this entry point instead
// uses a fixed scratch array compiled into the library, so it allocates nothing.
//
// The scratch is a file-scope __device__ array of PKV_STATIC_SCRATCH_BYTES (16 MiB): every GPU
// that loads the library holds it until the process exits. In host code the array's name is
// only a host-side stand-in, not a device address, so its device address is looked up once per
// device with cudaGetSymbolAddress and passed to the kernels.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchFloats = PKV_STATIC_SCRATCH_BYTES / sizeof(float);

// Split-K partial results of pkv_paged_decode_attention_static. Every call shares it.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

std::mutex g_scratch_mu;
float* g_scratch_addr[64] = {};

// Device address of this device's scratch array, resolved on the first call per device.
cudaError_t scratch_for_current_device(float** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

}  // namespace

extern "C" int pkv_paged_decode_attention_static(const pkv_cache_desc* d, int32_t layer, const void* q,
                                                 const void* k_pool, const void* v_pool,
                                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                 const int32_t* context_lens, int32_t n_seqs, float scale, void* out,
                                                 void* stream) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (layer < 0 || layer >= d->n_layers || n_seqs < 0) return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0) return PKV_OK;
    if (max_blocks_per_seq <= 0 || max_blocks_per_seq > (1 << 24)) return PKV_ERR_INVALID_ARG;
    if (n_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;

    const long long rows = (long long)d->num_blocks * d->n_kv_heads * d->block_size;
    if (d->dtype != PKV_F32 && rows >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;  // tensor-copy rows are 32-bit
    // Same partition geometry, hence the same scratch need, as pkv_paged_decode_attention.
    int bpp = 0, n_parts = 0;
    if (pkv::decode_geometry(d, rows, n_seqs, max_blocks_per_seq, &bpp, &n_parts) != cudaSuccess)
        return PKV_ERR_CUDA;
    size_t off_ml = 0, off_cnt = 0;
    const size_t need =
        pkv::decode_workspace_layout(n_seqs, d->n_q_heads, d->n_kv_heads, d->head_dim, n_parts, &off_ml, &off_cnt);
    if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_UNSUPPORTED;  // too big for the fixed scratch

    float* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return PKV_ERR_CUDA;

    pkv::DecodeArgs a;
    const size_t layer_bytes =
        (size_t)d->num_blocks * d->n_kv_heads * d->block_size * d->head_dim * elem_bytes(d->dtype);
    a.q = q;
    a.k_layer = static_cast<const char*>(k_pool) + (size_t)layer * layer_bytes;
    a.v_layer = static_cast<const char*>(v_pool) + (size_t)layer * layer_bytes;
    a.tables = block_tables;
    a.lens = context_lens;
    a.out = out;
    // Every partial the merge reads is written earlier in the same call, so stale partials from an
    // earlier call are never read; the arrival counters carry this call's tag, so whatever an
    // earlier call left in the array (counters or partials of another geometry) reads as zero.
    a.part_o = need ? scratch : nullptr;
    a.part_ml = need ? reinterpret_cast<float*>(reinterpret_cast<char*>(scratch) + off_ml) : nullptr;
    a.counters = need ? reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(scratch) + off_cnt) : nullptr;
    a.call_tag = pkv::next_call_tag();
    a.n_seqs = n_seqs;
    a.n_q = d->n_q_heads;
    a.n_kv = d->n_kv_heads;
    a.num_blocks = d->num_blocks;
    a.max_blocks = max_blocks_per_seq;
    a.n_parts = n_parts;
    a.bpp = bpp;
    a.scale_log2 = scale * 1.4426950408889634f;
    if (pkv::device_status_word(&a.status) != cudaSuccess) return PKV_ERR_CUDA;
    int launches = 0;
    cudaError_t err = pkv::launch_decode(d->dtype, d->head_dim, d->n_q_heads / d->n_kv_heads, a,
                                         static_cast<cudaStream_t>(stream), &launches);
    pkv::count_launches((uint64_t)launches);
    return pkv::launch_status(err);
}
