// abi.cu -- the C ABI of libpkv: argument validation, dispatch, device status word.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// Device status word: kernels OR PKV_DEV_* bits into it when they skip a bad device-side value.
__device__ unsigned int g_dev_status;

// One thread waits (bounded) on an mbarrier that expects an arrival nobody makes.
__global__ void wait_timeout_selftest_kernel(unsigned int* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    pkv::mbar_init(&bar, 1);
    pkv::fence_mbar_init();
    if (!pkv::mbar_wait_bounded(&bar, 0u)) atomicOr(status, (unsigned)PKV_DEV_WAIT_TIMEOUT);
}

std::atomic<uint64_t> g_launches{0};
std::mutex g_status_mu;
unsigned int* g_status_addr[64] = {};

// Device address of this device's status word (resolved once per device).
cudaError_t status_word(unsigned int** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_dev_status);
        if (err != cudaSuccess) return err;
        g_status_addr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_status_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

size_t layer_elems(const pkv_cache_desc* d) {
    return (size_t)d->num_blocks * d->n_kv_heads * d->block_size * d->head_dim;
}

// Workspace of a decode call with partitions of `bpp` table entries.
size_t decode_workspace(const pkv_cache_desc* d, int n_seqs, int max_blocks, int bpp, int* n_parts_out,
                        size_t* off_ml = nullptr, size_t* off_cnt = nullptr) {
    const int n_parts = pkv::decode_partitions(max_blocks, bpp);
    if (n_parts_out) *n_parts_out = n_parts;
    size_t ml = 0, cnt = 0;
    const size_t bytes =
        pkv::decode_workspace_layout(n_seqs, d->n_q_heads, d->n_kv_heads, d->head_dim, n_parts, &ml, &cnt);
    if (off_ml) *off_ml = ml;
    if (off_cnt) *off_cnt = cnt;
    return bytes;
}

long long pool_rows(const pkv_cache_desc* d) { return (long long)d->num_blocks * d->n_kv_heads * d->block_size; }

std::mutex g_sm_mu;
int g_sm_count[64] = {};
// CTAs per SM of each decode kernel: [device][dtype][head_dim 64/128/256][group 1/2/4/8][tensor-core path]
int g_ctas_per_sm[64][3][3][4][2] = {};

int dim_index(int head_dim) { return head_dim == 64 ? 0 : head_dim == 128 ? 1 : 2; }
int group_index(int g) { return g == 1 ? 0 : g == 2 ? 1 : g == 4 ? 2 : 3; }

}  // namespace

namespace pkv {

// Blocks per partition.
//  * One wave: when the grid's (sequence, KV head) pairs are fewer than the CTAs the GPU holds at
//    once, each pair takes parts = slots / pairs CTAs; if that fills at least 3/4 of the slots with
//    long partitions (>= 64 entries, which the tensor-core kernel streams), every context is cut
//    into `parts` equal partitions and the launch is one wave of equal CTAs: no CTA starts after
//    another has finished, so no SM idles through a tail while the last ones run (long documents:
//    10 sequences x 4 KV heads spread over 11 CTAs each instead of 2.9 waves of 33).
//  * Otherwise 64 entries (1,024 tokens), halved (down to 4) while the grid would hold fewer than
//    ~4 CTAs per SM, to spread a few long sequences over more SMs.
// Depends only on the arguments, so the workspace query and the launch agree as long as both pass
// the same device facts (both take them from decode_geometry).
int decode_blocks_per_partition(int n_seqs, int n_kv, int max_blocks, int sm_count, int ctas_per_sm, int max_bpp) {
    const long long pairs = (long long)n_seqs * n_kv;
    const long long sms = sm_count > 0 ? sm_count : 1;
    const long long slots = sms * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    if (pairs > 0 && pairs < slots) {
        const long long parts = slots / pairs;
        const long long bpp1 = (max_blocks + parts - 1) / parts;
        if (4 * pairs * parts >= 3 * slots && bpp1 >= kMaxBpp && bpp1 <= max_bpp) return (int)bpp1;
    }
    const long long target = 4LL * sms;
    int bpp = kMaxBpp;
    while (bpp > 4 && pairs * ((max_blocks + bpp - 1) / bpp) < target) bpp /= 2;
    return bpp < max_bpp ? bpp : max_bpp;
}

// SMs of the current device (cudaDevAttrMultiProcessorCount), read once per device.
cudaError_t current_sm_count(int* out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_sm_mu);
    if (g_sm_count[dev] <= 0) {
        int n = 0;
        err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        if (n <= 0) return cudaErrorInvalidValue;
        g_sm_count[dev] = n;
    }
    *out = g_sm_count[dev];
    return cudaSuccess;
}

cudaError_t decode_ctas_per_sm(int dtype, int head_dim, int group, long long rows, int* out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64 || dtype < 0 || dtype > 2) return cudaErrorInvalidValue;
    int& slot = g_ctas_per_sm[dev][dtype][dim_index(head_dim)][group_index(group)][decode_uses_mma(dtype, group, rows)];
    {
        std::lock_guard<std::mutex> lock(g_sm_mu);
        if (slot > 0) {
            *out = slot;
            return cudaSuccess;
        }
    }
    int n = 0;
    switch (dtype) {
    case PKV_F32: err = decode_ctas_per_sm_f32(head_dim, group, rows, &n); break;
    case PKV_F16: err = decode_ctas_per_sm_f16(head_dim, group, rows, &n); break;
    default: err = decode_ctas_per_sm_bf16(head_dim, group, rows, &n); break;
    }
    if (err != cudaSuccess) return err;
    if (n <= 0) return cudaErrorInvalidConfiguration;  // the kernel does not fit on an SM
    std::lock_guard<std::mutex> lock(g_sm_mu);
    slot = n;
    *out = n;
    return cudaSuccess;
}

cudaError_t decode_geometry(const pkv_cache_desc* d, long long rows, int n_seqs, int max_blocks, int* bpp,
                            int* n_parts) {
    int sms = 0, per_sm = 0;
    const int group = d->n_q_heads / d->n_kv_heads;
    cudaError_t err = current_sm_count(&sms);
    if (err == cudaSuccess) err = decode_ctas_per_sm(d->dtype, d->head_dim, group, rows, &per_sm);
    if (err != cudaSuccess) return err;
    *bpp = decode_blocks_per_partition(n_seqs, d->n_kv_heads, max_blocks, sms, per_sm,
                                       decode_max_bpp(d->dtype, group, rows));
    *n_parts = decode_partitions(max_blocks, *bpp);
    return cudaSuccess;
}

cudaError_t device_status_word(unsigned int** out) { return status_word(out); }

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

unsigned long long next_call_tag() {
    static std::atomic<unsigned long long> tag{0};
    unsigned long long t;
    do {
        t = (tag.fetch_add(1, std::memory_order_relaxed) + 1) & ((1ull << 40) - 1);
    } while (t == 0);
    return t;
}

cudaError_t launch_decode(int dtype, int head_dim, int group, const DecodeArgs& a, cudaStream_t stream,
                          int* n_launches) {
    switch (dtype) {
    case PKV_F32: return launch_decode_f32(head_dim, group, a, stream, n_launches);
    case PKV_F16: return launch_decode_f16(head_dim, group, a, stream, n_launches);
    case PKV_BF16: return launch_decode_bf16(head_dim, group, a, stream, n_launches);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv

extern "C" {

const char* pkv_status_str(int status) {
    switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG: invalid argument";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: shape outside the compiled set";
    case PKV_ERR_NO_BLOCKS: return "PKV_ERR_NO_BLOCKS: not enough free blocks";
    case PKV_ERR_BAD_STATE: return "PKV_ERR_BAD_STATE: internal inconsistency";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA runtime call failed";
    default: return "unknown pkv status";
    }
}

int pkv_validate_desc(const pkv_cache_desc* d) {
    if (!d) return PKV_ERR_INVALID_ARG;
    if (d->n_layers <= 0 || d->num_blocks <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 ||
        d->block_size <= 0)
        return PKV_ERR_INVALID_ARG;
    if (d->dtype != PKV_F32 && d->dtype != PKV_F16 && d->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (d->block_size != pkv::kBlock) return PKV_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return PKV_ERR_UNSUPPORTED;
    if (d->n_q_heads % d->n_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
    const int G = d->n_q_heads / d->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

uint64_t pkv_bytes_per_token(const pkv_cache_desc* d) {
    if (pkv_validate_desc(d) != PKV_OK) return 0;
    return 2ull * (uint64_t)d->n_layers * (uint64_t)d->n_kv_heads * (uint64_t)d->head_dim * elem_bytes(d->dtype);
}

uint64_t pkv_pool_bytes(const pkv_cache_desc* d) {
    if (pkv_validate_desc(d) != PKV_OK) return 0;
    return (uint64_t)d->n_layers * layer_elems(d) * elem_bytes(d->dtype);
}

int pkv_decode_split_geometry(const pkv_cache_desc* d, int32_t n_seqs, int32_t max_blocks_per_seq,
                              int32_t sm_count, int32_t ctas_per_sm, int32_t* blocks_per_partition,
                              int32_t* n_partitions, size_t* workspace_bytes) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (n_seqs <= 0 || max_blocks_per_seq <= 0 || sm_count <= 0 || ctas_per_sm <= 0) return PKV_ERR_INVALID_ARG;
    const int group = d->n_q_heads / d->n_kv_heads;
    const int bpp = pkv::decode_blocks_per_partition(n_seqs, d->n_kv_heads, max_blocks_per_seq, sm_count, ctas_per_sm,
                                                     pkv::decode_max_bpp(d->dtype, group, pool_rows(d)));
    int n_parts = 0;
    const size_t bytes = decode_workspace(d, n_seqs, max_blocks_per_seq, bpp, &n_parts);
    if (blocks_per_partition) *blocks_per_partition = bpp;
    if (n_partitions) *n_partitions = n_parts;
    if (workspace_bytes) *workspace_bytes = bytes;
    return PKV_OK;
}

int pkv_decode_ctas_per_sm(const pkv_cache_desc* d, int32_t* ctas_per_sm, int32_t* sm_count) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    int sms = 0, per_sm = 0;
    if (pkv::current_sm_count(&sms) != cudaSuccess ||
        pkv::decode_ctas_per_sm(d->dtype, d->head_dim, d->n_q_heads / d->n_kv_heads, pool_rows(d), &per_sm) !=
            cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (ctas_per_sm) *ctas_per_sm = per_sm;
    if (sm_count) *sm_count = sms;
    return PKV_OK;
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* d, int32_t n_seqs, int32_t max_blocks_per_seq) {
    if (pkv_validate_desc(d) != PKV_OK || n_seqs <= 0 || max_blocks_per_seq <= 0) return 0;
    int bpp = 0, n_parts = 0;
    if (pkv::decode_geometry(d, pool_rows(d), n_seqs, max_blocks_per_seq, &bpp, &n_parts) != cudaSuccess) {
        cudaGetLastError();  // no usable device: report nothing rather than a guess
        return 0;
    }
    return decode_workspace(d, n_seqs, max_blocks_per_seq, bpp, nullptr);
}

int pkv_kv_append(const pkv_cache_desc* d, int32_t layer, const void* k, const void* v, const int64_t* slot_mapping,
                  int32_t n_tokens, void* k_pool, void* v_pool, void* stream) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (layer < 0 || layer >= d->n_layers || n_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (n_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;
    pkv::AppendArgs a;
    a.k = k;
    a.v = v;
    a.slots = slot_mapping;
    const size_t layer_bytes = layer_elems(d) * elem_bytes(d->dtype);
    a.k_layer = static_cast<char*>(k_pool) + (size_t)layer * layer_bytes;
    a.v_layer = static_cast<char*>(v_pool) + (size_t)layer * layer_bytes;
    a.n_tok = n_tokens;
    a.n_kv = d->n_kv_heads;
    a.num_blocks = d->num_blocks;
    a.row_bytes = d->head_dim * (int)elem_bytes(d->dtype);
    if (status_word(&a.status) != cudaSuccess) return PKV_ERR_CUDA;
    if (pkv::launch_append(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PKV_OK;
}

// Shared body of the decode entry points; k_new / v_new are null unless the append is fused. With
// `dense`, k_pool / v_pool are dense caches [n_layers][n_seqs][n_kv][max_blocks*16][D] walked by
// identity (block_tables unused) instead of paged pools.
static int decode_call(uint32_t flags, const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_new,
                       const void* v_new,
                       const void* k_pool, const void* v_pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t n_seqs, float scale, void* out, void* workspace,
                       size_t workspace_bytes, void* stream, bool dense = false) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (layer < 0 || layer >= d->n_layers || n_seqs < 0) return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0) return PKV_OK;
    if (max_blocks_per_seq <= 0 || max_blocks_per_seq > (1 << 24)) return PKV_ERR_INVALID_ARG;
    if (n_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (dense && (long long)n_seqs * max_blocks_per_seq >= (1LL << 31) / (long long)(d->n_kv_heads * d->block_size))
        return PKV_ERR_UNSUPPORTED;  // chunk and row indices of the dense cache are 32-bit
    if (!q || !k_pool || !v_pool || (!block_tables && !dense) || !context_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;
    if ((k_new || v_new) && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;
    // a dense layer holds n_seqs * max_blocks 16-row chunks per KV head: the pool geometry with
    // num_blocks = n_seqs * max_blocks
    const int num_blocks = dense ? n_seqs * max_blocks_per_seq : d->num_blocks;
    const long long rows = (long long)num_blocks * d->n_kv_heads * d->block_size;
    if (d->dtype != PKV_F32 && rows >= (1LL << 31)) return PKV_ERR_UNSUPPORTED;  // tensor-copy rows are 32-bit
    int bpp = 0, n_parts = 0;
    if (pkv::decode_geometry(d, rows, n_seqs, max_blocks_per_seq, &bpp, &n_parts) != cudaSuccess) return PKV_ERR_CUDA;
    size_t off_ml = 0, off_cnt = 0;
    const size_t need = decode_workspace(d, n_seqs, max_blocks_per_seq, bpp, &n_parts, &off_ml, &off_cnt);
    if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need)) return PKV_ERR_INVALID_ARG;

    pkv::DecodeArgs a;
    const size_t layer_bytes =
        (size_t)num_blocks * d->n_kv_heads * d->block_size * d->head_dim * elem_bytes(d->dtype);
    a.q = q;
    a.k_layer = static_cast<const char*>(k_pool) + (size_t)layer * layer_bytes;
    a.v_layer = static_cast<const char*>(v_pool) + (size_t)layer * layer_bytes;
    a.tables = dense ? nullptr : block_tables;
    a.dense = dense;
    a.lens = context_lens;
    a.out = out;
    a.part_o = need ? static_cast<float*>(workspace) : nullptr;
    a.part_ml = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) + off_ml) : nullptr;
    a.counters = need ? reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + off_cnt) : nullptr;
    a.call_tag = pkv::next_call_tag();
    a.k_new = k_new;
    a.v_new = v_new;
    a.n_seqs = n_seqs;
    a.n_q = d->n_q_heads;
    a.n_kv = d->n_kv_heads;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks_per_seq;
    a.n_parts = n_parts;
    a.bpp = bpp;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.overlap_previous = (flags & PKV_DECODE_OVERLAP_PREVIOUS) != 0 && d->dtype != PKV_F32;
    if (status_word(&a.status) != cudaSuccess) return PKV_ERR_CUDA;
    int launches = 0;
    cudaError_t err = pkv::launch_decode(d->dtype, d->head_dim, d->n_q_heads / d->n_kv_heads, a,
                                         static_cast<cudaStream_t>(stream), &launches);
    g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
    return pkv::launch_status(err);
}

int pkv_paged_decode_attention(const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_pool,
                               const void* v_pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t n_seqs, float scale, void* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return decode_call(0u, d, layer, q, nullptr, nullptr, k_pool, v_pool, block_tables, max_blocks_per_seq,
                       context_lens, n_seqs, scale, out, workspace, workspace_bytes, stream);
}

int pkv_paged_decode_append_attention(const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_new,
                                      const void* v_new, void* k_pool, void* v_pool, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t n_seqs,
                                      float scale, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (n_seqs > 0 && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
    return decode_call(0u, d, layer, q, k_new, v_new, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens,
                       n_seqs, scale, out, workspace, workspace_bytes, stream);
}

int pkv_paged_decode_append_attention_ex(const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_new,
                                         const void* v_new, void* k_pool, void* v_pool, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t n_seqs,
                                         float scale, void* out, void* workspace, size_t workspace_bytes,
                                         uint32_t flags, void* stream) {
    if (flags & ~(uint32_t)PKV_DECODE_OVERLAP_PREVIOUS) return PKV_ERR_INVALID_ARG;
    if (n_seqs > 0 && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
    return decode_call(flags, d, layer, q, k_new, v_new, k_pool, v_pool, block_tables, max_blocks_per_seq,
                       context_lens, n_seqs, scale, out, workspace, workspace_bytes, stream);
}

int pkv_dense_decode_attention(const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_cache,
                               const void* v_cache, int32_t max_seq_len, const int32_t* context_lens, int32_t n_seqs,
                               float scale, void* out, void* workspace, size_t workspace_bytes, uint32_t flags,
                               void* stream) {
    if (flags & ~(uint32_t)PKV_DECODE_OVERLAP_PREVIOUS) return PKV_ERR_INVALID_ARG;
    if (!d || max_seq_len <= 0 || max_seq_len % pkv::kBlock != 0) return PKV_ERR_INVALID_ARG;
    return decode_call(flags, d, layer, q, nullptr, nullptr, k_cache, v_cache, nullptr, max_seq_len / pkv::kBlock,
                       context_lens, n_seqs, scale, out, workspace, workspace_bytes, stream, true);
}

static int prefill_call(uint32_t flags, const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_pool,
                        const void* v_pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, const int32_t* query_start, int32_t n_seqs, int32_t n_tokens,
                        int32_t max_query_len, float scale, void* out, void* stream) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (layer < 0 || layer >= d->n_layers || n_seqs < 0 || n_tokens < 0 || max_query_len < 0 ||
        max_query_len > n_tokens)
        return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0 || max_query_len == 0) return PKV_OK;
    if (max_blocks_per_seq <= 0 || max_blocks_per_seq > (1 << 24)) return PKV_ERR_INVALID_ARG;
    if (n_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (d->dtype != PKV_F32 && (long long)d->num_blocks * d->n_kv_heads * d->block_size >= (1LL << 31))
        return PKV_ERR_UNSUPPORTED;  // tensor-copy row coordinates are 32-bit
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !query_start || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;

    pkv::PrefillArgs a;
    const size_t layer_bytes = layer_elems(d) * elem_bytes(d->dtype);
    const int group = d->n_q_heads / d->n_kv_heads;
    const int per_cta = pkv::prefill_tokens_per_cta(d->dtype, d->head_dim, group);
    a.q = q;
    a.out = out;
    a.k_layer = static_cast<const char*>(k_pool) + (size_t)layer * layer_bytes;
    a.v_layer = static_cast<const char*>(v_pool) + (size_t)layer * layer_bytes;
    a.tables = block_tables;
    a.lens = context_lens;
    a.q_start = query_start;
    a.n_seqs = n_seqs;
    a.n_q = d->n_q_heads;
    a.n_kv = d->n_kv_heads;
    a.num_blocks = d->num_blocks;
    a.max_blocks = max_blocks_per_seq;
    a.n_tokens = n_tokens;
    a.q_tiles = (max_query_len + per_cta - 1) / per_cta;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.overlap_previous = (flags & PKV_PREFILL_OVERLAP_PREVIOUS) != 0 && d->dtype != PKV_F32;
    if (status_word(&a.status) != cudaSuccess) return PKV_ERR_CUDA;
    cudaError_t err = pkv::launch_prefill(d->dtype, d->head_dim, group, a, static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return pkv::launch_status(err);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PKV_OK;
}

int pkv_paged_prefill_attention(const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_pool,
                                const void* v_pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, const int32_t* query_start, int32_t n_seqs,
                                int32_t n_tokens, int32_t max_query_len, float scale, void* out, void* stream) {
    return prefill_call(0u, d, layer, q, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens, query_start,
                        n_seqs, n_tokens, max_query_len, scale, out, stream);
}

int pkv_paged_prefill_attention_ex(const pkv_cache_desc* d, int32_t layer, const void* q, const void* k_pool,
                                   const void* v_pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* query_start, int32_t n_seqs,
                                   int32_t n_tokens, int32_t max_query_len, float scale, void* out, uint32_t flags,
                                   void* stream) {
    if (flags & ~(uint32_t)PKV_PREFILL_OVERLAP_PREVIOUS) return PKV_ERR_INVALID_ARG;
    return prefill_call(flags, d, layer, q, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens,
                        query_start, n_seqs, n_tokens, max_query_len, scale, out, stream);
}

int pkv_prefill_wave_tokens(const pkv_cache_desc* d, int32_t* tokens) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (!tokens) return PKV_ERR_INVALID_ARG;
    int sms = 0, wave = 0;
    const int group = d->n_q_heads / d->n_kv_heads;
    if (pkv::current_sm_count(&sms) != cudaSuccess ||
        pkv::prefill_wave_ctas(d->dtype, d->head_dim, group, sms, &wave) != cudaSuccess || wave <= 0) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    // a CTA holds the rows of prefill_tokens_per_cta tokens of one KV head
    const long long t = (long long)wave * pkv::prefill_tokens_per_cta(d->dtype, d->head_dim, group) / d->n_kv_heads;
    *tokens = (int32_t)(t > 0 ? t : 1);
    return PKV_OK;
}

int pkv_copy_blocks(const pkv_cache_desc* d, void* k_pool, void* v_pool, const int32_t* pairs, int32_t n_pairs,
                    void* stream) {
    int rc = pkv_validate_desc(d);
    if (rc != PKV_OK) return rc;
    if (n_pairs < 0) return PKV_ERR_INVALID_ARG;
    if (n_pairs == 0) return PKV_OK;
    if (!k_pool || !v_pool || !pairs) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;
    if (d->n_layers > 65535) return PKV_ERR_UNSUPPORTED;
    pkv::CopyArgs a;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.pairs = pairs;
    a.n_pairs = n_pairs;
    a.n_layers = d->n_layers;
    a.num_blocks = d->num_blocks;
    a.block_bytes = (size_t)d->n_kv_heads * d->block_size * d->head_dim * elem_bytes(d->dtype);
    a.layer_bytes = a.block_bytes * (size_t)d->num_blocks;
    if (status_word(&a.status) != cudaSuccess) return PKV_ERR_CUDA;
    if (pkv::launch_copy_blocks(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PKV_OK;
}

int pkv_upload_metadata(void* dst, const void* src_host, size_t bytes, void* stream) {
    if (bytes == 0) return PKV_OK;
    if (!dst || !src_host || bytes % 4 != 0 || !aligned16(dst) || !aligned16(src_host)) return PKV_ERR_INVALID_ARG;
    if (bytes > ((size_t)1 << 30)) return PKV_ERR_INVALID_ARG;
    cudaPointerAttributes sa{}, da{};
    if (cudaPointerGetAttributes(&sa, src_host) != cudaSuccess) {
        cudaGetLastError();  // an unregistered pointer is an argument error, not a sticky one
        return PKV_ERR_INVALID_ARG;
    }
    if (cudaPointerGetAttributes(&da, dst) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_INVALID_ARG;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (sa.type != cudaMemoryTypeHost || !sa.devicePointer) return PKV_ERR_INVALID_ARG;
    if (da.type != cudaMemoryTypeDevice || da.device != dev) return PKV_ERR_INVALID_ARG;
    // the kernel reads through the device's view of the host buffer (the same address under
    // unified addressing); it must keep the 16-byte alignment the vector loads need
    if (!aligned16(sa.devicePointer)) return PKV_ERR_INVALID_ARG;
    if (pkv::launch_upload_metadata(dst, sa.devicePointer, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PKV_OK;
}

int pkv_get_device_status(void* stream, uint32_t* flags) {
    if (!flags) return PKV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    unsigned int* addr = nullptr;
    if (status_word(&addr) != cudaSuccess) return PKV_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, addr, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemset(addr, 0, sizeof(v)) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    *flags = v;
    return PKV_OK;
}

uint64_t pkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int pkv_selftest_wait_timeout(void* stream) {
    unsigned int* status = nullptr;
    if (status_word(&status) != cudaSuccess) return PKV_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PKV_OK;
}

}  // extern "C"
