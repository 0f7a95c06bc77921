// internal.h -- declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kBlock = 16;  // tokens per block; the only block size compiled
constexpr int kMaxBpp = 64; // largest partition (table entries per CTA); decode kernels stage them in smem

// Arguments of one paged decode attention launch (one layer). Pointers are device pointers
// already offset to the layer; element types are fixed by the template instantiation.
struct DecodeArgs {
    const void* q;          // [n_seqs][n_q][D]
    const void* k_layer;    // [num_blocks][n_kv][16][D]
    const void* v_layer;
    const int32_t* tables;  // [n_seqs][max_blocks]
    const int32_t* lens;    // [n_seqs]
    void* out;              // [n_seqs][n_q][D]
    float* part_o;          // [n_seqs][n_q][n_parts][D]   (split-K only)
    float* part_ml;         // [n_seqs][n_q][n_parts][2]   (running max, sum)
    unsigned long long* counters = nullptr;  // [n_seqs][n_kv] partition arrivals: (call tag << 24) | count
    unsigned long long call_tag = 0;         // 1 .. 2^40-1, distinct for consecutive calls
    const void* k_new = nullptr;       // fused append: [n_seqs][n_kv][D] rows of position ctx-1,
    const void* v_new = nullptr;       // written before attention; nullptr = no append
    unsigned int* status;   // device status word
    int n_seqs, n_q, n_kv, num_blocks, max_blocks;
    int n_parts;            // partitions per sequence row of the grid
    int bpp;                // blocks per partition
    float scale_log2;       // scale * log2(e): logits are kept in base 2
    bool overlap_previous = false;  // launch as a programmatic dependent of the previous kernel
    // Dense cache instead of a paged pool: k_layer / v_layer are [n_seqs][n_kv][max_blocks*16][D],
    // logical block i of sequence s is chunk (s*n_kv + g)*max_blocks + i (the identity walk, no
    // table); tables is unused and num_blocks = n_seqs * max_blocks (the same row count).
    bool dense = false;
};

// Arguments of one paged prefill attention launch (one layer). q / out hold the chunk tokens of
// all sequences packed in order: sequence s owns rows q_start[s] .. q_start[s+1]-1.
struct PrefillArgs {
    const void* q;          // [n_tokens][n_q][D]
    void* out;              // [n_tokens][n_q][D]
    const void* k_layer;    // [num_blocks][n_kv][16][D] (the CUDA-core kernel; the MMA kernel uses
    const void* v_layer;    //  tensor maps of the same layer)
    const int32_t* tables;  // [n_seqs][max_blocks]
    const int32_t* lens;    // [n_seqs] context lengths after the chunk
    const int32_t* q_start; // [n_seqs + 1]
    unsigned int* status;
    int n_seqs, n_q, n_kv, num_blocks, max_blocks, n_tokens;
    int q_tiles;            // CTAs along the chunk: ceil(max query length / tokens per CTA)
    float scale_log2;       // scale * log2(e)
    bool overlap_previous = false;  // launch as a programmatic dependent of the previous kernel
};

// Query rows (token x head-in-group) one prefill CTA covers; tokens per CTA = rows / group.
// tcgen05 kernel (fp16 / bf16): 128 rows, the M of one tensor-core instruction (one TMEM lane per
// row). CUDA-core kernel (fp32): 32 rows.
constexpr int kPrefillRowsUmma = 128;
constexpr int kPrefillRowsF32 = 32;
inline int prefill_tokens_per_cta(int dtype, int head_dim, int group) {
    (void)head_dim;
    return (dtype == PKV_F32 ? kPrefillRowsF32 : kPrefillRowsUmma) / group;
}

struct AppendArgs {
    const void* k;          // [n_tok][n_kv][D]
    const void* v;
    const int64_t* slots;   // [n_tok]
    void* k_layer;          // [num_blocks][n_kv][16][D]
    void* v_layer;
    unsigned int* status;
    int n_tok, n_kv, num_blocks;
    int row_bytes;          // D * element bytes
};

struct CopyArgs {
    void* k_pool;           // whole pools
    void* v_pool;
    const int32_t* pairs;   // [n_pairs][2]
    unsigned int* status;
    int n_pairs, n_layers, num_blocks;
    size_t block_bytes;     // n_kv * 16 * D * element bytes (one block of one layer)
    size_t layer_bytes;     // num_blocks * block_bytes
};

// Partition geometry shared by the workspace query and the launch. sm_count is the device's
// multiprocessor count, ctas_per_sm the number of CTAs of the chosen decode kernel one SM holds at
// once, max_bpp the largest partition that kernel takes (decode_max_bpp).
int decode_blocks_per_partition(int n_seqs, int n_kv, int max_blocks, int sm_count, int ctas_per_sm, int max_bpp);
cudaError_t current_sm_count(int* out);
// CTAs per SM of the decode kernel a call of this shape runs (pool rows decide the kernel, as in
// decode_uses_mma), measured by the occupancy calculator on the current device.
cudaError_t decode_ctas_per_sm(int dtype, int head_dim, int group, long long rows, int* out);
cudaError_t decode_ctas_per_sm_f32(int head_dim, int group, long long rows, int* out);
cudaError_t decode_ctas_per_sm_f16(int head_dim, int group, long long rows, int* out);
cudaError_t decode_ctas_per_sm_bf16(int head_dim, int group, long long rows, int* out);
// The geometry of a decode call on the current device (SM count and occupancy read once per device
// and kernel, then cached): blocks per partition and partitions per sequence.
cudaError_t decode_geometry(const pkv_cache_desc* d, long long rows, int n_seqs, int max_blocks, int* bpp,
                            int* n_parts);
inline int decode_partitions(int max_blocks, int bpp) { return (max_blocks + bpp - 1) / bpp; }

// Split-K workspace layout (0 bytes when n_parts <= 1): fp32 partial outputs
// [n_seqs][n_q][n_parts][D], then (max, sum) pairs [n_seqs][n_q][n_parts][2] at *off_ml, then the
// 64-bit arrival counters [n_seqs][n_kv] at *off_cnt (16-byte aligned). Returns the total bytes.
inline size_t decode_workspace_layout(int n_seqs, int n_q, int n_kv, int head_dim, int n_parts, size_t* off_ml,
                                      size_t* off_cnt) {
    *off_ml = *off_cnt = 0;
    if (n_parts <= 1) return 0;
    const size_t o = (size_t)n_seqs * n_q * n_parts * head_dim * sizeof(float);
    const size_t ml = (size_t)n_seqs * n_q * n_parts * 2 * sizeof(float);
    const size_t cnt = (size_t)n_seqs * n_kv * sizeof(unsigned long long);
    *off_ml = o;
    *off_cnt = (o + ml + 15) / 16 * 16;
    return *off_cnt + (cnt + 15) / 16 * 16;
}

// Launchers (decode_*.cu, append_copy.cu). Return the first CUDA error, or cudaSuccess.
cudaError_t launch_decode(int dtype, int head_dim, int group, const DecodeArgs& a, cudaStream_t stream,
                          int* n_launches);
cudaError_t launch_decode_f32(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches);
cudaError_t launch_decode_f16(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches);
cudaError_t launch_decode_bf16(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches);
cudaError_t launch_prefill(int dtype, int head_dim, int group, const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_f32(int head_dim, int group, const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_f16(int head_dim, int group, const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_bf16(int head_dim, int group, const PrefillArgs& a, cudaStream_t stream);
// CTAs of the prefill kernel of this shape that the current device (sms SMs) holds at once: the
// occupancy calculator per SM, tensor memory included, and for CTA pairs the clusters the GPU can
// place at once.
cudaError_t prefill_wave_ctas(int dtype, int head_dim, int group, int sms, int* out);
cudaError_t prefill_wave_ctas_f16(int head_dim, int group, int sms, int* out);
cudaError_t prefill_wave_ctas_bf16(int head_dim, int group, int sms, int* out);
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream);
// dst device, src device-visible page-locked host memory; both 16-byte aligned, bytes % 4 == 0.
cudaError_t launch_upload_metadata(void* dst, const void* src, size_t bytes, cudaStream_t stream);

// Tensor-core decode (decode_mma.cuh) serves 16-bit storage when G >= kMmaMinGroup and the pool's
// rows fit the 32-bit TMA row coordinate; everything else runs the CUDA-core kernel (decode.cuh).
constexpr int kMmaMinGroup = 1;
inline bool decode_uses_mma(int dtype, int group, long long rows) {
    return dtype != PKV_F32 && group >= kMmaMinGroup && rows < (1LL << 31);
}
// Largest partition (table entries per CTA) of the chosen kernel: the CUDA-core kernel stages a
// partition's entries in shared memory (kMaxBpp of them); the tensor-core kernel streams them
// through registers and takes any length.
constexpr int kMaxBppStreamed = 1 << 24;
inline int decode_max_bpp(int dtype, int group, long long rows) {
    return decode_uses_mma(dtype, group, rows) ? kMaxBppStreamed : kMaxBpp;
}

// Status of a launcher's result: a pool address the tensor maps refused (not device memory of the
// current device) is the caller's argument error; anything else from CUDA is PKV_ERR_CUDA.
inline int launch_status(cudaError_t err) {
    if (err == cudaSuccess) return PKV_OK;
    return err == cudaErrorInvalidDevicePointer ? PKV_ERR_INVALID_ARG : PKV_ERR_CUDA;
}

// Cached TMA tensor map of one pool layer seen as rows x head_dim 16-bit elements (tmap.cu).
enum { PKV_BOX_PANEL = 0, PKV_BOX_BLOCK = 1, PKV_BOX_BLOCK_HALF = 2 };
cudaError_t kv_tensor_map(const void* layer_base, long long rows, int head_dim, int dtype, int box, CUtensorMap* out);

// Shared with decode_static.cu (abi.cu owns both): the current device's status word, and the
// process-wide count of kernels launched by this library.
cudaError_t device_status_word(unsigned int** out);
void count_launches(uint64_t n);
// A fresh tag for one decode call's split-K arrival counters (never 0, wraps below 2^40).
unsigned long long next_call_tag();

}  // namespace pkv
