// internal.h -- declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kBlock = 16;  // tokens per block; the only block size compiled

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
    unsigned int* status;   // device status word
    int n_seqs, n_q, n_kv, num_blocks, max_blocks;
    int n_parts;            // partitions per sequence row of the grid
    int bpp;                // blocks per partition
    float scale_log2;       // scale * log2(e): logits are kept in base 2
};

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

// Partition geometry shared by the workspace query and the launch.
int decode_blocks_per_partition(int n_seqs, int n_kv, int max_blocks);
inline int decode_partitions(int max_blocks, int bpp) { return (max_blocks + bpp - 1) / bpp; }

// Launchers (decode_*.cu, append_copy.cu). Return the first CUDA error, or cudaSuccess.
cudaError_t launch_decode(int dtype, int head_dim, int group, const DecodeArgs& a, cudaStream_t stream,
                          int* n_launches);
cudaError_t launch_decode_f32(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches);
cudaError_t launch_decode_f16(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches);
cudaError_t launch_decode_bf16(int head_dim, int group, const DecodeArgs& a, cudaStream_t stream, int* n_launches);
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream);

// Shared with decode_static.cu (abi.cu owns both): the current device's status word, and the
// process-wide count of kernels launched by this library.
cudaError_t device_status_word(unsigned int** out);
void count_launches(uint64_t n);

}  // namespace pkv
