// tmap.cu -- TMA tensor maps over one layer of a K or V pool (host side).
//
// A pool layer [num_blocks][n_kv][16][D] of 16-bit elements is described as a 2-D tensor of
// num_blocks*n_kv*16 rows by D columns; the decode kernel copies 64-column x 16-row boxes (one
// panel of one (block, KV head) chunk) with the 128-byte swizzle. Encoding goes through the driver
// entry point cuTensorMapEncodeTiled, found once through the runtime; maps are cached by
// (address, shape, type, device) so steady-state calls do not re-encode.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace pkv {
namespace {

struct MapEntry {
    const void* base;
    long long rows;
    int head_dim;
    int dtype;
    int device;
    unsigned long long stamp;  // 0 = empty slot; else last use (least recently used is replaced)
    CUtensorMap map;
};

std::mutex g_map_mu;
MapEntry g_maps[64];
unsigned long long g_clock = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (err != cudaSuccess) return err;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}

}  // namespace

cudaError_t kv_tensor_map(const void* layer_base, long long rows, int head_dim, int dtype, CUtensorMap* out) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return cudaErrorInvalidValue;
    if (rows <= 0 || rows >= (1LL << 31) || (head_dim % 64) != 0) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_map_mu);
    MapEntry* victim = &g_maps[0];
    for (MapEntry& e : g_maps) {
        if (e.stamp && e.base == layer_base && e.rows == rows && e.head_dim == head_dim && e.dtype == dtype &&
            e.device == dev) {
            e.stamp = ++g_clock;
            *out = e.map;
            return cudaSuccess;
        }
        if (e.stamp < victim->stamp) victim = &e;
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    err = encoder(&encode);
    if (err != cudaSuccess) return err;
    const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBlock};
    const cuuint32_t elem_strides[2] = {1, 1};
    CUtensorMap map;
    CUresult r = encode(&map, dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void*>(layer_base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    victim->base = layer_base;
    victim->rows = rows;
    victim->head_dim = head_dim;
    victim->dtype = dtype;
    victim->device = dev;
    victim->stamp = ++g_clock;
    victim->map = map;
    *out = map;
    return cudaSuccess;
}

}  // namespace pkv
