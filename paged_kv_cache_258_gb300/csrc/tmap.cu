// tmap.cu -- TMA tensor maps over one layer of a K or V pool (host side).
//
// A pool layer [num_blocks][n_kv][16][D] of 16-bit elements is described as a tensor of
// num_blocks*n_kv*16 rows by D columns, copied with the 128-byte swizzle in one of two box shapes:
//   PKV_BOX_PANEL  2-D, a 64-column x 16-row box: one 64-column panel of one (block, KV head)
//                  chunk, placed by the caller (decode, and the K tiles of prefill, whose panels
//                  of several blocks must sit in one [panel][rows] array);
//   PKV_BOX_BLOCK  3-D (64 columns, rows, D/64 panels at a 128-byte stride), a 64 x 16 x D/64 box:
//                  the whole chunk in one copy, landing as [panel][16 rows][128 B] (the V tiles
//                  of prefill, read by the tensor cores one 16-key block at a time).
// Encoding goes through the driver entry point cuTensorMapEncodeTiled, found once through the
// runtime; maps are cached by (address, shape, type, box, device) so steady-state calls do not
// re-encode.
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
    int box;
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

cudaError_t kv_tensor_map(const void* layer_base, long long rows, int head_dim, int dtype, int box,
                          CUtensorMap* out) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return cudaErrorInvalidValue;
    if (box != PKV_BOX_PANEL && box != PKV_BOX_BLOCK) return cudaErrorInvalidValue;
    if (rows <= 0 || rows >= (1LL << 31) || (head_dim % 64) != 0) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_map_mu);
    MapEntry* victim = &g_maps[0];
    for (MapEntry& e : g_maps) {
        if (e.stamp && e.base == layer_base && e.rows == rows && e.head_dim == head_dim && e.dtype == dtype &&
            e.box == box && e.device == dev) {
            e.stamp = ++g_clock;
            *out = e.map;
            return cudaSuccess;
        }
        if (e.stamp < victim->stamp) victim = &e;
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    err = encoder(&encode);
    if (err != cudaSuccess) return err;
    const bool blk = box == PKV_BOX_BLOCK;
    const cuuint32_t rank = blk ? 3 : 2;
    // dims / box innermost first; strides (bytes) of dims 1.. (the panel dim of the 3-D form steps
    // 64 elements = 128 bytes inside a row)
    const cuuint64_t dims[3] = {blk ? 64u : (cuuint64_t)head_dim, (cuuint64_t)rows, (cuuint64_t)(head_dim / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128};
    const cuuint32_t boxdim[3] = {64, (cuuint32_t)kBlock, (cuuint32_t)(head_dim / 64)};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUtensorMap map;
    CUresult r = encode(&map, dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        rank, const_cast<void*>(layer_base), dims, strides, boxdim, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    victim->base = layer_base;
    victim->rows = rows;
    victim->head_dim = head_dim;
    victim->dtype = dtype;
    victim->box = box;
    victim->device = dev;
    victim->stamp = ++g_clock;
    victim->map = map;
    *out = map;
    return cudaSuccess;
}

}  // namespace pkv
