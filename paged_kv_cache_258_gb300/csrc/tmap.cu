// tmap.cu -- TMA tensor maps over one layer of a K or V pool (host side).
//
// A pool layer [num_blocks][n_kv][16][D] of 16-bit elements is described as a tensor of
// num_blocks*n_kv*16 rows by D columns, copied with the 128-byte swizzle in one of two box shapes:
//   PKV_BOX_PANEL  2-D, a 64-column x 16-row box: one 64-column panel of one (block, KV head)
//                  chunk, placed by the caller (decode, and the K tiles of prefill, whose panels
//                  of several blocks must sit in one [panel][rows] array);
//   PKV_BOX_BLOCK  3-D (64 columns, rows, D/64 panels at a 128-byte stride), a 64 x 16 x D/64 box:
//                  the whole chunk in one copy, landing as [panel][16 rows][128 B] (the V tiles
//                  of prefill, read by the tensor cores one 16-key block at a time);
//   PKV_BOX_BLOCK_HALF  the same with a 64 x 16 x D/128 box: half of the chunk's columns (the V
//                  blocks of a prefill CTA pair, whose CTAs each hold half of every V block).
// Encoding goes through the driver entry point cuTensorMapEncodeTiled, found once through the
// runtime; maps are cached by (address, shape, type, box, device) in a hash table so steady-state
// calls do not re-encode: a step touches up to 3 maps per layer (K panels, V panels, V blocks), so
// the table holds every map of several multi-layer caches at once. A map depends only on its key,
// so an entry stays valid even if its pool is freed and another one reuses the address. A new
// address is accepted only if it is device memory of the current device
// (cudaErrorInvalidDevicePointer otherwise, which the C ABI reports as PKV_ERR_INVALID_ARG).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "internal.h"

namespace pkv {
namespace {

struct MapKey {
    const void* base;
    long long rows;
    int head_dim;
    int dtype;
    int box;
    int device;
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && head_dim == o.head_dim && dtype == o.dtype && box == o.box &&
               device == o.device;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        unsigned long long h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
        h ^= (unsigned long long)k.rows + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2);
        h ^= (unsigned long long)((k.head_dim << 12) | (k.dtype << 8) | (k.box << 6) | (k.device & 63)) +
             (h << 6) + (h >> 2);
        return (size_t)h;
    }
};

// Beyond this many maps the table is emptied and refilled on demand (maps are cheap to re-encode;
// the bound only keeps a process that creates and drops many pools from growing the table).
constexpr size_t kMaxMaps = 4096;

std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash>* g_maps = nullptr;
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
    if (box != PKV_BOX_PANEL && box != PKV_BOX_BLOCK && box != PKV_BOX_BLOCK_HALF) return cudaErrorInvalidValue;
    if (box == PKV_BOX_BLOCK_HALF && (head_dim % 128) != 0) return cudaErrorInvalidValue;
    if (rows <= 0 || rows >= (1LL << 31) || (head_dim % 64) != 0) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const MapKey key{layer_base, rows, head_dim, dtype, box, dev};
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (!g_maps) g_maps = new std::unordered_map<MapKey, CUtensorMap, MapKeyHash>();  // lives until exit
    const auto hit = g_maps->find(key);
    if (hit != g_maps->end()) {
        *out = hit->second;
        return cudaSuccess;
    }
    // The copies read the pool directly: before a map is first built for an address, make sure it
    // is device memory of this device (not host memory, not another GPU's memory).
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, layer_base) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is an argument error, not a sticky one
        return cudaErrorInvalidDevicePointer;
    }
    if (pa.type != cudaMemoryTypeDevice || pa.device != dev) return cudaErrorInvalidDevicePointer;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    err = encoder(&encode);
    if (err != cudaSuccess) return err;
    const bool blk = box != PKV_BOX_PANEL;
    const cuuint32_t rank = blk ? 3 : 2;
    // dims / box innermost first; strides (bytes) of dims 1.. (the panel dim of the 3-D form steps
    // 64 elements = 128 bytes inside a row)
    const cuuint64_t dims[3] = {blk ? 64u : (cuuint64_t)head_dim, (cuuint64_t)rows, (cuuint64_t)(head_dim / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128};
    const cuuint32_t boxdim[3] = {64, (cuuint32_t)kBlock,
                                  (cuuint32_t)(box == PKV_BOX_BLOCK_HALF ? head_dim / 128 : head_dim / 64)};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUtensorMap map;
    CUresult r = encode(&map, dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        rank, const_cast<void*>(layer_base), dims, strides, boxdim, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (g_maps->size() >= kMaxMaps) g_maps->clear();
    g_maps->emplace(key, map);
    *out = map;
    return cudaSuccess;
}

}  // namespace pkv
