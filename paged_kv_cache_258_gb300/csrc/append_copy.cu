// append_copy.cu -- KV append scatter and copy-on-write block copy kernels (sm_103a).
//
// kv_append ("04 - Hacia PagedAttention (vista previa)", "La idea de PagedAttention", step 3):
// the new token's K and V rows go to row (slot / 16, head, slot % 16) of the layer's pools.
// copy_blocks ("PagedAttention e continuous batching", "01 - Conceito", paragraph 6): a
// diverging branch gets a private copy of the shared block before it writes into it.
// Both are pure byte moves with 16-byte vector accesses; they are bit-exact by construction.
#include "common.cuh"
#include "internal.h"

namespace pkv {

// One warp per (token, KV head): lanes move the K row's and the V row's 16-byte chunks.
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const int nch = a.row_bytes / 16;
    const long long n_items = (long long)a.n_tok * a.n_kv;
    const long long warps_total = (long long)gridDim.x * (blockDim.x / 32);
    for (long long item = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); item < n_items;
         item += warps_total) {
        const int t = (int)(item / a.n_kv);
        const int g = (int)(item % a.n_kv);
        const long long slot = a.slots[t];
        if (slot < 0) continue;  // padding token
        if (slot >= (long long)a.num_blocks * kBlock) {
            if (lane == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_SLOT);
            continue;
        }
        const long long phys = slot / kBlock;
        const int off = (int)(slot % kBlock);
        const size_t dst_row = (((size_t)phys * a.n_kv + g) * kBlock + off) * (size_t)a.row_bytes;
        const size_t src_row = ((size_t)t * a.n_kv + g) * (size_t)a.row_bytes;
        for (int c = lane; c < 2 * nch; c += 32) {
            const bool is_v = c >= nch;
            const int cc = is_v ? c - nch : c;
            const char* src = reinterpret_cast<const char*>(is_v ? a.v : a.k) + src_row + (size_t)cc * 16;
            char* dst = reinterpret_cast<char*>(is_v ? a.v_layer : a.k_layer) + dst_row + (size_t)cc * 16;
            *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
        }
    }
}

// grid (pair, layer, K/V): each CTA copies one block of one layer of one pool.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyArgs a) {
    const int pair = blockIdx.x;
    const int layer = blockIdx.y;
    const int src = a.pairs[2 * pair];
    const int dst = a.pairs[2 * pair + 1];
    if ((unsigned)src >= (unsigned)a.num_blocks || (unsigned)dst >= (unsigned)a.num_blocks) {
        if (threadIdx.x == 0 && layer == 0 && blockIdx.z == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_PAIR);
        return;
    }
    char* pool = reinterpret_cast<char*>(blockIdx.z == 0 ? a.k_pool : a.v_pool) + (size_t)layer * a.layer_bytes;
    const uint4* s = reinterpret_cast<const uint4*>(pool + (size_t)src * a.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(pool + (size_t)dst * a.block_bytes);
    const size_t n = a.block_bytes / 16;
    // eight 16-byte loads in flight per thread before their stores: source and destination lie in
    // the same pool, so a plain load-store loop would keep only one load outstanding
    constexpr int U = 8;
    for (size_t i0 = threadIdx.x; i0 < n; i0 += (size_t)U * blockDim.x) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t i = i0 + (size_t)u * blockDim.x;
            if (i < n) r[u] = s[i];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t i = i0 + (size_t)u * blockDim.x;
            if (i < n) d[i] = r[u];
        }
    }
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    const long long items = (long long)a.n_tok * a.n_kv;
    const int warps_per_cta = 8;
    long long ctas = (items + warps_per_cta - 1) / warps_per_cta;
    if (ctas > 65535LL * 64) ctas = 65535LL * 64;
    kv_append_kernel<<<(unsigned)ctas, warps_per_cta * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream) {
    copy_blocks_kernel<<<dim3(a.n_pairs, a.n_layers, 2), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
