// prefill_f32.cu -- paged prefill attention for fp32 storage on the CUDA cores, and the dtype
// dispatch of all prefill launches.
//
// Same operation as prefill_umma.cuh ("PagedAttention e continuous batching", "01 - Conceito",
// paragraph 5; "La idea de PagedAttention", step 5): chunk token i of sequence s sits at
// position c - n + i and attends to keys 0 .. that position, gathered through the block table.
// fp32 storage is the precision mode (1e-5 against the fp64 oracle), which tf32 tensor cores
// would miss, so this kernel stays on the FMA pipe and favours plainness over speed:
//  * CTA = (32 query rows, KV head, sequence), rows = token x head-in-group; warp w owns rows
//    w, w+8, w+16, w+24; lane l owns head dims [l * D/32, (l+1) * D/32);
//  * every 16-token block of K and V is staged in shared memory by the whole CTA, then each warp
//    takes its rows' 16 logits (warp all-reduce), one online-softmax rescale per block, and adds
//    the weighted V rows of the keys its row may see (selection: rows past the position or the
//    context are never read into the result).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

template <int D, int G>
__global__ void __launch_bounds__(256) paged_prefill_f32_kernel(const PrefillArgs a) {
    constexpr int ROWS = kPrefillRowsF32;
    constexpr int QT = ROWS / G;
    constexpr int EPL = D / 32;  // head dims per lane
    constexpr int RPW = ROWS / 8;  // rows per warp
    __shared__ __align__(16) float sk[kBlock][D];
    __shared__ __align__(16) float sv[kBlock][D];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = a.q_tiles - 1 - (int)blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    const int q0 = a.q_start[s];
    const int q1 = a.q_start[s + 1];
    const int n_new = q1 - q0;
    const int ctx = a.lens[s];
    if (q0 < 0 || q1 > a.n_tokens || n_new < 0 || n_new > a.q_tiles * QT || ctx < n_new ||
        ctx > a.max_blocks * kBlock) {
        if (blockIdx.x == 0 && g == 0 && threadIdx.x == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_QUERY_RANGE);
        return;
    }
    const int t0 = tile * QT;
    if (t0 >= n_new) return;
    const int t_end = min(t0 + QT, n_new);
    const int pos0 = ctx - n_new + t0;
    const int pos_last = ctx - n_new + t_end - 1;
    const int n_blk = pos_last / kBlock + 1;

    float qv[RPW][EPL], acc[RPW][EPL], m[RPW], l[RPW];
    int lim[RPW];
    bool live[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + 8 * i;
        const int tt = r / G;
        live[i] = t0 + tt < n_new;
        lim[i] = min(pos0 + tt, ctx - 1);
        const float* qrow = reinterpret_cast<const float*>(a.q) + ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + r % G) * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qv[i][e] = live[i] ? qrow[lane * EPL + e] : 0.f;
            acc[i][e] = 0.f;
        }
        m[i] = -INFINITY;
        l[i] = 0.f;
    }

    const float* kl = reinterpret_cast<const float*>(a.k_layer);
    const float* vl = reinterpret_cast<const float*>(a.v_layer);
    const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
    for (int b = 0; b < n_blk; ++b) {
        const int phys = trow[b];
        if ((unsigned)phys >= (unsigned)a.num_blocks) {  // skipped: its keys count as masked
            if (threadIdx.x == 0) atomicOr(a.status, (unsigned)PKV_DEV_BAD_BLOCK_ID);
            continue;
        }
        __syncthreads();  // the previous block's rows have been used
        const size_t base = ((size_t)phys * a.n_kv + g) * kBlock * D;
        for (int i = threadIdx.x; i < kBlock * D / 4; i += 256) {
            reinterpret_cast<float4*>(&sk[0][0])[i] = reinterpret_cast<const float4*>(kl + base)[i];
            reinterpret_cast<float4*>(&sv[0][0])[i] = reinterpret_cast<const float4*>(vl + base)[i];
        }
        __syncthreads();
        const int key0 = b * kBlock;
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            if (!live[i] || key0 > lim[i]) continue;  // warp-uniform
            const int nk = min(kBlock, lim[i] - key0 + 1);
            float z[kBlock];
            float mx = -INFINITY;
#pragma unroll
            for (int kk = 0; kk < kBlock; ++kk) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d = fmaf(qv[i][e], sk[kk][lane * EPL + e], d);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                z[kk] = kk < nk ? d * a.scale_log2 : -INFINITY;
                mx = fmaxf(mx, z[kk]);
            }
            const float mn = fmaxf(m[i], mx);
            const float al = m[i] == -INFINITY ? 0.f : exp2f(m[i] - mn);
            m[i] = mn;
            l[i] *= al;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[i][e] *= al;
#pragma unroll
            for (int kk = 0; kk < kBlock; ++kk) {
                if (kk < nk) {
                    const float p = exp2f(z[kk] - mn);
                    l[i] += p;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[i][e] = fmaf(p, sv[kk][lane * EPL + e], acc[i][e]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        if (!live[i]) continue;
        const int r = warp + 8 * i;
        const int tt = r / G;
        float* orow = reinterpret_cast<float*>(a.out) + ((size_t)(q0 + t0 + tt) * a.n_q + (size_t)g * G + r % G) * D;
        const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) orow[lane * EPL + e] = acc[i][e] * inv;
    }
}

template <int D, int G>
cudaError_t launch_f32_tpl(const PrefillArgs& a, cudaStream_t stream) {
    dim3 grid(a.q_tiles, a.n_kv, a.n_seqs);
    paged_prefill_f32_kernel<D, G><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t f32_wave_ctas_tpl(int sms, int* out) {
    int per_sm = 0;
    const cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, paged_prefill_f32_kernel<D, G>, 256, 0);
    *out = sms * per_sm;
    return err;
}

}  // namespace

cudaError_t prefill_wave_ctas(int dtype, int head_dim, int group, int sms, int* out) {
    if (dtype == PKV_F16) return prefill_wave_ctas_f16(head_dim, group, sms, out);
    if (dtype == PKV_BF16) return prefill_wave_ctas_bf16(head_dim, group, sms, out);
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return f32_wave_ctas_tpl<DD, GG>(sms, out);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_f32(int head_dim, int group, const PrefillArgs& a, cudaStream_t stream) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return launch_f32_tpl<DD, GG>(a, stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
    PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(int dtype, int head_dim, int group, const PrefillArgs& a, cudaStream_t stream) {
    switch (dtype) {
    case PKV_F32: return launch_prefill_f32(head_dim, group, a, stream);
    case PKV_F16: return launch_prefill_f16(head_dim, group, a, stream);
    case PKV_BF16: return launch_prefill_bf16(head_dim, group, a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
