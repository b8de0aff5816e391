// Split-K merge for both verify legs (the flash-decode combine step).
//
// One CTA per (query row, unit) where unit = (slot, kv head, row chunk); its
// 256 threads read the partials as float4 over four groups of splits at once.
// For a row with partials (m_i, l_i, o_i) from splits i:
//   M = max_i m_i,  w_i = e^(m_i - M) / sum_j e^(m_j - M) l_j,  o = sum_i w_i o_i
// (base-2 exponentials for the tensor-core leg, whose scores are in log2
// units), then out = H o / 16 back in the unrotated basis.
#include <math_constants.h>

#include "q3kv_common.cuh"
#include "q3kv_internal.h"

namespace q3kv {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kWChunk = 2048;     // split weights staged in shared memory at a time

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, w) : v + w;
    }
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = scratch[0];
    for (int i = 1; i < kMergeThreads / 32; ++i) r = is_max ? fmaxf(r, scratch[i]) : r + scratch[i];
    __syncthreads();
    return r;
}

template <bool LOG2>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(VerifyArgs a, int rows_per_chunk) {
    __shared__ float w[kWChunk];
    __shared__ float row[kHeadDim];
    __shared__ float scratch[kMergeThreads / 32];
    const int tid = threadIdx.x;
    const int r = blockIdx.x;
    const int unit = blockIdx.y;
    const int chunk = unit % a.row_chunks;
    const int g = (unit / a.row_chunks) % a.num_kv_heads;
    const int slot = unit / (a.row_chunks * a.num_kv_heads);

    const int T = a.n_q[slot];
    const int L = a.ctx_len[slot];
    if (T <= 0 || T > a.max_n_q || T > L || L > a.max_pages_per_slot * kPageSize) return;   // flagged by the verify kernel
    const int row0 = chunk * rows_per_chunk;
    const int Rc = min(rows_per_chunk, kGroup * T - row0);
    if (r >= Rc) return;
    const int n_pages = (L + kPageSize - 1) / kPageSize;
    const int n_splits = (n_pages + a.split_pages - 1) / a.split_pages;
    if (n_splits <= 1 || n_splits > a.num_splits) return;   // single split: the verify kernel wrote the row

    const float* pml = a.part_ml + ((int64_t)unit * a.num_splits * rows_per_chunk + r) * 2;
    const int64_t ml_stride = (int64_t)rows_per_chunk * 2;
    const int64_t o_stride = (int64_t)rows_per_chunk * kHeadDim;

    float M = -CUDART_INF_F;
    for (int i = tid; i < n_splits; i += kMergeThreads) M = fmaxf(M, __ldcg(pml + i * ml_stride));
    M = block_reduce(M, true, scratch);
    float den = 0.0f;
    for (int i = tid; i < n_splits; i += kMergeThreads) {
        const float mi = __ldcg(pml + i * ml_stride);
        if (mi != -CUDART_INF_F) den += (LOG2 ? exp2f(mi - M) : expf(mi - M)) * __ldcg(pml + i * ml_stride + 1);
    }
    den = block_reduce(den, false, scratch);
    const float inv = 1.0f / den;

    // thread = (split group sg of 4, dims 4c..4c+3): float4 loads, four groups
    // of splits in flight at once, combined through shared memory
    const int sg = tid >> 6, c = tid & 63;
    const float* po4 = a.part_o + ((int64_t)unit * a.num_splits * rows_per_chunk + r) * kHeadDim + 4 * c;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i0 = 0; i0 < n_splits; i0 += kWChunk) {
        const int ni = min(kWChunk, n_splits - i0);
        for (int i = tid; i < ni; i += kMergeThreads) {
            const float mi = __ldcg(pml + (i0 + i) * ml_stride);
            w[i] = (mi == -CUDART_INF_F) ? 0.0f : (LOG2 ? exp2f(mi - M) : expf(mi - M)) * inv;
        }
        __syncthreads();
#pragma unroll 4
        for (int i = sg; i < ni; i += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(po4 + (i0 + i) * o_stride));
            const float wi = w[i];
            acc.x = fmaf(wi, v.x, acc.x);
            acc.y = fmaf(wi, v.y, acc.y);
            acc.z = fmaf(wi, v.z, acc.z);
            acc.w = fmaf(wi, v.w, acc.w);
        }
        __syncthreads();
    }
    float4* part = reinterpret_cast<float4*>(w);     // [4 groups][64 quads]
    part[sg * 64 + c] = acc;
    __syncthreads();
    if (tid < 64) {
        float4 t = part[tid];
#pragma unroll
        for (int k = 1; k < 4; ++k) {
            const float4 u = part[k * 64 + tid];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        row[4 * tid] = t.x; row[4 * tid + 1] = t.y; row[4 * tid + 2] = t.z; row[4 * tid + 3] = t.w;
    }
    __syncthreads();
    rotate_rows(row, 1);
    const int ra = row0 + r;
    const int Hq = a.num_kv_heads * kGroup;
    a.out[(((int64_t)a.q_offsets[slot] + ra / kGroup) * Hq + g * kGroup + ra % kGroup) * kHeadDim + tid] =
        row[tid] * 0.0625f;
}

}  // namespace

cudaError_t launch_merge(const VerifyArgs& a, int rows_per_chunk, bool log2_units, cudaStream_t stream) {
    if (a.num_splits <= 1) return cudaSuccess;
    dim3 grid((unsigned)rows_per_chunk, (unsigned)(a.num_slots * a.num_kv_heads * a.row_chunks));
    if (log2_units) merge_kernel<true><<<grid, kMergeThreads, 0, stream>>>(a, rows_per_chunk);
    else merge_kernel<false><<<grid, kMergeThreads, 0, stream>>>(a, rows_per_chunk);
    return cudaGetLastError();
}

}  // namespace q3kv
