// Split-K merge for both verify legs (the flash-decode combine step).
//
// One CTA per (query row, unit) where unit = (slot, kv head, row chunk).
// For a row with partials (m_i, l_i, o_i) from splits i:
//   M = max_i m_i,  w_i = e^(m_i - M) / sum_j e^(m_j - M) l_j,  o = sum_i w_i o_i
// (base-2 exponentials for the tensor-core leg, whose scores are in log2
// units), then out = H o / 16 back in the unrotated basis (the fp8 cache is
// not rotated: out = o).
//
// The kernel is launched with programmatic stream serialisation: its CTAs may
// start while the verify kernel finishes and wait (griddepcontrol.wait) for
// its results before the first read.  Right after the wait each thread
// issues the loads of up to 24 partial rows of its split group (256 threads =
// 4 split groups x 64 float4 columns) together with the (m, l) pairs, which
// are read once; one warp finishes the row with register/shuffle butterflies
// for H.
#include <math_constants.h>

#include "q3kv_common.cuh"
#include "q3kv_internal.h"

namespace q3kv {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kWChunk = 2048;     // split weights staged in shared memory at a time

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// e^x (natural units) or 2^x (log2 units); -inf gives 0
template <bool LOG2>
__device__ __forceinline__ float pexp(float x) { return LOG2 ? exp2f(x) : __expf(x); }

template <bool LOG2, bool ROT>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(VerifyArgs a, int rows_per_chunk) {
    __shared__ float w[kWChunk];
    __shared__ __align__(16) float4 part[4][64];
    __shared__ float red[2][kMergeThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int unit = blockIdx.y;
    const int chunk = unit % a.row_chunks;
    const int g = (unit / a.row_chunks) % a.num_kv_heads;
    const int slot = unit / (a.row_chunks * a.num_kv_heads);

    // the next grid may be scheduled now; the verify kernel's partials (and
    // the lengths it validated) are complete after the wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int T = a.n_q[slot];
    const int L = a.ctx_len[slot];
    if (T <= 0 || T > a.max_n_q || T > L || L > a.max_pages_per_slot * kPageSize) return;   // flagged by the verify kernel
    const int row0 = chunk * rows_per_chunk;
    const int Rc = min(rows_per_chunk, kGroup * T - row0);
    if (r >= Rc) return;
    const int n_pages = (L + kPageSize - 1) / kPageSize;
    const int split_pages = split_pages_of(a);
    const int n_splits = (n_pages + split_pages - 1) / split_pages;
    if (n_splits <= 1 || n_splits > a.num_splits) return;   // single split: the verify kernel wrote the row

    const float2* pml = reinterpret_cast<const float2*>(a.part_ml) + ((int64_t)unit * a.num_splits * rows_per_chunk + r);
    const int64_t ml_stride = rows_per_chunk;
    const int64_t o_stride = (int64_t)rows_per_chunk * kHeadDim;

    // ---- the first kOPre partial rows of each split group are loaded now,
    // alongside the (m, l) pairs, so both reads overlap in one round trip
    const int sg = tid >> 6, c = tid & 63;          // split group of 4, float4 column
    const float* po4 = a.part_o + ((int64_t)unit * a.num_splits * rows_per_chunk + r) * kHeadDim + 4 * c;
    constexpr int kOPre = 24;
    float4 ov[kOPre];
#pragma unroll
    for (int k = 0; k < kOPre; ++k) {
        const int i = sg + 4 * k;
        ov[k] = i < n_splits ? __ldcg(reinterpret_cast<const float4*>(po4 + i * o_stride)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // ---- M, the denominator and the weights from one read of the (m, l)
    // pairs (held in registers for the first 2048 splits; any further ones are
    // read again in each pass)
    constexpr int kPerThread = kWChunk / kMergeThreads;
    float2 ml[kPerThread];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int i = k * kMergeThreads + tid;
        ml[k] = i < n_splits ? __ldcg(pml + i * ml_stride) : make_float2(-CUDART_INF_F, 0.0f);
        M = fmaxf(M, ml[k].x);
    }
#pragma unroll 1
    for (int i = kWChunk + tid; i < n_splits; i += kMergeThreads) M = fmaxf(M, __ldcg(pml + i * ml_stride).x);
    M = warp_max(M);
    if (lane == 0) red[0][warp] = M;
    __syncthreads();
    M = red[0][0];
#pragma unroll
    for (int k = 1; k < kMergeThreads / 32; ++k) M = fmaxf(M, red[0][k]);
    float den = 0.0f;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        ml[k].x = pexp<LOG2>(ml[k].x - M);           // e^(m_i - M); 0 for the padding
        den = fmaf(ml[k].x, ml[k].y, den);
    }
#pragma unroll 1
    for (int i = kWChunk + tid; i < n_splits; i += kMergeThreads) {
        const float2 v = __ldcg(pml + i * ml_stride);
        den = fmaf(pexp<LOG2>(v.x - M), v.y, den);
    }
    den = warp_sum(den);
    if (lane == 0) red[1][warp] = den;
    __syncthreads();
    den = 0.0f;
#pragma unroll
    for (int k = 0; k < kMergeThreads / 32; ++k) den += red[1][k];
    const float inv = 1.0f / den;

    // ---- o = sum_i w_i o_i, in passes of 2048 splits
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int i0 = 0; i0 < n_splits; i0 += kWChunk) {
        const int ni = min(kWChunk, n_splits - i0);
        if (i0 == 0) {
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) w[k * kMergeThreads + tid] = ml[k].x * inv;
        } else {
#pragma unroll 1
            for (int i = tid; i < ni; i += kMergeThreads) w[i] = pexp<LOG2>(__ldcg(pml + (i0 + i) * ml_stride).x - M) * inv;
        }
        __syncthreads();
        int i = sg;
        if (i0 == 0) {
#pragma unroll
            for (int k = 0; k < kOPre; ++k, i += 4) {
                const float wi = w[i];                   // 0 past the last split (padding weights)
                acc.x = fmaf(wi, ov[k].x, acc.x);
                acc.y = fmaf(wi, ov[k].y, acc.y);
                acc.z = fmaf(wi, ov[k].z, acc.z);
                acc.w = fmaf(wi, ov[k].w, acc.w);
            }
        }
#pragma unroll 1
        for (; i < ni; i += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(po4 + (i0 + i) * o_stride));
            const float wi = w[i];
            acc.x = fmaf(wi, v.x, acc.x);
            acc.y = fmaf(wi, v.y, acc.y);
            acc.z = fmaf(wi, v.z, acc.z);
            acc.w = fmaf(wi, v.w, acc.w);
        }
        __syncthreads();
    }
    part[sg][c] = acc;
    __syncthreads();
    if (warp != 0) return;

    // ---- one warp: sum the split groups, out = H o / 16 (lane holds dims 8 lane .. 8 lane + 7);
    // without ROT (the fp8 cache, unrotated) out = o
    float x[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float4 t = part[0][2 * lane + h];
#pragma unroll
        for (int k = 1; k < 4; ++k) {
            const float4 u = part[k][2 * lane + h];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        x[4 * h] = t.x; x[4 * h + 1] = t.y; x[4 * h + 2] = t.z; x[4 * h + 3] = t.w;
    }
    if (ROT) rotate_row_regs(x);
    const int ra = row0 + r;
    const int Hq = a.num_kv_heads * kGroup;
    float* dst = a.out + (((int64_t)a.q_offsets[slot] + ra / kGroup) * Hq + g * kGroup + ra % kGroup) * kHeadDim + 8 * lane;
    constexpr float kS = ROT ? 0.0625f : 1.0f;
    reinterpret_cast<float4*>(dst)[0] = make_float4(x[0] * kS, x[1] * kS, x[2] * kS, x[3] * kS);
    reinterpret_cast<float4*>(dst)[1] = make_float4(x[4] * kS, x[5] * kS, x[6] * kS, x[7] * kS);
}

template <bool LOG2, bool ROT>
cudaError_t launch(const VerifyArgs& a, int rows_per_chunk, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows_per_chunk, (unsigned)(a.num_slots * a.num_kv_heads * a.row_chunks));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<LOG2, ROT>, a, rows_per_chunk);
}

}  // namespace

cudaError_t launch_merge(const VerifyArgs& a, int rows_per_chunk, bool log2_units, cudaStream_t stream) {
    if (a.num_splits <= 1) return cudaSuccess;
    if (a.fmt == kFmtFp8) return launch<true, false>(a, rows_per_chunk, stream);   // tensor-core leg only
    return log2_units ? launch<true, true>(a, rows_per_chunk, stream) : launch<false, true>(a, rows_per_chunk, stream);
}

}  // namespace q3kv
