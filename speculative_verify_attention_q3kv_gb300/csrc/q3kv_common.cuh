// Device helpers shared by the two verify legs: input loads, the in-shared-
// memory Hadamard rotation of query/output rows, and the split-K merge.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "q3kv_internal.h"

namespace q3kv {

__device__ __forceinline__ float load_in(const float* p) { return *p; }
__device__ __forceinline__ float load_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// In-place unnormalised H (entries +-1) on rows [0, nrows) of a [rows][256]
// float array in shared memory; all threads of the block take part.
__device__ inline void rotate_rows(float* x, int nrows) {
    for (int h = 1; h < kHeadDim; h <<= 1) {
        for (int idx = threadIdx.x; idx < nrows * (kHeadDim / 2); idx += blockDim.x) {
            const int r = idx / (kHeadDim / 2);
            const int j = idx % (kHeadDim / 2);
            const int i = (j / h) * 2 * h + (j % h);
            float* row = x + r * kHeadDim;
            const float a = row[i], b = row[i + h];
            row[i] = a + b;
            row[i + h] = a - b;
        }
        __syncthreads();
    }
}

// Merge the split partials of one (slot, kv head, row chunk):
//   o[r][d] = sum_i w_i o_i[r][d],  w_i = e^(m_i - M) / sum_j e^(m_j - M) l_j
// (base-2 exponentials when LOG2, i.e. m in log2 units).  Result rows go to
// `out` ([rows][256] floats in shared memory).  `wts` is shared scratch of at
// least 16384 floats; `mrow`, `lrow` shared arrays of >= 64 floats.  Threads:
// blockDim.x == 256 (one output dim each).
template <bool LOG2>
__device__ inline void merge_splits(const float* po0, const float* pml0, int n_splits, int Rc, int rows_stride,
                                    float* wts, float* mrow, float* lrow, float* out) {
    const int tid = threadIdx.x;
    for (int r = tid; r < Rc; r += blockDim.x) {
        float M = -CUDART_INF_F;
        for (int i = 0; i < n_splits; ++i) M = fmaxf(M, __ldcg(pml0 + ((int64_t)i * rows_stride + r) * 2));
        float den = 0.0f;
        for (int i = 0; i < n_splits; ++i) {
            const float mi = __ldcg(pml0 + ((int64_t)i * rows_stride + r) * 2);
            if (mi != -CUDART_INF_F)
                den += (LOG2 ? exp2f(mi - M) : expf(mi - M)) * __ldcg(pml0 + ((int64_t)i * rows_stride + r) * 2 + 1);
        }
        mrow[r] = M;
        lrow[r] = den;
    }
    __syncthreads();
    const int chunk_splits = max(1, 16384 / rows_stride);
    float acc[kFmaRows];
#pragma unroll
    for (int r = 0; r < kFmaRows; ++r) acc[r] = 0.0f;
    for (int i0 = 0; i0 < n_splits; i0 += chunk_splits) {
        const int ni = min(chunk_splits, n_splits - i0);
        for (int idx = tid; idx < ni * rows_stride; idx += blockDim.x) {
            const int i = idx / rows_stride, r = idx % rows_stride;
            float wv = 0.0f;
            if (r < Rc) {
                const float mi = __ldcg(pml0 + ((int64_t)(i0 + i) * rows_stride + r) * 2);
                if (mi != -CUDART_INF_F) wv = (LOG2 ? exp2f(mi - mrow[r]) : expf(mi - mrow[r])) / lrow[r];
            }
            wts[idx] = wv;
        }
        __syncthreads();
        for (int i = 0; i < ni; ++i) {
            const float* src = po0 + (int64_t)(i0 + i) * rows_stride * kHeadDim + tid;
#pragma unroll
            for (int r = 0; r < kFmaRows; ++r)
                if (r < Rc) acc[r] = fmaf(wts[i * rows_stride + r], __ldcg(src + r * kHeadDim), acc[r]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < kFmaRows; ++r)
        if (r < Rc) out[r * kHeadDim + tid] = acc[r];
}

}  // namespace q3kv
