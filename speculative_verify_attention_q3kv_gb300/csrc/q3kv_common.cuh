// Device helpers shared by the verify legs and the merge kernel: input loads
// and the in-shared-memory Hadamard rotation of query/output rows.
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

}  // namespace q3kv
