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

// Unnormalised H (entries +-1) on one 256-element row held by a warp: lane l
// holds elements 8l .. 8l + 7, so strides 1, 2 and 4 pair elements within a
// lane and strides 8 .. 128 pair lane l with lane l ^ (stride / 8) (the lower
// lane keeps a + b, the upper a - b).  The stages run in the radix-2 order,
// stride 1 first, with the same two operations per pair, so the result equals
// the element-by-element butterfly bit for bit.
__device__ __forceinline__ void rotate_row_regs(float (&y)[8]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if ((i & h) == 0) {
                const float a = y[i], b = y[i + h];
                y[i] = a + b;
                y[i + h] = a - b;
            }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, y[i], m);
            y[i] = upper ? o - y[i] : y[i] + o;
        }
    }
}

// In-place unnormalised H on rows [0, nrows) of a [rows][256] float array in
// shared memory (16-byte aligned), one warp per row; all threads of the block
// take part (a block of whole warps), and the block is synchronised on return.
__device__ inline void rotate_rows(float* x, int nrows) {
    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    for (int r = threadIdx.x >> 5; r < nrows; r += nwarps) {
        float4* row = reinterpret_cast<float4*>(x + r * kHeadDim + 8 * lane);
        const float4 u = row[0], w = row[1];
        float y[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
        rotate_row_regs(y);
        row[0] = make_float4(y[0], y[1], y[2], y[3]);
        row[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
    __syncthreads();
}

// Pages per context split of this launch.  A caller-fixed size is used as it
// is.  The automatic policy sizes the splits from every slot's own length
// (not the longest one's): the smallest size d at which the CTAs of all
// slots, sum over slots of ceil(pages_b / d) x row chunks_b per kv head, are
// at most split_target / kv heads (one wave), and at least the size that
// keeps every slot within the num_splits partial slots the workspace holds
// per unit; no split when the units alone reach the target.  The search is a
// bisection between the even share of all pages, ceil(total / target), and
// ceil(total / (target - units)), which always fits (ceil(x / d) <= x / d + 1).
// Each warp evaluates it on its own (lane = slot, warp sums; 32-bit
// arithmetic), so no block barrier is needed, and every kernel of the call
// gets the same answer from the same lengths.  Both legs use 64-row chunks;
// split_target is per kv head.
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ inline int split_pages_of(const VerifyArgs& a) {
    if (!a.split_auto) return a.split_pages;
    // lane b holds slot b's pages and row chunks of 64 rows (0 for an invalid
    // slot); the host enables the policy only for 2..32 slots, so one pass of
    // lanes covers them and every sum below fits 32 bits
    const int lane = threadIdx.x & 31;
    int pages = 0, chunks = 0;
    if (lane < a.num_slots) {
        const int T = a.n_q[lane], L = a.ctx_len[lane];
        if (T > 0 && T <= a.max_n_q && T <= L && L <= a.max_pages_per_slot * kPageSize) {
            pages = (L + kPageSize - 1) / kPageSize;
            chunks = (kGroup * T + 63) >> 6;
        }
    }
    const int units = warp_sum_i(chunks);
    const int maxp = max(1, warp_max_i(pages));
    const int total = warp_sum_i(pages * chunks);
    const int target = a.split_target;                                    // CTAs per kv head
    const int floor_d = (maxp + a.num_splits - 1) / a.num_splits;          // the workspace's bound
    if (units >= target) return maxp;                                      // the units fill the GPU
    int lo = max(1, (total + target - 1) / target);                        // may not fit
    int hi = min(maxp, (total + (target - units) - 1) / (target - units)); // fits
    if (lo < hi && warp_sum_i(pages ? ((pages + lo - 1) / lo) * chunks : 0) <= target) hi = lo;
    while (hi - lo > 1) {                                                  // ctas(lo) > target >= ctas(hi)
        const int mid = (lo + hi) >> 1;
        if (warp_sum_i(pages ? ((pages + mid - 1) / mid) * chunks : 0) <= target) hi = mid;
        else lo = mid;
    }
    return max(hi, floor_d);
}

}  // namespace q3kv
