// Greedy acceptance of a verify step and the commit of the cache length.
//
// Source: "Quasar" (q27) wiki -- the sampler paragraph of "Serving" (greedy
// argmax is the default) and the "Model tool protocol" bullet (greedy
// speculative decode); the prefix-cache discussion (attention rows below the
// drafts' divergence point are append-only and stay valid, so rejected drafts
// are undone by shortening the length).
//
// Slot b verifies T query tokens (t_0 then drafts d_1 .. d_{T-1}); logits row
// j of the slot predicts the token after query token j.  g_j = argmax of row
// j (lowest index on equal maxima); drafts are accepted while d_{j+1} == g_j;
// a = accepted count, next token = g_a, committed length = ctx_len - (T-1-a).
//
// argmax_kernel: grid (vocab chunks, rows); each CTA streams one chunk of one
// row (16-byte loads when the rows are 16-byte aligned) and writes its
// (max, lowest index) to the workspace.  accept_kernel: one warp per slot,
// launched with programmatic stream serialisation, reduces the chunks of
// each of the slot's rows and runs the acceptance chain.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "q3kv_internal.h"

namespace q3kv {
namespace {

constexpr int kArgThreads = 256;

struct Best {
    float v;
    int i;
};

// a beats b: larger value, or the same value at a lower index
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
    return av > bv || (av == bv && ai < bi);
}

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, b.v, o);
        const int i = __shfl_xor_sync(0xffffffffu, b.i, o);
        if (beats(v, i, b.v, b.i)) { b.v = v; b.i = i; }
    }
    return b;
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(kArgThreads) argmax_kernel(AcceptArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ Best red[kArgThreads / 32];
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int64_t c0 = (int64_t)chunk * a.chunk_elems;
    const int64_t c1 = min((int64_t)a.vocab, c0 + a.chunk_elems);
    const T* lg = static_cast<const T*>(a.logits) + (int64_t)row * a.vocab;
    Best b{-CUDART_INF_F, INT32_MAX};
    bool nan = false;
    constexpr int kVec = 16 / sizeof(T);
    if (a.vec_ok) {
        // chunk_elems is a multiple of kVec and the rows are 16-byte aligned
        const uint4* p = reinterpret_cast<const uint4*>(lg + c0);
        const int64_t n = (c1 - c0) / kVec;
        constexpr int kUnroll = 4;                  // a thread's loads are all in flight at once
        for (int64_t k0 = threadIdx.x; k0 < n; k0 += kUnroll * kArgThreads) {
            uint4 u[kUnroll];
#pragma unroll
            for (int r = 0; r < kUnroll; ++r) {
                const int64_t k = k0 + (int64_t)r * kArgThreads;
                u[r] = k < n ? __ldcs(p + k) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int r = 0; r < kUnroll; ++r) {
                const int64_t k = k0 + (int64_t)r * kArgThreads;
                if (k >= n) break;
                const T* e = reinterpret_cast<const T*>(&u[r]);
#pragma unroll
                for (int m = 0; m < kVec; ++m) {
                    const float v = to_f(e[m]);
                    nan |= (v != v);
                    // ascending per thread: the first of equal maxima is kept
                    if (beats(v, (int)(c0 + k * kVec + m), b.v, b.i)) { b.v = v; b.i = (int)(c0 + k * kVec + m); }
                }
            }
        }
        for (int64_t k = c0 + n * kVec + threadIdx.x; k < c1; k += kArgThreads) {   // ragged tail
            const float v = to_f(lg[k]);
            nan |= (v != v);
            if (beats(v, (int)k, b.v, b.i)) { b.v = v; b.i = (int)k; }
        }
    } else {
        for (int64_t k = c0 + threadIdx.x; k < c1; k += kArgThreads) {
            const float v = to_f(lg[k]);
            nan |= (v != v);
            if (beats(v, (int)k, b.v, b.i)) { b.v = v; b.i = (int)k; }
        }
    }
    b = warp_best(b);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = b;
    if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0 && a.status)
        atomicOr(a.status, Q3KV_STATUS_NONFINITE_INPUT);
    __syncthreads();
    if (threadIdx.x < 32) {
        Best c = threadIdx.x < kArgThreads / 32 ? red[threadIdx.x] : Best{-CUDART_INF_F, INT32_MAX};
        c = warp_best(c);
        if (threadIdx.x == 0) {
            float2* out = reinterpret_cast<float2*>(a.partial) + (int64_t)row * a.num_chunks + chunk;
            *out = make_float2(c.v, __int_as_float(c.i));
        }
    }
}

__global__ void __launch_bounds__(32) accept_kernel(AcceptArgs a) {
    const int b = blockIdx.x, lane = threadIdx.x;
    // the argmax grid's partials are complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int T = a.n_q[b];
    const int32_t L = a.ctx_len[b];
    if (T <= 0 || T > a.max_n_q || T > L || a.q_offsets[b] < 0 || a.q_offsets[b] + T > a.num_rows) {
        if (lane == 0) {
            if (T != 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
            a.n_accepted[b] = 0;
            a.next_token[b] = -1;
            a.committed_len[b] = L;
        }
        return;
    }
    const int r0 = a.q_offsets[b];
    // every load up front: lane j < T holds query token j; lane k reduces
    // chunks k, k + 32, .. of all T rows at once
    const int tok = lane < T ? a.tokens[r0 + lane] : -1;
    const float2* pp = reinterpret_cast<const float2*>(a.partial) + (int64_t)r0 * a.num_chunks;
    Best c[kMaxNq];
#pragma unroll
    for (int j = 0; j < kMaxNq; ++j) c[j] = Best{-CUDART_INF_F, INT32_MAX};
    for (int k = lane; k < a.num_chunks; k += 32) {
#pragma unroll
        for (int j = 0; j < kMaxNq; ++j)
            if (j < T) {
                const float2 u = pp[(int64_t)j * a.num_chunks + k];
                if (beats(u.x, __float_as_int(u.y), c[j].v, c[j].i)) { c[j].v = u.x; c[j].i = __float_as_int(u.y); }
            }
    }
    int g_lane = -1;                                 // lane j: g_j
#pragma unroll
    for (int j = 0; j < kMaxNq; ++j)
        if (j < T) {
            const Best w = warp_best(c[j]);
            if (lane == j) g_lane = w.i;
        }
    // drafts accepted while d_{j+1} == g_j: the first lane j < T-1 that differs ends the chain
    const int next_tok = __shfl_down_sync(0xffffffffu, tok, 1);
    const unsigned miss = __ballot_sync(0xffffffffu, lane < T - 1 && next_tok != g_lane);
    const int acc = miss ? __ffs(miss) - 1 : T - 1;
    const int nxt = __shfl_sync(0xffffffffu, g_lane, acc);
    if (lane == 0) {
        a.n_accepted[b] = acc;
        a.next_token[b] = nxt;
        a.committed_len[b] = L - (T - 1 - acc);
    }
}

}  // namespace

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t stream) {
    if (a.num_rows > 0) {
        const dim3 grid((unsigned)a.num_chunks, (unsigned)a.num_rows);
        if (a.dtype == Q3KV_F32) argmax_kernel<float><<<grid, kArgThreads, 0, stream>>>(a);
        else argmax_kernel<__nv_bfloat16><<<grid, kArgThreads, 0, stream>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.num_slots);
    cfg.blockDim = dim3(32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_kernel, a);
}

}  // namespace q3kv
