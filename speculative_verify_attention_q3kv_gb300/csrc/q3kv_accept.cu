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

// ---------------------------------------------------------------- sampled acceptance
// Reading of the pages' sampled speculative decode (Gumbel-max sampling with
// rejection-sampled acceptance; the top-p nucleus filter is not built): drafts
// are point masses, so d_{j+1} is accepted iff u_j < p_j(d_{j+1}) with
// p_j = softmax(logits_j / tau); at the first rejection (row a) the next token
// is argmax over x != d_{a+1} of logits_a[x] / tau + G(a, x), else the argmax
// over all x of the last row's keys.  G = -log(-log U), U from the counter-based
// SplitMix64 stream: U = ((z >> 41) + 0.5) / 2^23 with z output number
// row * 2^32 + x of the stream seeded with `seed`.

__device__ __forceinline__ float noise_uniform(uint64_t seed, uint32_t row, uint32_t x) {
    const uint64_t k = ((uint64_t)row << 32) + x;
    uint64_t z = seed + (k + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return ((float)(uint32_t)(z >> 41) + 0.5f) * (1.0f / 8388608.0f);
}

// f(k, logit) for every vocabulary entry k of [c0, c1) of one row, with four
// loads of each thread in flight at once: 16-byte loads when the rows are
// 16-byte aligned (chunk bounds are then multiples of 16 bytes too), else
// element loads.
template <typename T, typename F>
__device__ __forceinline__ void for_each_logit(const AcceptArgs& a, const T* lg, int64_t c0, int64_t c1, F&& f) {
    constexpr int kU = 4;
    if (a.vec_ok) {
        constexpr int kVec = 16 / sizeof(T);
        const uint4* p = reinterpret_cast<const uint4*>(lg + c0);
        const int64_t n = (c1 - c0) / kVec;
        for (int64_t k0 = threadIdx.x; k0 < n; k0 += kU * kArgThreads) {
            uint4 u[kU];
#pragma unroll
            for (int r = 0; r < kU; ++r) {
                const int64_t k = k0 + (int64_t)r * kArgThreads;
                u[r] = k < n ? __ldcs(p + k) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int r = 0; r < kU; ++r) {
                const int64_t k = k0 + (int64_t)r * kArgThreads;
                if (k >= n) break;
                const T* e = reinterpret_cast<const T*>(&u[r]);
#pragma unroll
                for (int m = 0; m < kVec; ++m) f(c0 + k * kVec + m, to_f(e[m]));
            }
        }
    } else {
        for (int64_t k0 = c0 + threadIdx.x; k0 < c1; k0 += kU * kArgThreads) {
            float v[kU];
#pragma unroll
            for (int r = 0; r < kU; ++r) {
                const int64_t k = k0 + (int64_t)r * kArgThreads;
                v[r] = k < c1 ? to_f(lg[k]) : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < kU; ++r) {
                const int64_t k = k0 + (int64_t)r * kArgThreads;
                if (k < c1) f(k, v[r]);
            }
        }
    }
}

// Per (row, chunk): online (max, sum of exp) of logits / tau, and the best
// Gumbel key overall and without the row's next query token.
struct SampleStat {
    float m, s;
    float k1;
    int i1;
    float k2;
    int i2;
};

__device__ __forceinline__ SampleStat stat_merge(SampleStat a, SampleStat b) {
    SampleStat r;
    r.m = fmaxf(a.m, b.m);
    r.s = (a.m == -CUDART_INF_F ? 0.0f : a.s * __expf(a.m - r.m)) + (b.m == -CUDART_INF_F ? 0.0f : b.s * __expf(b.m - r.m));
    const bool b1 = beats(b.k1, b.i1, a.k1, a.i1);
    r.k1 = b1 ? b.k1 : a.k1;
    r.i1 = b1 ? b.i1 : a.i1;
    const bool b2 = beats(b.k2, b.i2, a.k2, a.i2);
    r.k2 = b2 ? b.k2 : a.k2;
    r.i2 = b2 ? b.i2 : a.i2;
    return r;
}

__device__ __forceinline__ SampleStat stat_warp(SampleStat v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        SampleStat w;
        w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
        w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
        w.k1 = __shfl_xor_sync(0xffffffffu, v.k1, o);
        w.i1 = __shfl_xor_sync(0xffffffffu, v.i1, o);
        w.k2 = __shfl_xor_sync(0xffffffffu, v.k2, o);
        w.i2 = __shfl_xor_sync(0xffffffffu, v.i2, o);
        v = stat_merge(v, w);
    }
    return v;
}

__device__ __forceinline__ SampleStat stat_empty() {
    return SampleStat{-CUDART_INF_F, 0.0f, -CUDART_INF_F, INT32_MAX, -CUDART_INF_F, INT32_MAX};
}

template <typename T>
__global__ void __launch_bounds__(kArgThreads) sample_stats_kernel(AcceptArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ SampleStat red[kArgThreads / 32];
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int64_t c0 = (int64_t)chunk * a.chunk_elems;
    const int64_t c1 = min((int64_t)a.vocab, c0 + a.chunk_elems);
    const T* lg = static_cast<const T*>(a.logits) + (int64_t)row * a.vocab;
    const int excl = row + 1 < a.num_rows ? a.tokens[row + 1] : -1;
    SampleStat st = stat_empty();
    bool nan = false;
    for_each_logit(a, lg, c0, c1, [&](int64_t k, float raw) {
        const float l = raw * a.inv_tau;
        nan |= (l != l);
        // running max and sum of exp(l - max)
        if (l > st.m) {
            st.s = (st.m == -CUDART_INF_F ? 0.0f : st.s * __expf(st.m - l)) + 1.0f;
            st.m = l;
        } else {
            st.s += __expf(l - st.m);
        }
        const float key = l - logf(-logf(noise_uniform(a.seed, (uint32_t)row, (uint32_t)k)));
        if (beats(key, (int)k, st.k1, st.i1)) { st.k1 = key; st.i1 = (int)k; }
        if ((int)k != excl && beats(key, (int)k, st.k2, st.i2)) { st.k2 = key; st.i2 = (int)k; }
    });
    st = stat_warp(st);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = st;
    if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0 && a.status)
        atomicOr(a.status, Q3KV_STATUS_NONFINITE_INPUT);
    __syncthreads();
    if (threadIdx.x < 32) {
        SampleStat c = threadIdx.x < kArgThreads / 32 ? red[threadIdx.x] : stat_empty();
        c = stat_warp(c);
        if (threadIdx.x == 0) reinterpret_cast<SampleStat*>(a.partial)[(int64_t)row * a.num_chunks + chunk] = c;
    }
}

template <typename TIn>
__global__ void __launch_bounds__(32) sample_accept_kernel(AcceptArgs a) {
    const int b = blockIdx.x, lane = threadIdx.x;
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
    // lane j < T: row j's statistics (lanes reduce the chunks together), its
    // draft test and its two candidates
    const int tok_next = lane + 1 < T ? a.tokens[r0 + lane + 1] : -1;
    const float u = lane < T ? a.uniforms[r0 + lane] : 1.0f;
    const float l_d = (lane + 1 < T && tok_next >= 0 && tok_next < a.vocab)
                          ? to_f(static_cast<const TIn*>(a.logits)[(int64_t)(r0 + lane) * a.vocab + tok_next]) * a.inv_tau
                          : -CUDART_INF_F;
    const SampleStat* pp = reinterpret_cast<const SampleStat*>(a.partial) + (int64_t)r0 * a.num_chunks;
    SampleStat mine = stat_empty();
    for (int j = 0; j < T; ++j) {
        SampleStat c = stat_empty();
        for (int k = lane; k < a.num_chunks; k += 32) c = stat_merge(c, pp[(int64_t)j * a.num_chunks + k]);
        c = stat_warp(c);
        if (lane == j) mine = c;
    }
    const float p = (lane + 1 < T) ? __expf(l_d - mine.m) / mine.s : 0.0f;
    const unsigned miss = __ballot_sync(0xffffffffu, lane + 1 < T && !(u < p));
    const int acc = miss ? __ffs(miss) - 1 : T - 1;
    const int cand = (acc < T - 1) ? mine.i2 : mine.i1;            // residual sample, or the bonus token
    const int nxt = __shfl_sync(0xffffffffu, cand, acc);
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

namespace q3kv {

cudaError_t launch_accept_sample(const AcceptArgs& a, cudaStream_t stream) {
    if (a.num_rows > 0) {
        const dim3 grid((unsigned)a.num_chunks, (unsigned)a.num_rows);
        if (a.dtype == Q3KV_F32) sample_stats_kernel<float><<<grid, kArgThreads, 0, stream>>>(a);
        else sample_stats_kernel<__nv_bfloat16><<<grid, kArgThreads, 0, stream>>>(a);
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
    if (a.dtype == Q3KV_F32) return cudaLaunchKernelEx(&cfg, sample_accept_kernel<float>, a);
    return cudaLaunchKernelEx(&cfg, sample_accept_kernel<__nv_bfloat16>, a);
}

}  // namespace q3kv

// ---------------------------------------------------------------------------
// Top-p nucleus for the sampled acceptance.
//
// Source: "Quasar" (q27 wiki), "Model tool protocol" bullet (sampled
// speculative decode: top-p nucleus, Gumbel-max, rejection-sampled
// acceptance) and the sampler paragraph of "Serving" (the nucleus is taken on
// the temperature-scaled distribution).  Reading: the nucleus of row j is
// {x : l_x >= l*}, l* the largest logit of the row whose tokens at or above it
// carry at least top_p of softmax(l / tau) -- every token tied with the cut is
// kept.
//
// The cut is found by a radix select over the logits' order keys, 8 bits per
// level from the top (4 levels for f32 logits, 2 for bf16, whose low 16 bits
// are zero): each level histograms the probability mass of the tokens that
// match the prefix found so far, and a one-CTA-per-row step picks the bin where
// the mass counted from the top first reaches top_p of the total.  Masses are
// 2^-40 fixed point (each e^(l/tau - max) <= 1), so the sums are exact integers
// whatever the order of the atomic adds: the search is deterministic.
namespace q3kv {
namespace {


struct NucleusRow {
    float m;                       // max of l / tau
    uint32_t prefix;               // order-key bits of the cut found so far
    unsigned long long above;      // mass of the tokens above the prefix's key range
    unsigned long long target;     // ceil(top_p * total mass)
    unsigned long long zn;         // mass of the nucleus (after the last level)
    uint32_t key_star;             // order key of l*
};
static_assert(sizeof(NucleusRow) <= kNucleusRowBytes, "nucleus row");

// Monotone key of a logit value (-0 taken as +0, so equal values get equal keys).
__device__ __forceinline__ uint32_t order_key(float l) {
    const uint32_t u = __float_as_uint(l == 0.0f ? 0.0f : l);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ NucleusRow* nrow(const AcceptArgs& a, int row) {
    return reinterpret_cast<NucleusRow*>(static_cast<uint8_t*>(a.nucleus) + (size_t)row * kNucleusRowBytes);
}
__device__ __forceinline__ unsigned long long* nhist(const AcceptArgs& a, int row) {
    return reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.nucleus) + (size_t)a.num_rows * kNucleusRowBytes +
                                                 (size_t)row * kNucleusHistBytes);
}

// Per (chunk, row): max of l / tau (into the chunk partial's m), NaN flag.
template <typename T>
__global__ void __launch_bounds__(kArgThreads) nucleus_max_kernel(AcceptArgs a) {
    __shared__ float red[kArgThreads / 32];
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int64_t c0 = (int64_t)chunk * a.chunk_elems;
    const int64_t c1 = min((int64_t)a.vocab, c0 + a.chunk_elems);
    const T* lg = static_cast<const T*>(a.logits) + (int64_t)row * a.vocab;
    float m = -CUDART_INF_F;
    bool nan = false;
    for_each_logit(a, lg, c0, c1, [&](int64_t, float raw) {
        const float l = raw * a.inv_tau;
        nan |= (l != l);
        m = fmaxf(m, l);
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_NONFINITE_INPUT);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kArgThreads / 32; ++w) m = fmaxf(m, red[w]);
        SampleStat st = stat_empty();
        st.m = m;
        reinterpret_cast<SampleStat*>(a.partial)[(int64_t)row * a.num_chunks + chunk] = st;
    }
}

// One CTA per row: the row maximum; clears the level-0 histogram.
__global__ void __launch_bounds__(256) nucleus_init_kernel(AcceptArgs a) {
    const int row = blockIdx.x;
    __shared__ float red[8];
    const SampleStat* pp = reinterpret_cast<const SampleStat*>(a.partial) + (int64_t)row * a.num_chunks;
    float m = -CUDART_INF_F;
    for (int k = threadIdx.x; k < a.num_chunks; k += 256) m = fmaxf(m, pp[k].m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    nhist(a, row)[threadIdx.x] = 0ull;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
        NucleusRow* r = nrow(a, row);
        r->m = m;
        r->prefix = 0u;
        r->above = 0ull;
        r->target = 0ull;
        r->zn = 0ull;
        r->key_star = 0u;
    }
}

// Per (chunk, row): fixed-point mass histogram of the next 8 key bits of the
// tokens whose higher bits equal the prefix.  Each warp adds into its own
// shared-memory histogram (logits bunch into few bins at the top levels, so a
// shared one would serialise the warps); the eight are summed at the end.
template <typename T>
__global__ void __launch_bounds__(kArgThreads) nucleus_hist_kernel(AcceptArgs a, int level) {
    __shared__ unsigned long long h[kArgThreads / 32][256];
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int w = 0; w < kArgThreads / 32; ++w) h[w][threadIdx.x] = 0ull;
    __syncthreads();
    const NucleusRow* r = nrow(a, row);
    const float m = r->m;
    const uint32_t prefix = r->prefix;
    const int shift = 24 - 8 * level;
    const int64_t c0 = (int64_t)chunk * a.chunk_elems;
    const int64_t c1 = min((int64_t)a.vocab, c0 + a.chunk_elems);
    const T* lg = static_cast<const T*>(a.logits) + (int64_t)row * a.vocab;
    for_each_logit(a, lg, c0, c1, [&](int64_t, float raw) {
        const uint32_t key = order_key(raw);
        if (level > 0 && (key >> (shift + 8)) != prefix) return;
        // mass = round(e 2^40) for e = e^(l/tau - max) <= 1, as an exact split
        // at 2^20: e 2^20 and its fraction are exact floats
        const float e20 = __expf(raw * a.inv_tau - m) * 1048576.0f;
        const uint32_t hi = (uint32_t)e20;
        const uint32_t lo = __float2uint_rn((e20 - (float)hi) * 1048576.0f);
        const unsigned long long mass = ((unsigned long long)hi << 20) + lo;
        if (mass) atomicAdd(&h[warp][(key >> shift) & 0xFFu], mass);
    });
    __syncthreads();
    unsigned long long t = 0ull;
#pragma unroll
    for (int w = 0; w < kArgThreads / 32; ++w) t += h[w][threadIdx.x];
    if (t) atomicAdd(&nhist(a, row)[threadIdx.x], t);
}

// One CTA per row: the bin where the mass counted from the top first reaches
// the target; extends the prefix; clears the histogram for the next level.
// Warp 0 scans: lane l holds bins 8 (31 - l) .. 8 (31 - l) + 7 (the top bins
// in lane 0), and a prefix sum over the lanes gives each lane the mass above.
__global__ void __launch_bounds__(256) nucleus_select_kernel(AcceptArgs a, int level, int last) {
    const int row = blockIdx.x;
    __shared__ unsigned long long h[256];
    unsigned long long* gh = nhist(a, row);
    h[threadIdx.x] = gh[threadIdx.x];
    __syncthreads();
    gh[threadIdx.x] = 0ull;
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    NucleusRow* r = nrow(a, row);
    const int base = 8 * (31 - lane);
    unsigned long long mine = 0ull;
#pragma unroll
    for (int j = 0; j < 8; ++j) mine += h[base + j];
    unsigned long long incl = mine;                 // lanes 0..lane (lane 0 = the top bins)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    unsigned long long target;
    if (level == 0) {
        const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
        const double t = ceil((double)a.top_p * (double)total);
        target = t < (double)total ? (unsigned long long)t : total;
        if (lane == 0) r->target = target;
    } else {
        target = r->target;
    }
    const unsigned long long above0 = r->above;
    // the first lane from the top whose inclusive mass reaches the target
    const unsigned hit = __ballot_sync(0xffffffffu, above0 + incl >= target);
    const int sl = hit ? __ffs(hit) - 1 : 31;
    if (lane == sl) {
        unsigned long long cum = above0 + incl - mine;     // mass above this lane's bins
        int sel = base;
        for (int b = base + 7; b >= base; --b) {
            if (cum + h[b] >= target) {
                sel = b;
                break;
            }
            cum += h[b];
        }
        r->prefix = (r->prefix << 8) | (uint32_t)sel;
        r->above = cum;
        if (last) {
            r->key_star = r->prefix << (24 - 8 * level);   // bf16 stops after two levels: the low key bits are the same
            r->zn = cum + h[sel];
        }
    }
}

// Per (chunk, row): Gumbel-max candidates over the nucleus (overall and
// without the row's next query token).
template <typename T>
__global__ void __launch_bounds__(kArgThreads) nucleus_gumbel_kernel(AcceptArgs a, uint32_t low_fill) {
    __shared__ SampleStat red[kArgThreads / 32];
    const int row = blockIdx.y, chunk = blockIdx.x;
    const int64_t c0 = (int64_t)chunk * a.chunk_elems;
    const int64_t c1 = min((int64_t)a.vocab, c0 + a.chunk_elems);
    const T* lg = static_cast<const T*>(a.logits) + (int64_t)row * a.vocab;
    const int excl = row + 1 < a.num_rows ? a.tokens[row + 1] : -1;
    const uint32_t key_star = nrow(a, row)->key_star | low_fill;
    SampleStat st = stat_empty();
    for_each_logit(a, lg, c0, c1, [&](int64_t k, float raw) {
        if ((order_key(raw) | low_fill) < key_star) return;
        const float key = raw * a.inv_tau - logf(-logf(noise_uniform(a.seed, (uint32_t)row, (uint32_t)k)));
        if (beats(key, (int)k, st.k1, st.i1)) { st.k1 = key; st.i1 = (int)k; }
        if ((int)k != excl && beats(key, (int)k, st.k2, st.i2)) { st.k2 = key; st.i2 = (int)k; }
    });
    st = stat_warp(st);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = st;
    __syncthreads();
    if (threadIdx.x < 32) {
        SampleStat c = threadIdx.x < kArgThreads / 32 ? red[threadIdx.x] : stat_empty();
        c = stat_warp(c);
        if (threadIdx.x == 0) reinterpret_cast<SampleStat*>(a.partial)[(int64_t)row * a.num_chunks + chunk] = c;
    }
}

// One warp per slot: the draft tests against the filtered distribution, then
// the residual or bonus candidate.
template <typename TIn>
__global__ void __launch_bounds__(32) nucleus_accept_kernel(AcceptArgs a, uint32_t low_fill) {
    const int b = blockIdx.x, lane = threadIdx.x;
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
    const int tok_next = lane + 1 < T ? a.tokens[r0 + lane + 1] : -1;
    const float u = lane < T ? a.uniforms[r0 + lane] : 1.0f;
    float p = 0.0f;
    if (lane + 1 < T && tok_next >= 0 && tok_next < a.vocab) {
        const NucleusRow* r = nrow(a, r0 + lane);
        const float raw = to_f(static_cast<const TIn*>(a.logits)[(int64_t)(r0 + lane) * a.vocab + tok_next]);
        if ((order_key(raw) | low_fill) >= (r->key_star | low_fill)) {
            const float e20 = __expf(raw * a.inv_tau - r->m) * 1048576.0f;   // the histogram's fixed point
            const uint32_t hi = (uint32_t)e20;
            const uint32_t lo = __float2uint_rn((e20 - (float)hi) * 1048576.0f);
            p = (float)((double)(((unsigned long long)hi << 20) + lo) / (double)r->zn);
        }
    }
    const SampleStat* pp = reinterpret_cast<const SampleStat*>(a.partial) + (int64_t)r0 * a.num_chunks;
    SampleStat mine = stat_empty();
    for (int j = 0; j < T; ++j) {
        SampleStat c = stat_empty();
        for (int k = lane; k < a.num_chunks; k += 32) c = stat_merge(c, pp[(int64_t)j * a.num_chunks + k]);
        c = stat_warp(c);
        if (lane == j) mine = c;
    }
    const unsigned miss = __ballot_sync(0xffffffffu, lane + 1 < T && !(u < p));
    const int acc = miss ? __ffs(miss) - 1 : T - 1;
    const int cand = (acc < T - 1) ? mine.i2 : mine.i1;
    const int nxt = __shfl_sync(0xffffffffu, cand, acc);
    if (lane == 0) {
        a.n_accepted[b] = acc;
        a.next_token[b] = nxt;
        a.committed_len[b] = L - (T - 1 - acc);
    }
}

template <typename T>
cudaError_t launch_nucleus_typed(const AcceptArgs& a, cudaStream_t stream) {
    // bf16 logits: two levels of 8 key bits decide the value (the low 16 bits
    // of every key are equal: 0 for positive values, all ones for negative
    // ones; comparisons below fill them with ones so both read the same)
    const int levels = (a.dtype == Q3KV_F32) ? 4 : 2;
    const uint32_t low_fill = (a.dtype == Q3KV_F32) ? 0u : 0xFFFFu;
    if (a.num_rows > 0) {
        const dim3 grid((unsigned)a.num_chunks, (unsigned)a.num_rows);
        nucleus_max_kernel<T><<<grid, kArgThreads, 0, stream>>>(a);
        nucleus_init_kernel<<<a.num_rows, 256, 0, stream>>>(a);
        for (int lv = 0; lv < levels; ++lv) {
            nucleus_hist_kernel<T><<<grid, kArgThreads, 0, stream>>>(a, lv);
            nucleus_select_kernel<<<a.num_rows, 256, 0, stream>>>(a, lv, lv == levels - 1 ? 1 : 0);
        }
        nucleus_gumbel_kernel<T><<<grid, kArgThreads, 0, stream>>>(a, low_fill);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    nucleus_accept_kernel<T><<<a.num_slots, 32, 0, stream>>>(a, low_fill);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_accept_nucleus(const AcceptArgs& a, cudaStream_t stream) {
    if (a.dtype == Q3KV_F32) return launch_nucleus_typed<float>(a, stream);
    return launch_nucleus_typed<__nv_bfloat16>(a, stream);
}

}  // namespace q3kv
