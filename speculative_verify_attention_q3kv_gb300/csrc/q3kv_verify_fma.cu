// Verify attention, CUDA-core fp32 leg (the reference flash-decode leg); also
// the leg that reads the turbo5k-style cache (template FMT = kFmtT5k: 5-bit
// Lloyd-Max K records, 3-bit V records, in that format's page layout).
//
// Source: "Quasar" (q27 wiki), "Self-speculation as the whole design" (one
// shared-KV verify of all drafted tokens), the Defaults paragraph of
// "Serving" (an fd2 reference flash-decode leg beside the MMA legs), and
// "KV cache" (verify reads the 3-bit cache directly).
//
// One CTA = (slot, kv head, chunk of <= 64 query rows, split of the context).
// Rows of a kv head are r = t*8 + hh (token t, q head g*8 + hh), so the GQA
// group and all drafted tokens share every K/V byte the CTA reads.  The CTA
// walks its positions in tiles of 32: dequantise K and V into shared memory
// (float32, exact), S = Q K^T on CUDA cores, online softmax, O += P V.  With
// one split the CTA rotates its result back by H and stores it; otherwise it
// stores its partial (m, l, o) for the merge kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "q3kv_common.cuh"
#include "q3kv_internal.h"

namespace q3kv {
namespace {

constexpr int kTile = 32;                 // positions per tile
constexpr int kKStride = 260;             // padded row of the K tile (floats)
constexpr int kThreads = 256;

struct FmaSmem {
    float q[kFmaRows][kHeadDim];          // rotated, scaled queries; reused for the output
    float k[kTile][kKStride];
    float v[kTile][kHeadDim];
    float p[kFmaRows][kTile];
    float m_run[kFmaRows];
    float l_run[kFmaRows];
    float alpha[kFmaRows];
};

// Decode the 32 codes of block b from its three words into (c - 3.5) * s.
__device__ __forceinline__ void decode_block(const uint8_t* rec, int b, float* dst) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(rec) + 3 * b;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
    const float s = __half2float(reinterpret_cast<const __half*>(rec + 96)[b]);
    const uint32_t ws[3] = {w0, w1, w2};
#pragma unroll
    for (int m = 0; m < 15; ++m) {
        const uint32_t word = ws[m / 5] >> (3 * (m % 5));
        dst[2 * m] = ((float)(word & 7u) - 3.5f) * s;
        dst[2 * m + 1] = ((float)((word >> 16) & 7u) - 3.5f) * s;
    }
    const uint32_t c30 = ((w0 >> 15) & 1u) | (((w1 >> 15) & 1u) << 1) | (((w2 >> 15) & 1u) << 2);
    const uint32_t c31 = ((w0 >> 31) & 1u) | (((w1 >> 31) & 1u) << 1) | (((w2 >> 31) & 1u) << 2);
    dst[30] = ((float)c30 - 3.5f) * s;
    dst[31] = ((float)c31 - 3.5f) * s;
}

// turbo5k K: the 32 elements of block b (dims 32 b ..) from the low nibbles,
// the 5th-bit plane and the scale of their 128-dim half: c_code * s.
__device__ __forceinline__ void decode_t5k_block(const uint8_t* rec, int b, const T5kTable& tab, float* dst) {
    const uint32_t* nib = reinterpret_cast<const uint32_t*>(rec) + 4 * b;        // 16 bytes: 32 nibbles
    const uint32_t top = reinterpret_cast<const uint32_t*>(rec + 128)[b];       // 32 fifth bits
    const float s = __half2float(reinterpret_cast<const __half*>(rec + 160)[b >> 2]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w = nib[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int d = 8 * j + e;
            const uint32_t c = ((w >> (4 * e)) & 0xFu) | (((top >> d) & 1u) << 4);
            dst[d] = tab.c[c] * s;
        }
    }
}

template <typename TIn, int FMT>
__global__ void __launch_bounds__(kThreads, 1) verify_fma_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    FmaSmem& sm = *reinterpret_cast<FmaSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // units run fastest in the grid, each slot's last row chunk first (see
    // the tensor-core leg)
    const int unit_id = blockIdx.x;
    const int split = blockIdx.y;
    const int chunk = a.row_chunks - 1 - unit_id % a.row_chunks;
    const int g = (unit_id / a.row_chunks) % a.num_kv_heads;
    const int slot = unit_id / (a.row_chunks * a.num_kv_heads);

    const int T = a.n_q[slot];
    const int L = a.ctx_len[slot];
    if (T <= 0) return;
    if (T > a.max_n_q || T > L || L > a.max_pages_per_slot * kPageSize) {
        if (tid == 0 && split == 0 && chunk == 0 && g == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    const int R = kGroup * T;
    const int row0 = chunk * kFmaRows;
    const int Rc = min(kFmaRows, R - row0);
    if (Rc <= 0) return;
    const int n_pages = (L + kPageSize - 1) / kPageSize;
    const int split_pages = split_pages_of(a);
    const int n_splits = (n_pages + split_pages - 1) / split_pages;
    if (n_splits > a.num_splits) {   // context longer than the host bound the workspace was sized for
        if (tid == 0 && split == 0 && chunk == 0 && g == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    if (split >= n_splits) return;
    const int p_begin = split * split_pages * kPageSize;
    const int p_end = min(L, p_begin + split_pages * kPageSize);
    const int N = L - T;
    const int Hq = a.num_kv_heads * kGroup;
    const int64_t q_base = a.q_offsets[slot];

    // ---- queries: load, rotate by H, scale by 1/16 (H) * 1/16 (softmax)
    const TIn* qin = static_cast<const TIn*>(a.q);
    for (int idx = tid; idx < Rc * kHeadDim; idx += kThreads) {
        const int r = idx / kHeadDim, d = idx % kHeadDim;
        const int ra = row0 + r;
        const int t = ra / kGroup, hh = ra % kGroup;
        sm.q[r][d] = load_in(qin + ((q_base + t) * Hq + g * kGroup + hh) * kHeadDim + d);
    }
    if (tid < kFmaRows) {
        sm.m_run[tid] = -CUDART_INF_F;
        sm.l_run[tid] = 0.0f;
    }
    __syncthreads();
    rotate_rows(&sm.q[0][0], Rc);
    for (int idx = tid; idx < Rc * kHeadDim; idx += kThreads) sm.q[idx / kHeadDim][idx % kHeadDim] *= (1.0f / 256.0f);

    float acc_o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc_o[j][c] = 0.0f;
    const int c4 = tid & 63;   // dims 4*c4 .. 4*c4+3
    const int rg = tid >> 6;   // rows 16*rg .. 16*rg+15

    const int32_t* pt_row = a.page_table + (int64_t)slot * a.max_pages_per_slot;
    bool bad_page = false;

    for (int p0 = p_begin; p0 < p_end; p0 += kTile) {
        __syncthreads();   // previous tile fully consumed (and q ready on the first pass)
        {   // dequantise: thread = (position i, block b)
            const int i = tid >> 3, b = tid & 7;
            const int pos = p0 + i;
            float kv_k[32], kv_v[32];
            bool ok = pos < p_end;
            int32_t page = 0;
            if (ok) {
                page = pt_row[pos / kPageSize];
                if (page < 0 || page >= a.num_pages) { ok = false; bad_page = true; }
            }
            if (ok) {
                if (FMT == kFmtT5k) {
                    decode_t5k_block(a.pool + t5k_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 0, pos % kPageSize),
                                     b, a.t5k, kv_k);
                    decode_block(a.pool + t5k_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 1, pos % kPageSize),
                                 b, kv_v);
                } else {
                    const uint8_t* rk = a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 0, pos % kPageSize);
                    const uint8_t* rv = a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 1, pos % kPageSize);
                    decode_block(rk, b, kv_k);
                    decode_block(rv, b, kv_v);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) { kv_k[e] = 0.0f; kv_v[e] = 0.0f; }
            }
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                *reinterpret_cast<float4*>(&sm.k[i][32 * b + e]) = make_float4(kv_k[e], kv_k[e + 1], kv_k[e + 2], kv_k[e + 3]);
                *reinterpret_cast<float4*>(&sm.v[i][32 * b + e]) = make_float4(kv_v[e], kv_v[e + 1], kv_v[e + 2], kv_v[e + 3]);
            }
        }
        __syncthreads();

        {   // scores for rows warp + 8j, position lane; online softmax
            float s[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) s[j] = 0.0f;
            const float* krow = sm.k[lane];
            for (int d = 0; d < kHeadDim; d += 4) {
                const float4 kk = *reinterpret_cast<const float4*>(krow + d);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int r = warp + 8 * j;
                    const float4 qq = *reinterpret_cast<const float4*>(&sm.q[r][d]);
                    s[j] = fmaf(qq.x, kk.x, s[j]);
                    s[j] = fmaf(qq.y, kk.y, s[j]);
                    s[j] = fmaf(qq.z, kk.z, s[j]);
                    s[j] = fmaf(qq.w, kk.w, s[j]);
                }
            }
            const int pos = p0 + lane;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = warp + 8 * j;
                if (r >= Rc) continue;                    // warp-uniform
                const int t = (row0 + r) / kGroup;
                const bool vis = pos < p_end && pos <= N + t;
                const float sv = vis ? s[j] : -CUDART_INF_F;
                float mx = sv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = sm.m_run[r];
                const float m_new = fmaxf(m_old, mx);
                float pr = 0.0f, alpha = 1.0f;
                if (m_new != -CUDART_INF_F) {
                    pr = vis ? expf(sv - m_new) : 0.0f;
                    alpha = expf(m_old - m_new);
                }
                float sum = pr;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                sm.p[r][lane] = pr;
                __syncwarp();
                if (lane == 0) {
                    sm.m_run[r] = m_new;
                    sm.l_run[r] = sm.l_run[r] * alpha + sum;
                    sm.alpha[r] = alpha;
                }
            }
        }
        __syncthreads();

        {   // O = O * alpha + P V
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int r = 16 * rg + j;
                const float al = (r < Rc) ? sm.alpha[r] : 1.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) acc_o[j][c] *= al;
            }
            if (16 * rg < Rc) {
                for (int p = 0; p < kTile; ++p) {
                    const float4 vv = *reinterpret_cast<const float4*>(&sm.v[p][4 * c4]);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float pr = sm.p[min(16 * rg + j, kFmaRows - 1)][p];
                        acc_o[j][0] = fmaf(pr, vv.x, acc_o[j][0]);
                        acc_o[j][1] = fmaf(pr, vv.y, acc_o[j][1]);
                        acc_o[j][2] = fmaf(pr, vv.z, acc_o[j][2]);
                        acc_o[j][3] = fmaf(pr, vv.w, acc_o[j][3]);
                    }
                }
            }
        }
    }
    if (bad_page && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_PAGE);
    __syncthreads();

    const int unit = (slot * a.num_kv_heads + g) * a.row_chunks + chunk;
    float* out = a.out;
    if (n_splits == 1) {
        // normalise into shared memory, rotate back, store
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int r = 16 * rg + j;
            if (r < Rc) {
                const float inv = 1.0f / sm.l_run[r];
#pragma unroll
                for (int c = 0; c < 4; ++c) sm.q[r][4 * c4 + c] = acc_o[j][c] * inv;
            }
        }
    } else {
        float* po = a.part_o + ((int64_t)unit * a.num_splits + split) * kFmaRows * kHeadDim;
        float* pml = a.part_ml + ((int64_t)unit * a.num_splits + split) * kFmaRows * 2;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int r = 16 * rg + j;
            if (r < Rc)
                *reinterpret_cast<float4*>(po + r * kHeadDim + 4 * c4) =
                    make_float4(acc_o[j][0], acc_o[j][1], acc_o[j][2], acc_o[j][3]);
        }
        if (tid < Rc) {
            pml[2 * tid] = sm.m_run[tid];
            pml[2 * tid + 1] = sm.l_run[tid];
        }
        return;   // the merge kernel combines the splits
    }
    __syncthreads();
    rotate_rows(&sm.q[0][0], Rc);
    for (int idx = tid; idx < Rc * kHeadDim; idx += kThreads) {
        const int r = idx / kHeadDim, d = idx % kHeadDim;
        const int ra = row0 + r;
        const int t = ra / kGroup, hh = ra % kGroup;
        out[((q_base + t) * Hq + g * kGroup + hh) * kHeadDim + d] = sm.q[r][d] * 0.0625f;
    }
}

}  // namespace

namespace {
template <typename TIn, int FMT>
cudaError_t launch_fma_typed(const VerifyArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(FmaSmem);
    const dim3 grid((unsigned)(a.num_slots * a.num_kv_heads * a.row_chunks), (unsigned)a.num_splits);
    const cudaError_t e =
        cudaFuncSetAttribute(verify_fma_kernel<TIn, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    verify_fma_kernel<TIn, FMT><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_verify_fma(const VerifyArgs& a, cudaStream_t stream) {
    const bool f32 = a.dtype == Q3KV_F32;
    if (a.fmt == kFmtT5k)
        return f32 ? launch_fma_typed<float, kFmtT5k>(a, stream) : launch_fma_typed<__nv_bfloat16, kFmtT5k>(a, stream);
    return f32 ? launch_fma_typed<float, kFmtQ3>(a, stream) : launch_fma_typed<__nv_bfloat16, kFmtQ3>(a, stream);
}

}  // namespace q3kv
