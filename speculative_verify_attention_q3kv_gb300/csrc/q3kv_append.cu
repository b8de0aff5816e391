// Quantise-append: rotate each new K/V head vector by the Walsh-Hadamard
// matrix, code it with the 3-bit block codec and store its 112-byte record.
//
// Source: "Quasar" (q27 wiki), "turbo3 3-bit KV cache" and the "KV cache"
// stack bullet (WHT-rotated 3-bit blocks, symmetric K+V; the same cache serves
// decode, verify and batched prefill).  The codec's exact rounding is this
// library's stated one:
//   y = H x by radix-2 butterflies over index bits 0..7 in float32 RNE, then
//       one exact multiply by 1/16;
//   s = fp16_rn(absmax_fp32 / 3.5f)  (IEEE divide);
//   q = clamp(rint(fp32(y / s) + 3.5f), 0, 7), q = 4 when s == 0.
// Every float operation below is an explicitly rounded intrinsic, so the
// compiler cannot contract or reorder it and the codes match the oracle bit
// for bit.
//
// Work layout: one warp per (slot, token, kv head, K|V) vector.  Lane l holds
// elements 8l..8l+7, so butterfly strides 1, 2, 4 stay in registers and strides
// 8..128 are lane exchanges (shfl_xor 1..16).  A 32-element block lives on
// four consecutive lanes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q3kv_internal.h"

namespace q3kv {
namespace {

__device__ __forceinline__ void load8(const float* src, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(src)[0];
    const float4 b = reinterpret_cast<const float4*>(src)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* src, float (&x)[8]) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[0];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Code-word bits contributed by element e (0..31 inside its block) with code c.
// Returns the contribution to words 0, 1, 2 of the block.
__device__ __forceinline__ void place_code(int e, uint32_t c, uint32_t (&w)[3]) {
    if (e < 30) {
        const int m = e >> 1;
        const int off = ((e & 1) << 4) + 3 * (m % 5);
        const int wi = m / 5;
        const uint32_t bits = c << off;
        w[0] |= (wi == 0) ? bits : 0u;
        w[1] |= (wi == 1) ? bits : 0u;
        w[2] |= (wi == 2) ? bits : 0u;
    } else {
        const int top = (e == 30) ? 15 : 31;
#pragma unroll
        for (int k = 0; k < 3; ++k) w[k] |= ((c >> k) & 1u) << top;
    }
}

// turbo5k K (template FMT = kFmtT5k, K vectors only): after the same rotation,
// per 128-dim half (lanes 16h .. 16h + 15) the fp16 root-mean-square scale
// (float32 squares summed from each lane's first element on, then over lane
// pairs 1, 2, 4, 8 apart), codes = the number of boundaries below y / s, and a
// 164-byte record: low nibbles (4 bytes per lane), 5th bits (1 byte per lane),
// the two scales.
__device__ __forceinline__ void t5k_encode_store(const float (&x)[8], int lane, const T5kTable& tab, uint8_t* rec,
                                                 bool& overflow) {
    float acc = __fmul_rn(x[0], x[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) acc = __fadd_rn(acc, __fmul_rn(x[i], x[i]));
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, m));
    const __half s16 = __float2half_rn(__fsqrt_rn(__fmul_rn(acc, 0.0078125f)));
    const float s = __half2float(s16);
    overflow = isinf(s);
    uint32_t nib = 0u, top = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t c = 16u;
        if (s != 0.0f) {
            const float v = __fdiv_rn(x[i], s);
            c = 0u;
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1)   // boundaries below v, by bisection
                if (c + step - 1 < 31u && v > tab.b[c + step - 1]) c += step;
        }
        nib |= (c & 0xFu) << (4 * i);
        top |= (c >> 4) << i;
    }
    reinterpret_cast<uint32_t*>(rec)[lane] = nib;
    rec[128 + lane] = (uint8_t)top;
    if ((lane & 15) == 0) reinterpret_cast<__half*>(rec + 160)[lane >> 4] = s16;
}

template <typename T, int FMT>
__global__ void __launch_bounds__(128) append_kernel(AppendArgs a) {
    // launched with programmatic stream serialisation: let the next grid be
    // scheduled, and wait for the previous one before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int slot = blockIdx.y;
    const int t = blockIdx.x;
    const int n_new = a.n_new[slot];
    if (t >= n_new) return;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (n_new > a.max_n_new) {
        if (t == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    const int64_t pos = (int64_t)a.slot_len[slot] + t;
    if (pos < 0 || pos >= (int64_t)a.max_pages_per_slot * kPageSize) {
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    const int32_t page = a.page_table[(int64_t)slot * a.max_pages_per_slot + (pos / kPageSize)];
    if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_PAGE);
        return;
    }
    const int64_t row = (int64_t)a.row_offsets[slot] + t;
    const T* kin = static_cast<const T*>(a.k);
    const T* vin = static_cast<const T*>(a.v);

    for (int vec = warp; vec < a.num_kv_heads * 2; vec += blockDim.x >> 5) {
        const int head = vec >> 1;
        const int kv = vec & 1;
        const T* src = (kv == 0 ? kin : vin) + (row * a.num_kv_heads + head) * kHeadDim + lane * 8;
        float x[8];
        load8(src, x);

        bool finite = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) finite = finite && isfinite(x[i]);

        // butterflies over index bits 0, 1, 2 (in registers)
#pragma unroll
        for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if ((i & h) == 0) {
                    const float lo = x[i], hi = x[i + h];
                    x[i] = __fadd_rn(lo, hi);
                    x[i + h] = __fsub_rn(lo, hi);
                }
            }
        }
        // butterflies over index bits 3..7 (lane bits 0..4)
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
                x[i] = upper ? __fsub_rn(other, x[i]) : __fadd_rn(x[i], other);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], 0.0625f);

        if (FMT == kFmtT5k && kv == 0) {
            bool overflow = false;
            t5k_encode_store(x, lane, a.t5k,
                             a.pool + t5k_offset(a.num_layers, a.num_kv_heads, page, a.layer, head, 0,
                                                 (int)(pos % kPageSize)),
                             overflow);
            const bool any_nonfinite = __any_sync(0xffffffffu, !finite);
            const bool any_overflow = __any_sync(0xffffffffu, overflow);
            if (lane == 0 && a.status) {
                if (any_nonfinite) atomicOr(a.status, Q3KV_STATUS_NONFINITE_INPUT);
                else if (any_overflow) atomicOr(a.status, Q3KV_STATUS_SCALE_OVERFLOW);
            }
            continue;
        }

        // block absmax over 4 lanes
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const __half s16 = __float2half_rn(__fdiv_rn(amax, 3.5f));
        const float s = __half2float(s16);

        uint32_t w[3] = {0u, 0u, 0u};
        const int e0 = (lane & 3) * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t c = 4u;
            if (s != 0.0f) {
                float tq = rintf(__fadd_rn(__fdiv_rn(x[i], s), 3.5f));
                tq = fminf(fmaxf(tq, 0.0f), 7.0f);   // NaN -> 0 (non-finite input is flagged)
                c = (uint32_t)tq;
            }
            place_code(e0 + i, c, w);
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            w[k] |= __shfl_xor_sync(0xffffffffu, w[k], 1);
            w[k] |= __shfl_xor_sync(0xffffffffu, w[k], 2);
        }

        const bool any_nonfinite = __any_sync(0xffffffffu, !finite);
        const bool any_overflow = __any_sync(0xffffffffu, isinf(s));
        if (lane == 0 && a.status) {
            if (any_nonfinite) atomicOr(a.status, Q3KV_STATUS_NONFINITE_INPUT);
            else if (any_overflow) atomicOr(a.status, Q3KV_STATUS_SCALE_OVERFLOW);
        }

        uint8_t* rec = a.pool + (FMT == kFmtT5k
                                     ? t5k_offset(a.num_layers, a.num_kv_heads, page, a.layer, head, kv,
                                                  (int)(pos % kPageSize))
                                     : record_offset(a.num_layers, a.num_kv_heads, page, a.layer, head, kv,
                                                     (int)(pos % kPageSize)));
        const int blk = lane >> 2;
        const int k = lane & 3;
        if (k < 3) reinterpret_cast<uint32_t*>(rec)[3 * blk + k] = w[k];
        else reinterpret_cast<__half*>(rec + 96)[blk] = s16;
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    if (a.max_n_new == 0 || a.num_slots == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.max_n_new, (unsigned)a.num_slots);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.fmt == kFmtT5k) {
        if (a.dtype == Q3KV_F32) return cudaLaunchKernelEx(&cfg, append_kernel<float, kFmtT5k>, a);
        return cudaLaunchKernelEx(&cfg, append_kernel<__nv_bfloat16, kFmtT5k>, a);
    }
    if (a.dtype == Q3KV_F32) return cudaLaunchKernelEx(&cfg, append_kernel<float, kFmtQ3>, a);
    return cudaLaunchKernelEx(&cfg, append_kernel<__nv_bfloat16, kFmtQ3>, a);
}

}  // namespace q3kv
