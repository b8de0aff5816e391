// Append into the fp8 E4M3 comparison cache.
//
// Source: "Quasar" (q27 wiki), "KV cache" stack bullet: K and V stored as fp8
// E4M3 with a scale-free, saturating conversion (no per-row scale, no
// rotation).  Each new K/V head vector becomes a 256-byte record of E4M3
// bytes, dims in order, in the same page layout as the 3-bit cache.  The
// conversion is cvt.rn.satfinite: round to nearest even, magnitudes above 448
// (and infinities) to +-448, NaN to NaN; a non-finite input also sets
// Q3KV_STATUS_NONFINITE_INPUT.
//
// Work layout: one warp per (slot, token, kv head, K|V) vector; lane l
// converts elements 8l..8l+7 and stores their 8 bytes.
#include <cuda_bf16.h>

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

// Two floats -> two E4M3 bytes (lo in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <typename T>
__global__ void __launch_bounds__(128) append_fp8_kernel(AppendArgs a) {
    // programmatic stream serialisation, as the 3-bit append
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
        float x[8];
        load8((kv == 0 ? kin : vin) + (row * a.num_kv_heads + head) * kHeadDim + lane * 8, x);
        bool finite = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) finite = finite && isfinite(x[i]);
        const uint32_t w0 = e4m3x2(x[0], x[1]) | (e4m3x2(x[2], x[3]) << 16);
        const uint32_t w1 = e4m3x2(x[4], x[5]) | (e4m3x2(x[6], x[7]) << 16);
        if (__any_sync(0xffffffffu, !finite) && lane == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_NONFINITE_INPUT);
        uint8_t* rec = a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, head, kv,
                                              (int)(pos % kPageSize), kFp8RecordBytes);
        reinterpret_cast<uint2*>(rec)[lane] = make_uint2(w0, w1);
    }
}

}  // namespace

cudaError_t launch_append_fp8(const AppendArgs& a, cudaStream_t stream) {
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
    if (a.dtype == Q3KV_F32) return cudaLaunchKernelEx(&cfg, append_fp8_kernel<float>, a);
    return cudaLaunchKernelEx(&cfg, append_fp8_kernel<__nv_bfloat16>, a);
}

}  // namespace q3kv
