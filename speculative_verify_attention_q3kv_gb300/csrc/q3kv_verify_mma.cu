// Verify attention, tensor-core leg: tcgen05.mma with TMEM accumulators.
//
// Source: "Quasar" (q27 wiki) -- "Self-speculation as the whole design" (all
// drafted tokens checked in one shared-KV MMA verify), the Defaults paragraph
// of "Serving" (MMA verify legs: e4m3 tiles or fp16 tiles "h16", beside the fd2
// reference), and "KV cache" (verify reads the WHT-rotated 3-bit cache).  The
// pages' legs are mma.sync kernels for consumer GPUs without tcgen05; this is
// a new design for sm_103a.  The e4m3 staging of the pages is not used: it
// adds error on top of the codec's, and the output tolerance here is tight.
//
// Work unit: one CTA = (slot, kv head, chunk of <= 64 query rows, split of the
// context), 256 threads, positions in tiles of 128.
//
// Precision.  The output must stay within 2e-3 of an fp64 reference, which a
// single fp16 operand per side misses by 10-20x on outlier-heavy caches.  So
// every operand is carried as an exact or near-exact fp16 pair:
//   K_hat = (c - 3.5) s = (c - 3.5) s_hi + (c - 3.5) s_lo, with s_hi = s rounded
//           down to 8 significant bits; both products are exact in fp16;
//   V_hat likewise; Q = Q_hi + Q_lo and P = P_hi + P_lo (round-to-nearest
//   splits); and each contraction sums the three leading products
//   (hi.hi + hi.lo + lo.hi) in fp32 tensor-core accumulation.
//
// Data flow of one tile (128 positions):
//   1. thread 0 streams the tile's packed K and V records (2 x 14,336 B, one
//      contiguous run each inside a page) into a 2-stage shared-memory ring
//      with cp.async.bulk + mbarrier, two tiles ahead;
//   2. all warps dequantise K_hat (hi, lo) straight into TMEM (lane =
//      position), the A operand of S^T = K_hat Q^T (M = 128 positions,
//      N = rows padded to 16, K = 256), B = Q (hi, lo) resident in shared
//      memory, K-major;
//   3. while the MMAs run, the warps dequantise V_hat for positions 0..63 into
//      shared memory (MN-major A operand of O^T = V_hat^T P^T);
//   4. softmax on S^T (thread = position): scores are in log2 units; the
//      running row maximum is only raised when a score exceeds it by more
//      than 8 (then the O^T accumulator columns are rescaled in TMEM), so the
//      common tile needs no cross-lane maximum; P = 2^(s - m) <= 256 is split
//      into fp16 hi/lo and stored MN-major as the B operand; row sums use a
//      transposing butterfly (lane j ends with row j);
//   5. O^T (two 128-lane halves of the 256 dims, fp32 in TMEM) += V_hat^T P^T
//      for positions 0..63, then 64..127 after their V_hat is in place.
// After the last tile each thread reads one output dim of O^T from TMEM.  The
// split partials (m, l, o) are merged by the last CTA of the unit to finish,
// which also rotates the result back by H.
//
// Every mbarrier wait is bounded (about a second); on a timeout the CTA sets
// Q3KV_STATUS_TIMEOUT, stops issuing work, waits (bounded) for what it has in
// flight, frees its TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "q3kv_common.cuh"
#include "q3kv_internal.h"

namespace q3kv {
namespace {

constexpr int kThreads = 256;
constexpr int kTileP = 128;                 // positions per tile (MMA M of S^T)
constexpr int kSubP = 64;                   // positions per V sub-tile
constexpr int kRows = 64;                   // max query rows per CTA (MMA N <= 64)
constexpr int kStageBytes = kTileP * kRecordBytes;   // 14,336 B of K (or V) records
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P <= 256
constexpr long long kWaitCycles = 2000000000LL;
constexpr float kMaxScale = 18688.0f;       // 3.5 * s must stay below the fp16 maximum

// TMEM columns (allocation of 512)
constexpr uint32_t kColKHi = 0;
constexpr uint32_t kColKLo = 128;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColO0 = 320;
constexpr uint32_t kColO1 = 384;
constexpr uint32_t kTmemCols = 512;

struct __align__(1024) MmaSmem {
    __half qhi[kRows * kHeadDim];           // B of QK, K-major core layout
    __half qlo[kRows * kHeadDim];
    __half vhi[kSubP * kHeadDim];           // A of PV, MN-major core layout
    __half vlo[kSubP * kHeadDim];
    __half phi[kTileP * kRows];             // B of PV, MN-major core layout
    __half plo[kTileP * kRows];
    uint8_t stage[2][2][kStageBytes];       // [stage][K|V][records]
    float m_run[kRows];
    float l_run[kRows];
    float alpha[kRows];
    float red[8][32];
    unsigned long long full_bar[2];
    unsigned long long mma_bar;
    uint32_t tmem_base;
    int tile_ok[2];
    int issued[2];                          // tiles streamed into each stage so far
    int flag;
    int abort;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; on a timeout marks the CTA aborted and returns false.
__device__ bool mbar_wait(unsigned long long* bar, uint32_t parity, volatile int* abort) {
    if (*abort) return false;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

// Bounded wait used while draining after an abort.
__device__ void mbar_drain(unsigned long long* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - t0 <= kWaitCycles) {
    }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory matrix descriptor, no swizzle ("interleaved" core matrices of
// 8 rows x 16 bytes, 128 contiguous bytes each).  lbo = byte stride between
// core matrices along K, sbo = along M/N.
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, M = 128.
__host__ __device__ constexpr uint32_t make_idesc(int n, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// ---------------------------------------------------------------- layouts (element offsets)
// Q (B of QK; N = rows r, K = dims k), K-major: core (r/8, k/8) at ((r/8)*32 + k/8)*64 elements.
__device__ __forceinline__ int q_off(int r, int k) { return (((r >> 3) * 32 + (k >> 3)) << 6) + ((r & 7) << 3) + (k & 7); }
// V_hat sub-tile (A of PV; M = dims d, K = positions p < 64), MN-major: core (d/8, p/8).
__device__ __forceinline__ int v_off(int d, int p) { return (((d >> 3) * 8 + (p >> 3)) << 6) + ((p & 7) << 3) + (d & 7); }
// P^T (B of PV; N = rows r, K = positions p < 128), MN-major: core (r/8, p/8).
__device__ __forceinline__ int p_off(int r, int p) { return (((r >> 3) * 16 + (p >> 3)) << 6) + ((p & 7) << 3) + (r & 7); }
constexpr uint32_t kQLbo = 128, kQSbo = 32 * 128;
constexpr uint32_t kVLbo = 128, kVSbo = 8 * 128;
constexpr uint32_t kPLbo = 128, kPSbo = 16 * 128;

// ---------------------------------------------------------------- dequantisation
// fp16 pair (c_even, c_odd) + 512 from two 3-bit fields at bit offsets off and
// off+16: 0x6000 is 512 with ulp 0.5, so the code goes in at bit 1.
__device__ __forceinline__ uint32_t code_pair_word(uint32_t w, int off) {
    const uint32_t x = (off >= 1) ? (w >> (off - 1)) : (w << 1);
    return (x & 0x000E000Eu) | 0x60006000u;
}
__device__ __forceinline__ uint32_t code_pair_last(uint32_t w0, uint32_t w1, uint32_t w2) {
    // element 30: bit 15 of w0, w1, w2 -> code bits 0,1,2 (into fp16 mantissa bits 1,2,3)
    // element 31: bit 31 of w0, w1, w2
    const uint32_t x = ((w0 >> 14) & 0x00020002u) | ((w1 >> 13) & 0x00040004u) | ((w2 >> 12) & 0x00080008u);
    return x | 0x60006000u;
}

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// One 32-element block: 16 pairs of (c - 3.5) s_hi and (c - 3.5) s_lo.
__device__ __forceinline__ void dequant_block(const uint32_t* w3, __half s, uint32_t (&hi)[16], uint32_t (&lo)[16]) {
    const __half s_hi = __ushort_as_half((unsigned short)(__half_as_ushort(s) & 0xFFF8u));
    const __half s_lo = __hsub(s, s_hi);
    const __half2 sh2 = __halves2half2(s_hi, s_hi);
    const __half2 sl2 = __halves2half2(s_lo, s_lo);
    const __half2 off = __float2half2_rn(515.5f);        // 512 + 3.5
    const uint32_t w0 = w3[0], w1 = w3[1], w2 = w3[2];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        uint32_t x;
        if (m < 15) {
            const uint32_t w = (m < 5) ? w0 : (m < 10 ? w1 : w2);
            x = code_pair_word(w, 3 * (m % 5));
        } else {
            x = code_pair_last(w0, w1, w2);
        }
        const __half2 c = __hsub2(as_h2(x), off);         // (c_even - 3.5, c_odd - 3.5), exact
        hi[m] = as_u32(__hmul2(c, sh2));                   // exact: 3 x 8 significant bits
        lo[m] = as_u32(__hmul2(c, sl2));                   // exact: 3 x 3 significant bits
    }
}

// ---------------------------------------------------------------- butterfly reductions
// v[0..31] per lane; afterwards lane l holds op over all lanes of v[l].
template <bool MAX>
__device__ __forceinline__ float transpose_reduce(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            const float got = __shfl_xor_sync(0xffffffffu, send, half);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1) verify_mma_kernel(VerifyArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    MmaSmem& sm = *reinterpret_cast<MmaSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    const int slot = blockIdx.z;
    const int g = blockIdx.y / a.row_chunks;
    const int chunk = blockIdx.y % a.row_chunks;
    const int split = blockIdx.x;

    const int T = a.n_q[slot];
    const int L = a.ctx_len[slot];
    if (T <= 0) return;
    if (T > a.max_n_q || T > L || L > a.max_pages_per_slot * kPageSize) {
        if (tid == 0 && split == 0 && chunk == 0 && g == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    const int R = kGroup * T;
    const int row0 = chunk * kRows;
    const int Rc = min(kRows, R - row0);
    if (Rc <= 0) return;
    const int n_pages = (L + kPageSize - 1) / kPageSize;
    const int n_splits = (n_pages + a.split_pages - 1) / a.split_pages;
    if (n_splits > a.num_splits) {
        if (tid == 0 && split == 0 && chunk == 0 && g == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    if (split >= n_splits) return;
    const int p_begin = split * a.split_pages * kPageSize;
    const int p_end = min(L, p_begin + a.split_pages * kPageSize);
    const int n_tiles = (p_end - p_begin + kTileP - 1) / kTileP;
    const int Nctx = L - T;
    const int Hq = a.num_kv_heads * kGroup;
    const int64_t q_base = a.q_offsets[slot];
    const int N = (Rc + 15) & ~15;      // MMA N: rows padded to 16
    const int Nh = N >> 1;              // columns per softmax warp half
    const uint32_t idesc_qk = make_idesc(N, false, false);
    const uint32_t idesc_pv = make_idesc(N, true, true);
    const int32_t* pt_row = a.page_table + (int64_t)slot * a.max_pages_per_slot;
    volatile int* abort = &sm.abort;

    // ---- set-up: barriers, TMEM, queries
    if (tid == 0) {
        mbar_init(&sm.full_bar[0], 1);
        mbar_init(&sm.full_bar[1], 1);
        mbar_init(&sm.mma_bar, 1);
        sm.abort = 0;
        sm.issued[0] = sm.issued[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid < kRows) {
        sm.m_run[tid] = -CUDART_INF_F;
        sm.l_run[tid] = 0.0f;
    }
    // raw queries -> fp32 scratch (the V_hat area), rows r = t*8 + hh of this chunk
    float* qf = reinterpret_cast<float*>(sm.vhi);
    const TIn* qin = static_cast<const TIn*>(a.q);
    for (int idx = tid; idx < kRows * kHeadDim; idx += kThreads) {
        const int r = idx / kHeadDim, d = idx % kHeadDim;
        float x = 0.0f;
        if (r < Rc) {
            const int ra = row0 + r;
            x = load_in(qin + ((q_base + ra / kGroup) * Hq + g * kGroup + ra % kGroup) * kHeadDim + d);
        }
        qf[idx] = x;
    }
    __syncthreads();
    rotate_rows(qf, Rc);
    // scale: 1/16 (H normalisation) * 1/16 (softmax) * log2(e); split into fp16 hi + lo
    for (int idx = tid; idx < kRows * kHeadDim; idx += kThreads) {
        const int r = idx / kHeadDim, d = idx % kHeadDim;
        const float x = qf[idx] * (1.4426950408889634f / 256.0f);
        const __half h = __float2half_rn(x);
        const __half l = __float2half_rn(x - __half2float(h));
        sm.qhi[q_off(r, d)] = h;
        sm.qlo[q_off(r, d)] = l;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    // ---- prologue: stream the first two tiles
    auto issue_tile = [&](int it, int stg) {
        const int pos0 = p_begin + it * kTileP;
        const int32_t page = pt_row[pos0 / kPageSize];
        if (page < 0 || page >= a.num_pages) {
            sm.tile_ok[stg] = 0;
            mbar_arrive(&sm.full_bar[stg]);
            if (a.status) atomicOr(a.status, Q3KV_STATUS_BAD_PAGE);
            return;
        }
        sm.tile_ok[stg] = 1;
        sm.issued[stg] += 1;
        const uint8_t* src_k = a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 0, pos0 % kPageSize);
        const uint8_t* src_v = a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 1, pos0 % kPageSize);
        mbar_arrive_expect_tx(&sm.full_bar[stg], 2 * kStageBytes);
        bulk_g2s(sm.stage[stg][0], src_k, kStageBytes, &sm.full_bar[stg]);
        bulk_g2s(sm.stage[stg][1], src_v, kStageBytes, &sm.full_bar[stg]);
    };
    if (tid == 0) {
        issue_tile(0, 0);
        if (n_tiles > 1) issue_tile(1, 1);
    }

    uint32_t mma_phase = 0;
    int waited[2] = {0, 0};                 // tiles of each stage consumed
    bool have_o = false;
    bool range_bad = false;
    const int quarter = warp & 3;     // TMEM lane quarter of this warp
    const int whalf = warp >> 2;      // 0: K dims 0..127 / S columns [0,Nh) / O dims 0..127
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;

    for (int it = 0; it < n_tiles; ++it) {
        const int stg = it & 1;
        const int pos0 = p_begin + it * kTileP;
        mbar_wait(&sm.full_bar[stg], (uint32_t)((it >> 1) & 1), abort);
        const bool tile_ok = sm.tile_ok[stg] != 0;

        // (2) K_hat -> TMEM: position 32*quarter + lane, blocks 4*whalf .. 4*whalf+3
        {
            const int p = quarter * 32 + lane;
            const bool valid = tile_ok && (pos0 + p) < p_end;
            const uint8_t* rec = sm.stage[stg][0] + p * kRecordBytes;
            const __half* sc = reinterpret_cast<const __half*>(rec + 96);
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const int b = whalf * 4 + bb;
                uint32_t hi[16], lo[16];
                if (valid) {
                    dequant_block(reinterpret_cast<const uint32_t*>(rec) + 3 * b, sc[b], hi, lo);
                    range_bad |= !(__half2float(sc[b]) <= kMaxScale);
                } else {
#pragma unroll
                    for (int m = 0; m < 16; ++m) hi[m] = lo[m] = 0u;
                }
                tmem_st16(tmem + lane_base + kColKHi + 16 * b, hi);
                tmem_st16(tmem + lane_base + kColKLo + 16 * b, lo);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();

        // (2b) QK MMAs: S^T[p][r] = sum_k K[p][k] Q[r][k]
        if (tid == 0 && !*abort) {
            tc_fence_after();
            const uint32_t qh = smem_u32(sm.qhi), ql = smem_u32(sm.qlo);
#pragma unroll 1
            for (int j = 0; j < 16; ++j) {
                const uint64_t bh = make_desc(qh + j * 256, kQLbo, kQSbo);
                const uint64_t bl = make_desc(ql + j * 256, kQLbo, kQSbo);
                mma_ts(tmem + kColS, tmem + kColKHi + 8 * j, bh, idesc_qk, j > 0 ? 1u : 0u);
                mma_ts(tmem + kColS, tmem + kColKHi + 8 * j, bl, idesc_qk, 1u);
                mma_ts(tmem + kColS, tmem + kColKLo + 8 * j, bh, idesc_qk, 1u);
            }
            mma_commit(&sm.mma_bar);
        }

        // (3) V_hat positions 0..63 -> shared memory while the MMAs run
        auto dequant_v = [&](int sub) {
            const int pl = tid & 63;                 // position within the sub-tile
            const int p = sub * kSubP + pl;          // position within the tile
            const bool valid = tile_ok && (pos0 + p) < p_end;
            const uint8_t* rec = sm.stage[stg][1] + p * kRecordBytes;
            const __half* sc = reinterpret_cast<const __half*>(rec + 96);
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = (tid >> 6) * 2 + bb;
                uint32_t hi[16], lo[16];
                if (valid) {
                    dequant_block(reinterpret_cast<const uint32_t*>(rec) + 3 * b, sc[b], hi, lo);
                    range_bad |= !(__half2float(sc[b]) <= kMaxScale);
                } else {
#pragma unroll
                    for (int m = 0; m < 16; ++m) hi[m] = lo[m] = 0u;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {          // 8 dims per 16-byte chunk
                    const int d0 = 32 * b + 8 * c;
                    *reinterpret_cast<uint4*>(&sm.vhi[v_off(d0, pl)]) =
                        make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
                    *reinterpret_cast<uint4*>(&sm.vlo[v_off(d0, pl)]) =
                        make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
                }
            }
            fence_proxy_async();
        };
        dequant_v(0);

        if (mbar_wait(&sm.mma_bar, mma_phase, abort)) mma_phase ^= 1;
        tc_fence_after();

        // (4) softmax: thread = position 32*quarter + lane; rows [whalf*Nh, whalf*Nh + Nh)
        {
            const int p = quarter * 32 + lane;
            const int pos = pos0 + p;
            const bool valid = tile_ok && pos < p_end;
            float x[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (8 * c < Nh) {
                    float v8[8];
                    tmem_ld8(tmem + lane_base + kColS + whalf * Nh + 8 * c, v8);
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[8 * c + i] = v8[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[8 * c + i] = -CUDART_INF_F;
                }
            }
            tmem_ld_wait();
            int over = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = whalf * Nh + j;
                const bool vis = valid && j < Nh && r < Rc && pos <= Nctx + (row0 + r) / kGroup;
                x[j] = vis ? x[j] : -CUDART_INF_F;
                if (vis && x[j] > sm.m_run[r] + kRescaleThreshold) over = 1;
            }
            if (__syncthreads_or(over)) {
                // raise the running maxima to the tile maxima, rescale l and O
                float t[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) t[j] = x[j];
                const float mx = transpose_reduce<true>(t);
                sm.red[warp][lane] = mx;
                __syncthreads();
                if (tid < N) {
                    const int hh = tid / Nh, j = tid % Nh;
                    float mt = -CUDART_INF_F;
#pragma unroll
                    for (int q = 0; q < 4; ++q) mt = fmaxf(mt, sm.red[hh * 4 + q][j]);
                    const float m_old = sm.m_run[tid];
                    const float m_new = fmaxf(m_old, mt);
                    const float al = (m_old == -CUDART_INF_F) ? 0.0f : exp2f(m_old - m_new);
                    sm.m_run[tid] = m_new;
                    sm.l_run[tid] *= al;
                    sm.alpha[tid] = al;
                }
                __syncthreads();
                if (have_o) {
                    const uint32_t col = whalf ? kColO1 : kColO0;
                    for (int c = 0; c < N; c += 8) {
                        float v8[8];
                        tmem_ld8(tmem + lane_base + col + c, v8);
                        tmem_ld_wait();
                        uint32_t u8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) u8[i] = __float_as_uint(v8[i] * sm.alpha[c + i]);
                        tmem_st8(tmem + lane_base + col + c, u8);
                    }
                    tmem_st_wait();
                }
            }
            // P = 2^(s - m), split hi/lo, store P^T; row sums
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = whalf * Nh + j;
                const float m = (j < Nh) ? sm.m_run[min(r, kRows - 1)] : 0.0f;
                x[j] = (x[j] == -CUDART_INF_F) ? 0.0f : fast_exp2(x[j] - m);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (8 * c < Nh) {
                    uint32_t h4[4], l4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float a0 = x[8 * c + 2 * i], a1 = x[8 * c + 2 * i + 1];
                        const __half2 hh2 = __floats2half2_rn(a0, a1);
                        const float2 hf = __half22float2(hh2);
                        const __half2 ll2 = __floats2half2_rn(a0 - hf.x, a1 - hf.y);
                        h4[i] = as_u32(hh2);
                        l4[i] = as_u32(ll2);
                    }
                    const int r0 = whalf * Nh + 8 * c;
                    *reinterpret_cast<uint4*>(&sm.phi[p_off(r0, p)]) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                    *reinterpret_cast<uint4*>(&sm.plo[p_off(r0, p)]) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                }
            }
            fence_proxy_async();
            const float ls = transpose_reduce<false>(x);
            sm.red[warp][lane] = ls;
        }
        tc_fence_before();
        __syncthreads();
        if (tid < N) {
            const int hh = tid / Nh, j = tid % Nh;
            float s = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) s += sm.red[hh * 4 + q][j];
            sm.l_run[tid] += s;
        }

        // (5) PV, positions 0..63
        auto issue_pv = [&](int sub) {
            tc_fence_after();
            const uint32_t vh = smem_u32(sm.vhi), vl = smem_u32(sm.vlo);
            const uint32_t ph = smem_u32(sm.phi), pl = smem_u32(sm.plo);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const uint32_t dcol = tmem + (h ? kColO1 : kColO0);
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    const uint32_t aoff = (uint32_t)(16 * h) * kVSbo + (uint32_t)(2 * j) * kVLbo;
                    const uint32_t boff = (uint32_t)(8 * sub + 2 * j) * kPLbo;
                    const uint64_t avh = make_desc(vh + aoff, kVLbo, kVSbo);
                    const uint64_t avl = make_desc(vl + aoff, kVLbo, kVSbo);
                    const uint64_t bph = make_desc(ph + boff, kPLbo, kPSbo);
                    const uint64_t bpl = make_desc(pl + boff, kPLbo, kPSbo);
                    const uint32_t acc0 = (have_o || sub > 0 || j > 0) ? 1u : 0u;
                    mma_ss(dcol, avh, bph, idesc_pv, acc0);
                    mma_ss(dcol, avl, bph, idesc_pv, 1u);
                    mma_ss(dcol, avh, bpl, idesc_pv, 1u);
                }
            }
            mma_commit(&sm.mma_bar);
        };
        if (tid == 0 && !*abort) issue_pv(0);
        if (mbar_wait(&sm.mma_bar, mma_phase, abort)) mma_phase ^= 1;

        // V_hat positions 64..127 (the V buffer is free again), then PV for them
        dequant_v(1);
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && !*abort) {
            issue_pv(1);
            if (it + 2 < n_tiles) issue_tile(it + 2, stg);   // this stage is fully consumed
        }
        have_o = true;
        if (mbar_wait(&sm.mma_bar, mma_phase, abort)) mma_phase ^= 1;
        tc_fence_after();
        waited[stg] += 1;
    }

    // ---- epilogue: O^T from TMEM; thread = output dim d, N rows
    const int d = whalf * 128 + quarter * 32 + lane;
    float o[kRows];
    {
        const uint32_t col = whalf ? kColO1 : kColO0;
#pragma unroll
        for (int c = 0; c < kRows; c += 8) {
            if (c < N) {
                float v8[8];
                tmem_ld8(tmem + lane_base + col + c, v8);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[c + i] = v8[i];
            }
        }
        tmem_ld_wait();
    }
    if (range_bad && a.status) atomicOr(a.status, Q3KV_STATUS_RANGE);
    __syncthreads();
    if (*abort) {
        // let every copy and MMA this CTA started finish (bounded) before the
        // shared memory and TMEM are given back
        if (tid == 0) {
            mbar_drain(&sm.mma_bar, mma_phase);
            for (int st = 0; st < 2; ++st)
                for (int k = waited[st]; k < sm.issued[st]; ++k) mbar_drain(&sm.full_bar[st], (uint32_t)(k & 1));
        }
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    if (*abort) {
        if (tid == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_TIMEOUT);
        return;
    }

    const int unit = (slot * a.num_kv_heads + g) * a.row_chunks + chunk;
    float* outs = reinterpret_cast<float*>(sm.qhi);      // [64][256] floats (Q no longer needed)
    if (n_splits == 1) {
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (r < Rc) outs[r * kHeadDim + d] = o[r] / sm.l_run[r];
    } else {
        float* po = a.part_o + ((int64_t)unit * a.num_splits + split) * kRows * kHeadDim;
        float* pml = a.part_ml + ((int64_t)unit * a.num_splits + split) * kRows * 2;
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (r < Rc) po[r * kHeadDim + d] = o[r];
        if (tid < Rc) {
            pml[2 * tid] = sm.m_run[tid];
            pml[2 * tid + 1] = sm.l_run[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) sm.flag = (atomicAdd(a.tickets + unit, 1) == n_splits - 1);
        __syncthreads();
        if (!sm.flag) return;
        __threadfence();
        merge_splits<true>(a.part_o + (int64_t)unit * a.num_splits * kRows * kHeadDim,
                           a.part_ml + (int64_t)unit * a.num_splits * kRows * 2, n_splits, Rc, kRows,
                           reinterpret_cast<float*>(sm.vhi), sm.m_run, sm.l_run, outs);
        if (tid == 0) a.tickets[unit] = 0;
    }
    __syncthreads();
    rotate_rows(outs, Rc);
    for (int idx = tid; idx < Rc * kHeadDim; idx += kThreads) {
        const int r = idx / kHeadDim, dd = idx % kHeadDim;
        const int ra = row0 + r;
        a.out[((q_base + ra / kGroup) * Hq + g * kGroup + ra % kGroup) * kHeadDim + dd] = outs[idx] * 0.0625f;
    }
}

}  // namespace

size_t verify_mma_smem_bytes() { return sizeof(MmaSmem); }

cudaError_t launch_verify_mma(const VerifyArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(MmaSmem);
    dim3 grid((unsigned)a.num_splits, (unsigned)(a.num_kv_heads * a.row_chunks), (unsigned)a.num_slots);
    static bool attr_set[2] = {false, false};
    cudaError_t e = cudaSuccess;
    if (a.dtype == Q3KV_F32) {
        if (!attr_set[0]) {
            e = cudaFuncSetAttribute(verify_mma_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            attr_set[0] = true;
        }
        verify_mma_kernel<float><<<grid, kThreads, smem, stream>>>(a);
    } else {
        if (!attr_set[1]) {
            e = cudaFuncSetAttribute(verify_mma_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
            if (e != cudaSuccess) return e;
            attr_set[1] = true;
        }
        verify_mma_kernel<__nv_bfloat16><<<grid, kThreads, smem, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace q3kv
