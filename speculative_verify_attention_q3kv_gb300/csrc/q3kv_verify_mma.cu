// Verify attention, tensor-core leg: tcgen05.mma with TMEM accumulators.
//
// Source: "Quasar" (q27 wiki) -- "Self-speculation as the whole design" (all
// drafted tokens checked in one shared-KV MMA verify), the Defaults paragraph
// of "Serving" (MMA verify legs: e4m3 tiles or fp16 tiles "h16", beside the fd2
// reference), and "KV cache" (verify reads the WHT-rotated 3-bit cache; the
// server's default fp8 E4M3 cache is the second format this kernel reads).  The
// pages' legs are mma.sync kernels for consumer GPUs without tcgen05; this is
// a new design for sm_103a.  The e4m3 staging of the pages is not used: it
// adds error on top of the codec's, and the output tolerance here is tight.
//
// Work unit: one CTA = (slot, kv head, chunk of <= 64 query rows, split of the
// context), positions in tiles of 128.
//
// Precision.  The output must stay within 2e-3 of an fp64 reference, which a
// single fp16 operand per side misses by 10-20x on outlier-heavy caches.  So
// every operand is carried as an exact or near-exact fp16 pair:
//   K_hat = (c - 3.5) s = (c - 3.5) s_hi + (c - 3.5) s_lo, with s_hi = s rounded
//           down to 8 significant bits; both products are exact in fp16 and
//           each is one fused multiply-add from the code;
//   V_hat likewise; Q = Q_hi + Q_lo and P = P_hi + P_lo (round-to-nearest
//   splits); each contraction sums the three leading products
//   (hi.hi + hi.lo + lo.hi) with fp32 accumulation in TMEM.  The dropped
//   lo.lo products are below 2^-20 of the scores and of P.V_hat.
// The fp8 format (template FMT = kFmtFp8) decodes K and V exactly into single
// fp16 values (one conversion per pair), so each contraction has two products
// (K.Q_hi + K.Q_lo, V.P_hi + V.P_lo); it is not rotated, so the query kernel
// skips H and the epilogue and merge skip H^-1.
//
// Contractions (M = 128 for both):
//   S^T[p][r] = K_hat[p][:] . Q[r][:]    A = K_hat in TMEM (lane = position),
//                                        B = Q in shared memory (K-major),
//                                        N = query rows padded to 16, K = 256
//   O^T[d][r] += V_hat[:][d] . P[:][r]   A = V_hat^T in shared memory (MN-major),
//                                        B = P^T in shared memory (MN-major),
//                                        two 128-dim halves, K = 16 positions
//
// Issue rate, not the tensor pipe, limits small-N MMAs on this GPU: one thread
// issues a K=16 MMA about every 54 cycles, while an M=128, N=48 MMA executes
// in about 24.  So four warps issue, each into its own accumulator and each
// waiting only for its own operands: QK over dims 0..127 into S, then (after
// those MMAs completed) over dims 128..255 onto S, PV into the two 128-dim halves of
// O^T.  Every MMA sequence is fully unrolled, its descriptors formed by
// constant offsets.
//
// Records: each K thread loads its own position's record straight from the
// pool into registers a tile (fp8: half a record) ahead; the V warps each
// bulk-copy their two 16-record groups of a tile into shared memory
// (cp.async.bulk completing on their own mbarrier) and refill them as soon as
// they have read them.  A tile's 128 positions are contiguous in a page.
//
// Warp roles (20 warps, 96 registers each), handing tiles on with mbarriers:
//   A   warps 0-7   softmax: thread = position (lane quarter warp & 3) for 32
//                   query rows (warp >> 2 picks rows 0-31 or 32-63); reads its
//                   S columns from TMEM; scores are in log2 units and the
//                   running row maximum is only raised when a score exceeds it
//                   by more than 14 (then l and the O^T columns of those rows
//                   are rescaled; each 32-row half decides on its own), so most
//                   tiles need no cross-lane maximum; P = 2^(s - m) <= 2^14 goes
//                   to shared memory as fp16 hi/lo; row sums accumulate per lane
//                   in TMEM and are reduced across lanes once, after the last
//                   tile.  Two warps per lane quarter halve each warp's chain
//                   of dependent work per tile, which is what sets the tile rate
//                   when every scheduler also runs dequantising warps.
//   B1  warps 8-11  thread = position: its K record in registers, K_hat into
//                   TMEM in two halves (dims 0..127, 128..255), each as soon
//                   as the QK half of the previous tile has read it.
//   B2  warps 12-15 V_hat in 16-position sub-tiles through a ring of five
//                   shared-memory buffers; warp q fills sub-tiles q and q + 4
//                   of each tile, lane = (position, 32-dim block).
//   MQa, MQb  warps 16-17   one thread each issues a QK half
//   MP0, MP1  warps 18-19   one thread each issues the PV of an O^T half
// TMEM (512 columns): K_hat hi | K_hat lo | S | row-sum partials | O^T dims 0..127 | 128..255.
//
// After the last tile the A warps read O^T (thread = one output dim, warp >> 2
// picks the 128-dim half, 16 rows per TMEM round trip) and either finish the rows (one split: times 1/l, then
// H back for the rotated format) or store the split partial (m, l, o) for the
// merge kernel.
//
// Every mbarrier wait is bounded (about a second); on a timeout the CTA sets
// Q3KV_STATUS_TIMEOUT, stops issuing, waits (bounded) for the MMAs and copies
// it has in flight, frees its TMEM and returns.  Named barriers are only used
// inside a warp group whose warps all run the same number of iterations, also
// after a timeout.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <atomic>

#include "q3kv_common.cuh"
#include "q3kv_internal.h"

namespace q3kv {
namespace {

constexpr int kWarps = 20;
constexpr int kThreads = kWarps * 32;
constexpr int kTileP = 128;                 // positions per tile (MMA M of S^T)
constexpr int kSubP = 16;                   // positions per V sub-tile (one MMA K step)
constexpr int kSubTiles = kTileP / kSubP;   // 8
constexpr int kVBufs = 5;                   // V_hat sub-tile ring (5/8 of a tile)
// Per cache format: record bytes, whether K_hat / V_hat carry an fp16 lo part
// (the 3-bit codec's values need 14 significant bits; E4M3 values are exact in
// fp16), and whether queries and outputs are rotated by H.
template <int FMT>
struct Fmt {
    static constexpr int kRecB = kRecordBytes;
    static constexpr bool kLo = true;
    static constexpr bool kRot = true;
};
template <>
struct Fmt<kFmtFp8> {
    static constexpr int kRecB = kFp8RecordBytes;
    static constexpr bool kLo = false;
    static constexpr bool kRot = false;
};
constexpr int kRows = 64;                   // max query rows per CTA (MMA N <= 64)
constexpr float kRescaleThreshold = 14.0f;  // log2 units: P <= 2^14, exact to split into fp16 hi/lo
// Initial running maximum: finite, so 2^(s - m) of a masked score (-inf) is 0
// without a select, and any finite score exceeds it by more than the threshold.
constexpr float kMInit = -1.0e30f;
constexpr long long kWaitCycles = 2000000000LL;
// A waiting thread is suspended (not spinning) until the phase completes or
// this many nanoseconds pass, so idle warps leave the issue slots to the others.
constexpr uint32_t kSuspendHintNs = 100000;
constexpr float kMaxScale = 5458.0f;        // 12 * s must stay below the fp16 maximum
constexpr float kMaxT5kScale = 20000.0f;    // turbo5k K: the largest centroid (3.27) times s within fp16

// TMEM columns (allocation of 512)
constexpr uint32_t kColKHi = 0;
constexpr uint32_t kColKLo = 128;
constexpr uint32_t kColS = 256;             // S^T (QK over dims 0..127, then 128..255)
constexpr uint32_t kColL = 320;             // row-sum partials: lane = position slot, column = row
constexpr uint32_t kColO0 = 384;
constexpr uint32_t kColO1 = 448;
constexpr uint32_t kTmemCols = 512;

// named barriers
constexpr int kBarA = 1;                    // the 256 softmax threads
constexpr int kBarHalf = 2;                 // + h: the 128 softmax threads of rows 32h .. 32h + 31

struct Bars {
    unsigned long long vfull[4][2]; // V records of B2 warp q's sub-tile q + 4e landed
    unsigned long long kready[2];   // K_hat dims half in TMEM (4 B1 warps)
    unsigned long long qk_done[2];  // QK half h done (S complete after half 1), that K_hat half read
    unsigned long long s_free;      // S read (8 A warps)
    unsigned long long q_ready;     // Q hi/lo copied in (bulk copy bytes)
    unsigned long long p_ready[2];  // P^T buffer b stored, O^T rescaled (8 A warps)
    unsigned long long v_ready[kVBufs];  // V_hat buffer b filled (one B2 warp)
    unsigned long long v_free[kVBufs];   // V_hat buffer b read (2 commits)
    unsigned long long pv_done[2];  // all PV MMAs of a tile with P^T buffer b done (2 commits)
    unsigned long long drain[4];    // everything an issuer started is done (1 commit)
};

template <int FMT>
struct __align__(16) MmaSmem {
    __half qhi[kRows * kHeadDim];           // B of QK, K-major core layout
    __half qlo[kRows * kHeadDim];
    __half v[kVBufs][Fmt<FMT>::kLo ? 2 : 1][kSubP * kHeadDim];  // [buffer][hi|lo]: A of PV, MN-major
    __half phi[2][kTileP * kRows];          // B of PV, MN-major, double-buffered by tile
    __half plo[2][kTileP * kRows];
    uint8_t vrec[kTileP * Fmt<FMT>::kRecB];  // V record stage: one 16-record copy per sub-tile
    float m_run[kRows];
    float thr[kRows];                       // m_run + threshold
    float l_run[kRows];
    float alpha[kRows];
    float red[4][kRows];
    Bars bar;
    uint32_t tmem_base;
    int abort;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(unsigned long long* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; on a timeout marks the CTA aborted and returns false.  A
// phase that is already complete is seen by a non-blocking test first.
__device__ bool mbar_wait(unsigned long long* bar, uint32_t parity, volatile int* abort) {
    if (mbar_test_wait(bar, parity)) return true;
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

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Bulk copy global -> shared (16-byte aligned ends, size a multiple of 16),
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// One lane of the (converged) warp, chosen by the hardware.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier among `n` threads (id 1.. ; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// OR of `pred` over the `n` threads of named barrier `id` (also a barrier).
__device__ __forceinline__ int named_or(int id, int n, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(n)
        : "memory");
    return r;
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
// V_hat sub-tile (A of PV; M = dims d, K = positions p < 16), MN-major: core (d/8, p/8).
__device__ __forceinline__ int v_off(int d, int p) { return (((d >> 3) * 2 + (p >> 3)) << 6) + ((p & 7) << 3) + (d & 7); }
// P^T (B of PV; N = rows r, K = positions p < 128), MN-major: core (r/8, p/8).
__device__ __forceinline__ int p_off(int r, int p) { return (((r >> 3) * 16 + (p >> 3)) << 6) + ((p & 7) << 3) + (r & 7); }
constexpr uint32_t kQLbo = 128, kQSbo = 32 * 128;
constexpr uint32_t kVLbo = 128, kVSbo = 2 * 128;
constexpr uint32_t kPLbo = 128, kPSbo = 16 * 128;

// ---------------------------------------------------------------- dequantisation
// fp16 pair (8.5 + c_even, 8.5 + c_odd) from two 3-bit fields at bit offsets
// off and off + 16: 0x4800 is 8 with ulp 1/128, so a code goes in at bit 7,
// and 0x0040 adds the half (exact: 8.5 + c has at most 5 significant bits).
__device__ __forceinline__ uint32_t code_pair_word(uint32_t w, int off) {
    const uint32_t x = (off >= 7) ? (w >> (off - 7)) : (w << (7 - off));
    return (x & 0x03800380u) | 0x48404840u;
}
__device__ __forceinline__ uint32_t code_pair_last(uint32_t w0, uint32_t w1, uint32_t w2) {
    // element 30: bit 15 of w0, w1, w2 -> code bits 0,1,2 (into fp16 mantissa bits 7,8,9)
    // element 31: bit 31 of w0, w1, w2
    const uint32_t x = ((w0 >> 8) & 0x00800080u) | ((w1 >> 7) & 0x01000100u) | ((w2 >> 6) & 0x02000200u);
    return x | 0x48404840u;
}

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Four E4M3 bytes (b0 lowest) -> fp16 pairs (b0, b1) and (b2, b3), low half
// first; every E4M3 value is exact in fp16.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& p01, uint32_t& p23) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(p01), "=r"(p23)
        : "r"(w));
}

// One 32-element block: 16 pairs of (c - 3.5) s_hi and (c - 3.5) s_lo, where
// s_hi keeps the top 8 significant bits of s and s_lo = s - s_hi the other 3.
// With x = 8.5 + c, (c - 3.5) s_part = x s_part - 12 s_part: the constant
// 12 s_part (2 + 8 or 2 + 3 bits) and the result (3 + 8 or 3 + 3 bits) are
// exact in fp16, so one fused multiply-add per half gives each product
// exactly, for s <= 65504 / 12 (larger scales are flagged).  With 8 bits in
// s_hi the products the three-product contractions drop, Q_lo . K_hat_lo and
// P_lo . V_hat_lo, are below 2^-20 of the scores and of P . V_hat (a 6-bit
// s_hi left Q_lo . K_hat_lo at 2^-18, which at scores near 100 in log2 units,
// with outlier-heavy queries and keys, alone cost up to 2e-3 of output).
template <int M0 = 0, int NM = 16>
__device__ __forceinline__ void dequant_block(const uint32_t* w3, __half s, uint32_t (&hi)[NM], uint32_t (&lo)[NM]) {
    const __half s_hi = __ushort_as_half((unsigned short)(__half_as_ushort(s) & 0xFFF8u));
    const __half s_lo = __hsub(s, s_hi);
    const __half m12 = __ushort_as_half((unsigned short)0xCA00u);   // -12
    const __half2 sh2 = __halves2half2(s_hi, s_hi);
    const __half2 sl2 = __halves2half2(s_lo, s_lo);
    const __half ch = __hmul(s_hi, m12), cl = __hmul(s_lo, m12);
    const __half2 ch2 = __halves2half2(ch, ch);
    const __half2 cl2 = __halves2half2(cl, cl);
    const uint32_t w0 = w3[0], w1 = w3[1], w2 = w3[2];
#pragma unroll
    for (int mm = 0; mm < NM; ++mm) {
        const int m = M0 + mm;                           // pair m of the block
        uint32_t x;
        if (m < 15) {
            const uint32_t w = (m < 5) ? w0 : (m < 10 ? w1 : w2);
            x = code_pair_word(w, 3 * (m % 5));
        } else {
            x = code_pair_last(w0, w1, w2);
        }
        hi[mm] = as_u32(__hfma2(as_h2(x), sh2, ch2));    // (c - 3.5) s_hi, exact
        lo[mm] = as_u32(__hfma2(as_h2(x), sl2, cl2));    // (c - 3.5) s_lo, exact
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

__device__ __forceinline__ void load8(const float* src, float (&x)[8]) {
    const float4 u = reinterpret_cast<const float4*>(src)[0];
    const float4 w = reinterpret_cast<const float4*>(src)[1];
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* src, float (&x)[8]) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[0];
    const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(ww[i] << 16);
        x[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
}

// All lanes wait; the warp agrees on the outcome (a timeout anywhere fails all).
__device__ __forceinline__ bool warp_wait(unsigned long long* bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Page of the tile starting at pos0, or -1 if the page table entry is out of range.
__device__ __forceinline__ int32_t tile_page(const VerifyArgs& a, const int32_t* pt_row, int pos0) {
    const int32_t page = pt_row[pos0 / kPageSize];
    return (page >= 0 && page < a.num_pages) ? page : -1;
}

// Issues the bulk copy of n records (kv 0 = K, 1 = V) of the tile at pos0,
// starting at row r0 of the tile, or, for a page id out of range, flags it
// and completes the phase without data (the readers zero that tile).
template <int FMT>
__device__ __forceinline__ void issue_rec_copy(const VerifyArgs& a, const int32_t* pt_row, int g, int kv, int pos0,
                                               int r0, int n, uint8_t* dst, unsigned long long* full) {
    const int32_t page = pt_row[pos0 / kPageSize];
    if (page < 0 || page >= a.num_pages) {
        if (a.status) atomicOr(a.status, Q3KV_STATUS_BAD_PAGE);
        mbar_arrive(full);
        return;
    }
    constexpr int RECB = Fmt<FMT>::kRecB;
    const uint8_t* src =
        a.pool + (FMT == kFmtT5k ? t5k_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, kv, pos0 % kPageSize + r0)
                                 : record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, kv,
                                                 pos0 % kPageSize + r0, RECB));
    const uint32_t bytes = (uint32_t)(n * RECB);
    fence_proxy_async();
    mbar_arrive_expect_tx(full, bytes);
    bulk_g2s(dst, src, bytes, full);
}

// Queries of one unit (slot, kv head, 64-row chunk) in the verify kernel's
// shared-memory operand layout, fp16 hi then lo; padding rows are zeros.  CTA
// (unit, group of 8 rows), one row per warp.  ROT (the 3-bit cache): register
// butterflies for H, then scale 1/16 (H) * 1/16 (softmax) * log2(e); without
// ROT (the fp8 cache) only 1/16 (softmax) * log2(e).  Then a round-to-nearest
// hi/lo split.
template <typename TIn, bool ROT>
__global__ void __launch_bounds__(256) qprep_kernel(VerifyArgs a) {
    // wait for the previous grid before reading anything; only then let the
    // verify grid start (it reads the cache and lengths before its own wait,
    // which covers only the queries written here)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int unit = blockIdx.x;
    const int r = 8 * blockIdx.y + warp;                 // row within the unit's 64
    const int chunk = unit % a.row_chunks;
    const int g = (unit / a.row_chunks) % a.num_kv_heads;
    const int slot = unit / (a.row_chunks * a.num_kv_heads);
    const int T = a.n_q[slot];
    const int row0 = chunk * kRows;
    const int Rc = max(0, min(kRows, kGroup * min(T, a.max_n_q) - row0));
    __half* qhi = static_cast<__half*>(a.q_prep) + (size_t)unit * (kQPrepBytes / 2);
    __half* qlo = qhi + kRows * kHeadDim;
    float y[8];
    if (r < Rc) {
        const int ra = row0 + r;
        const int Hq = a.num_kv_heads * kGroup;
        load8(static_cast<const TIn*>(a.q) + (((int64_t)a.q_offsets[slot] + ra / kGroup) * Hq + g * kGroup + ra % kGroup) *
                                                 kHeadDim + 8 * lane,
              y);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = 0.0f;
    }
    if (ROT) {
#pragma unroll
        for (int h = 1; h < 8; h <<= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((i & h) == 0) {
                    const float lo = y[i], hi = y[i + h];
                    y[i] = lo + hi;
                    y[i + h] = lo - hi;
                }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float o = __shfl_xor_sync(0xffffffffu, y[i], m);
                y[i] = fmaf(sgn, y[i], o);                    // lower lane: o + y, upper lane: o - y
            }
        }
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        constexpr float kScale = ROT ? 1.4426950408889634f / 256.0f : 1.4426950408889634f / 16.0f;
        const float x0 = y[2 * i] * kScale;
        const float x1 = y[2 * i + 1] * kScale;
        const __half2 h2 = __floats2half2_rn(x0, x1);
        const float2 hf = __half22float2(h2);
        hw[i] = as_u32(h2);
        lw[i] = as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
    }
    *reinterpret_cast<uint4*>(&qhi[q_off(r, 8 * lane)]) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(&qlo[q_off(r, 8 * lane)]) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

template <typename TIn, int FMT>
__global__ void __launch_bounds__(kThreads, 1) verify_mma_kernel(VerifyArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    MmaSmem<FMT>& sm = *reinterpret_cast<MmaSmem<FMT>*>(smem_raw);
    constexpr int kRecB = Fmt<FMT>::kRecB;
    // the split-merge kernel may be scheduled once every CTA of this grid runs;
    // it waits for this grid's completion before reading the partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // units run fastest in the grid, so every unit's first splits are
    // dispatched before any unit's later ones (most of which exit at once).
    // Within a (slot, kv head) the last row chunk comes first: in a causal
    // prefill a chunk's visible context grows with its index, so the longest
    // CTAs are dispatched first and the short ones fill the last wave.
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
    const int row0 = chunk * kRows;
    const int Rc = min(kRows, R - row0);
    if (Rc <= 0) return;
    const int n_pages = (L + kPageSize - 1) / kPageSize;
    const int split_pages = split_pages_of(a);
    const int n_splits = (n_pages + split_pages - 1) / split_pages;
    if (n_splits > a.num_splits) {
        if (tid == 0 && split == 0 && chunk == 0 && g == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_BAD_LENGTH);
        return;
    }
    if (split >= n_splits) return;
    const int p_begin = split * split_pages * kPageSize;
    const int Nctx = L - T;
    // positions past the causal limit of this CTA's last row are masked for all
    // of its rows, so they are not read (long prefills: later rows see more);
    // at least one position is kept so every CTA of a split writes its partial
    const int p_vis = Nctx + (row0 + Rc - 1) / kGroup + 1;
    const int p_end = min(min(L, p_begin + split_pages * kPageSize), max(p_vis, p_begin + 1));
    const int n_tiles = (p_end - p_begin + kTileP - 1) / kTileP;
    const int Hq = a.num_kv_heads * kGroup;
    const int64_t q_base = a.q_offsets[slot];
    const int N = (Rc + 15) & ~15;      // MMA N: rows padded to 16
    const int32_t* pt_row = a.page_table + (int64_t)slot * a.max_pages_per_slot;
    volatile int* abort = &sm.abort;
    Bars& bar = sm.bar;

    // ---- set-up: barriers, TMEM, row state; then the first tile's record
    // copies (K/V warps, which start dequantising at once) and the queries
    // (softmax and issuer warps, published through q_ready)
    if (tid == 0) {
        for (int q = 0; q < 4; ++q) {
            mbar_init(&bar.vfull[q][0], 1);
            mbar_init(&bar.vfull[q][1], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bar.kready[h], 4);
            mbar_init(&bar.qk_done[h], 1);
            mbar_init(&bar.p_ready[h], 8);
            mbar_init(&bar.pv_done[h], 2);
        }
        mbar_init(&bar.s_free, 8);
        mbar_init(&bar.q_ready, 1);
        for (int b = 0; b < kVBufs; ++b) {
            mbar_init(&bar.v_ready[b], 1);
            mbar_init(&bar.v_free[b], 2);
        }
        for (int k = 0; k < 4; ++k) mbar_init(&bar.drain[k], 1);
        sm.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 16) tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid < kRows) {
        // padding rows (>= Rc) get a running maximum of 0 and a threshold no
        // score exceeds: they never trigger a rescale and are never stored
        sm.m_run[tid] = (tid < Rc) ? kMInit : 0.0f;
        sm.thr[tid] = (tid < Rc) ? kMInit + kRescaleThreshold : CUDART_INF_F;
        sm.l_run[tid] = 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp >= 12 && warp < 16 && lane == 0 && n_tiles > 0) {
        // each V-dequantising warp copies its own positions of the first tile
        const int q = warp & 3;
        for (int e = 0; e < 2; ++e) {
            const int r0 = kSubP * (q + 4 * e);
            issue_rec_copy<FMT>(a, pt_row, g, 1, p_begin, r0, kSubP, sm.vrec + kRecB * r0, &bar.vfull[q][e]);
        }
    }
    if (warp == 16 && lane == 0) {
        // the rotated queries of this unit, written by the query kernel that
        // precedes this grid: wait for it, then one bulk copy of hi and lo
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int unit = (slot * a.num_kv_heads + g) * a.row_chunks + chunk;
        const uint8_t* src = static_cast<const uint8_t*>(a.q_prep) + (size_t)unit * kQPrepBytes;
        mbar_arrive_expect_tx(&bar.q_ready, (uint32_t)kQPrepBytes);
        bulk_g2s(sm.qhi, src, (uint32_t)kQPrepBytes, &bar.q_ready);
    }
    const uint32_t tmem = sm.tmem_base;
    bool range_bad = false;
    float* outs = reinterpret_cast<float*>(sm.qhi);      // [64][256] floats once Q is no longer read

    if (warp < 8) {
        // ================================================================ A: softmax
        const int q = warp & 3;                         // lane quarter: positions 32q .. 32q + 31
        const int rh = warp >> 2;                       // rows 32rh .. 32rh + 31 (S^T columns)
        const int r0 = 32 * rh;
        const int p = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int bar_half = kBarHalf + rh;
        bool ok = true;
        for (int i = 0; i < n_tiles; ++i) {
            const int pb = i & 1;                       // P^T buffer of this tile
            // the second QK half is issued only after the first one completed,
            // so its commit covers the whole S
            ok = ok && mbar_wait(&bar.qk_done[1], (uint32_t)(i & 1), abort);
            tc_fence_after();
            // this warp's 32 S columns, in one TMEM round trip; columns >= N are -inf
            float x[32];
#pragma unroll
            for (int c = 0; c < 2; ++c)
                if (r0 + 16 * c < N) tmem_ld16(tmem + lane_base + kColS + r0 + 16 * c, &x[16 * c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.s_free);
#pragma unroll
            for (int c = 0; c < 2; ++c)
                if (r0 + 16 * c >= N)
#pragma unroll
                    for (int k = 0; k < 16; ++k) x[16 * c + k] = -CUDART_INF_F;

            const int pos0 = p_begin + i * kTileP;
            const int pos = pos0 + p;
            const bool tile_ok = tile_page(a, pt_row, pos0) >= 0;
            const bool interior = tile_ok && pos0 + kTileP - 1 <= min(Nctx, p_end - 1);
            if (!interior) {
                // causal / length mask.  Row r (token (row0 + r) / 8) sees
                // positions <= Nctx + (row0 + r) / 8, so position pos is seen by
                // rows r >= 8 (pos - Nctx) - row0; nothing past p_end is seen.
                const int r_min = (tile_ok && pos < p_end) ? max(0, kGroup * (pos - Nctx) - row0) : kRows;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (r0 + j < r_min) x[j] = -CUDART_INF_F;
            }
            int over = 0;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 t4 = reinterpret_cast<const float4*>(sm.thr + r0)[c];
                over |= (x[4 * c] > t4.x) | (x[4 * c + 1] > t4.y) | (x[4 * c + 2] > t4.z) | (x[4 * c + 3] > t4.w);
            }
            const int slow = named_or(bar_half, 128, over);
            if (slow) {
                // raise the running maxima of these 32 rows to cover this tile;
                // rescale their l and O^T columns below
                {
                    float t[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) t[k] = x[k];
                    sm.red[q][r0 + lane] = transpose_reduce<true>(t);
                }
                named_sync(bar_half, 128);
                if (q == 0 && r0 + lane < Rc) {
                    const int r = r0 + lane;
                    const float mt = fmaxf(fmaxf(sm.red[0][r], sm.red[1][r]), fmaxf(sm.red[2][r], sm.red[3][r]));
                    const float m_old = sm.m_run[r];
                    const float m_new = fmaxf(m_old, mt);
                    const float al = exp2f(m_old - m_new);
                    sm.m_run[r] = m_new;
                    sm.thr[r] = m_new + kRescaleThreshold;
                    sm.alpha[r] = al;
                }
                named_sync(bar_half, 128);
            }
            // P = 2^(s - m) in place (a masked score gives 0)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 m4 = reinterpret_cast<const float4*>(sm.m_run + r0)[c];
                x[4 * c] = fast_exp2(x[4 * c] - m4.x);
                x[4 * c + 1] = fast_exp2(x[4 * c + 1] - m4.y);
                x[4 * c + 2] = fast_exp2(x[4 * c + 2] - m4.z);
                x[4 * c + 3] = fast_exp2(x[4 * c + 3] - m4.w);
            }
            // P^T buffer pb was last read by the PV of tile i - 2; a rescale of
            // O^T needs every earlier PV finished (tile i - 1)
            if (slow && i > 0) {
                ok = ok && mbar_wait(&bar.pv_done[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1), abort);
                tc_fence_after();
                const int c_end = min(r0 + 32, N);
#pragma unroll 1
                for (int h = 0; h < 3; ++h) {           // O^T halves and the row-sum partials
                    const uint32_t col = h == 0 ? kColO0 : (h == 1 ? kColO1 : kColL);
#pragma unroll 1
                    for (int c = r0; c < c_end; c += 8) {
                        float v8[8];
                        tmem_ld8(tmem + lane_base + col + c, v8);
                        tmem_ld_wait();
                        uint32_t u8[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) u8[k] = __float_as_uint(v8[k] * sm.alpha[c + k]);
                        tmem_st8(tmem + lane_base + col + c, u8);
                    }
                }
                tmem_st_wait();
            } else if (i > 1) {
                ok = ok && mbar_wait(&bar.pv_done[pb], (uint32_t)(((i - 2) >> 1) & 1), abort);
            }
            __half* phi = sm.phi[pb];
            __half* plo = sm.plo[pb];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (r0 + 8 * c < N) {
                    uint32_t h4[4], l4[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a0 = x[8 * c + 2 * k], a1 = x[8 * c + 2 * k + 1];
                        const __half2 hh2 = __floats2half2_rn(a0, a1);
                        const float2 hf = __half22float2(hh2);
                        h4[k] = as_u32(hh2);
                        l4[k] = as_u32(__floats2half2_rn(a0 - hf.x, a1 - hf.y));
                    }
                    *reinterpret_cast<uint4*>(&phi[p_off(r0 + 8 * c, p)]) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                    *reinterpret_cast<uint4*>(&plo[p_off(r0 + 8 * c, p)]) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.p_ready[pb]);
            // row sums: this thread's P values added to its lane's TMEM partials
            // (the cross-lane sum is taken once, after the last tile)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (r0 + 16 * c < N) {
                    uint32_t u16[16];
                    if (i > 0) {
                        float y[16];
                        tmem_ld16(tmem + lane_base + kColL + r0 + 16 * c, y);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k) u16[k] = __float_as_uint(y[k] + x[16 * c + k]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) u16[k] = __float_as_uint(x[16 * c + k]);
                    }
                    tmem_st16(tmem + lane_base + kColL + r0 + 16 * c, u16);
                }
            }
            tmem_st_wait();
        }
        // l = column sums of the row-sum partials over the 128 lanes
        {
            float y[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (r0 + 16 * c < N && n_tiles > 0) tmem_ld16(tmem + lane_base + kColL + r0 + 16 * c, &y[16 * c]);
                else
#pragma unroll
                    for (int k = 0; k < 16; ++k) y[16 * c + k] = 0.0f;
            }
            tmem_ld_wait();
            sm.red[q][r0 + lane] = transpose_reduce<false>(y);
            named_sync(kBarA, 256);
            if (tid < N) {
                const float l = (sm.red[0][tid] + sm.red[1][tid]) + (sm.red[2][tid] + sm.red[3][tid]);
                sm.l_run[tid] = l;
                sm.alpha[tid] = (n_splits == 1) ? 1.0f / l : 1.0f;   // the epilogue's row multiplier
            }
        }
        named_sync(kBarA, 256);   // l_run complete
        // ---- epilogue: O^T -> partial or finished rows
        if (n_tiles > 0) ok = ok && mbar_wait(&bar.pv_done[(n_tiles - 1) & 1], (uint32_t)(((n_tiles - 1) >> 1) & 1), abort);
        tc_fence_after();
        if (ok) {
            const int unit = (slot * a.num_kv_heads + g) * a.row_chunks + chunk;
            float* po = a.part_o + ((int64_t)unit * a.num_splits + split) * kRows * kHeadDim;
            // 16 rows of this thread's dim per TMEM round trip: a short loop,
            // since this code runs once per CTA and is fetched cold
            float* dst = (n_splits == 1) ? outs : po;
            const int d = 128 * rh + 32 * q + lane;
            const uint32_t col = rh ? kColO1 : kColO0;
#pragma unroll 1
            for (int c = 0; c < Rc; c += 16) {
                float v[16];
                tmem_ld16(tmem + lane_base + col + c, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (c + k < Rc) dst[(c + k) * kHeadDim + d] = v[k] * sm.alpha[c + k];
            }
            if (n_splits > 1 && tid < Rc) {
                float* pml = a.part_ml + ((int64_t)unit * a.num_splits + split) * kRows * 2;
                pml[2 * tid] = sm.m_run[tid];
                pml[2 * tid + 1] = sm.l_run[tid];
            }
        }
    } else if (warp < 12) {
        // ================================================================ B1: K_hat -> TMEM
        const int q = warp - 8;
        const int p = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        if constexpr (FMT == kFmtFp8) {
            // thread p's 256-byte E4M3 record, half (128 dims) at a time, the
            // next half's 8 x 16-byte loads in flight while this one converts
            auto fetch_half = [&](int i, int hh, uint32_t (&w)[32]) {
                const int pos0 = p_begin + i * kTileP;
                const int32_t page = (i < n_tiles) ? tile_page(a, pt_row, pos0) : -1;
                if (page >= 0 && pos0 + p < p_end) {
                    const uint4* r4 = reinterpret_cast<const uint4*>(
                        a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 0,
                                               pos0 % kPageSize + p, kRecB)) + 8 * hh;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const uint4 u = __ldg(r4 + m);
                        w[4 * m] = u.x; w[4 * m + 1] = u.y; w[4 * m + 2] = u.z; w[4 * m + 3] = u.w;
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 32; ++m) w[m] = 0u;
                }
            };
            uint32_t wn[32];
            fetch_half(0, 0, wn);
            bool ok = true;
            for (int i = 0; i < n_tiles; ++i) {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t w[32];
#pragma unroll
                    for (int m = 0; m < 32; ++m) w[m] = wn[m];
                    fetch_half(hh ? i + 1 : i, hh ^ 1, wn);
                    if (i > 0) ok = ok && warp_wait(&bar.qk_done[hh], (uint32_t)((i - 1) & 1), abort);
                    tc_fence_after();
                    const uint32_t col = tmem + lane_base + kColKHi + 64 * hh;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t h8[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) e4m3x4_to_f16(w[4 * c + k], h8[2 * k], h8[2 * k + 1]);
                        tmem_st8(col + 8 * c, h8);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.kready[hh]);
                }
            }
        } else if constexpr (FMT == kFmtT5k) {
            // turbo5k K: thread p's 164-byte record, a 128-dim half at a time (64
            // nibble bytes, 16 bytes of 5th bits, the two scales), the next half's
            // loads in flight while this one decodes.  A code's centroid comes from
            // a shuffle (lane l holds centroid l); K_hat = centroid * s in float32,
            // split into round-to-nearest fp16 hi/lo (within 2^-22 of K_hat).
            const float cent = a.t5k.c[lane];
            auto fetch_half = [&](int i, int hh, uint32_t (&w)[21]) {
                const int pos0 = p_begin + i * kTileP;
                const int32_t page = (i < n_tiles) ? tile_page(a, pt_row, pos0) : -1;
                if (page >= 0 && pos0 + p < p_end) {
                    const uint32_t* r = reinterpret_cast<const uint32_t*>(
                        a.pool + t5k_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 0, pos0 % kPageSize + p));
#pragma unroll
                    for (int m = 0; m < 16; ++m) w[m] = __ldg(r + 16 * hh + m);
#pragma unroll
                    for (int m = 0; m < 4; ++m) w[16 + m] = __ldg(r + 32 + 4 * hh + m);
                    w[20] = __ldg(r + 40);
                } else {
#pragma unroll
                    for (int m = 0; m < 21; ++m) w[m] = 0u;
                }
            };
            uint32_t wn[21];
            fetch_half(0, 0, wn);
            bool ok = true;
            for (int i = 0; i < n_tiles; ++i) {
                const bool valid = ok && p_begin + i * kTileP + p < p_end;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t w[21];
#pragma unroll
                    for (int m = 0; m < 21; ++m) w[m] = wn[m];
                    fetch_half(hh ? i + 1 : i, hh ^ 1, wn);
                    if (i > 0) ok = ok && warp_wait(&bar.qk_done[hh], (uint32_t)((i - 1) & 1), abort);
                    tc_fence_after();
                    const float s = __half2float(__ushort_as_half((unsigned short)(hh ? (w[20] >> 16) : (w[20] & 0xFFFFu))));
                    range_bad |= valid && !(s <= kMaxT5kScale);
                    const uint32_t col = tmem + lane_base + 64 * hh;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {               // 8 pairs (16 dims) at a time
                        const int bb = e >> 1;
                        uint32_t hi[8], lo[8];
                        const uint32_t top = w[16 + bb];
#pragma unroll
                        for (int mm = 0; mm < 8; ++mm) {
                            const int m = 8 * (e & 1) + mm;
                            const uint32_t nw = w[4 * bb + m / 4];
                            const int sh = 8 * (m % 4);
                            const uint32_t c0 = ((nw >> sh) & 0xFu) | (((top >> (2 * m)) & 1u) << 4);
                            const uint32_t c1 = ((nw >> (sh + 4)) & 0xFu) | (((top >> (2 * m + 1)) & 1u) << 4);
                            const float v0 = __shfl_sync(0xffffffffu, cent, (int)c0) * s;
                            const float v1 = __shfl_sync(0xffffffffu, cent, (int)c1) * s;
                            const __half2 h2 = __floats2half2_rn(v0, v1);
                            const float2 hf = __half22float2(h2);
                            hi[mm] = as_u32(h2);
                            lo[mm] = as_u32(__floats2half2_rn(v0 - hf.x, v1 - hf.y));
                        }
                        tmem_st8(col + kColKHi + 8 * e, hi);
                        tmem_st8(col + kColKLo + 8 * e, lo);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.kready[hh]);
                }
            }
        } else {
            // thread p's 112-byte record straight from the pool into registers,
            // a tile ahead (7 x 16-byte read-only loads)
            auto fetch = [&](int i, uint32_t (&w)[24], uint32_t (&sc)[4]) {
                const int pos0 = p_begin + i * kTileP;
                const int32_t page = (i < n_tiles) ? tile_page(a, pt_row, pos0) : -1;
                if (page >= 0 && pos0 + p < p_end) {
                    const uint4* r4 = reinterpret_cast<const uint4*>(
                        a.pool + record_offset(a.num_layers, a.num_kv_heads, page, a.layer, g, 0, pos0 % kPageSize + p));
#pragma unroll
                    for (int m = 0; m < 6; ++m) {
                        const uint4 u = __ldg(r4 + m);
                        w[4 * m] = u.x; w[4 * m + 1] = u.y; w[4 * m + 2] = u.z; w[4 * m + 3] = u.w;
                    }
                    const uint4 u = __ldg(r4 + 6);
                    sc[0] = u.x; sc[1] = u.y; sc[2] = u.z; sc[3] = u.w;
                } else {
#pragma unroll
                    for (int m = 0; m < 24; ++m) w[m] = 0u;
                    sc[0] = sc[1] = sc[2] = sc[3] = 0u;
                }
            };
            uint32_t wn[24], sn[4];
            fetch(0, wn, sn);
            bool ok = true;
            for (int i = 0; i < n_tiles; ++i) {
                uint32_t w[24], sc[4];
#pragma unroll
                for (int m = 0; m < 24; ++m) w[m] = wn[m];
#pragma unroll
                for (int m = 0; m < 4; ++m) sc[m] = sn[m];
                fetch(i + 1, wn, sn);                    // the next tile's record is in flight meanwhile
                const bool valid = ok && p_begin + i * kTileP + p < p_end;
                // two halves of the dims, each after its QK half of the previous tile
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t wh[12], sh[2];
#pragma unroll
                    for (int m = 0; m < 12; ++m) wh[m] = hh ? w[12 + m] : w[m];
                    sh[0] = hh ? sc[2] : sc[0];
                    sh[1] = hh ? sc[3] : sc[1];
                    if (i > 0) ok = ok && warp_wait(&bar.qk_done[hh], (uint32_t)((i - 1) & 1), abort);
                    tc_fence_after();
                    const uint32_t col = tmem + lane_base + 64 * hh;
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        // eight pairs at a time keep the dequantised values in
                        // 16 registers beside the two records
                        const __half s = __ushort_as_half((unsigned short)((bb & 1) ? (sh[bb >> 1] >> 16) : (sh[bb >> 1] & 0xFFFFu)));
                        range_bad |= valid && !(__half2float(s) <= kMaxScale);
                        {
                            uint32_t hi[8], lo[8];
                            dequant_block<0, 8>(&wh[3 * bb], s, hi, lo);
                            tmem_st8(col + kColKHi + 16 * bb, hi);
                            tmem_st8(col + kColKLo + 16 * bb, lo);
                        }
                        {
                            uint32_t hi[8], lo[8];
                            dequant_block<8, 8>(&wh[3 * bb], s, hi, lo);
                            tmem_st8(col + kColKHi + 16 * bb + 8, hi);
                            tmem_st8(col + kColKLo + 16 * bb + 8, lo);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.kready[hh]);
                }
            }
        }
    } else if (warp < 16) {
        // ================================================================ B2: V_hat sub-tiles -> shared memory
        // Warp q fills sub-tiles q and q + 4 of every tile (sub-tile u = 8 i + s
        // goes to ring buffer u % 5) from its own two 16-record copies.  Lane = (position pl, 32-dim block
        // blk); item j covers pl = 8 (j >> 1) + (lane & 7), blk = 4 (j & 1) + (lane >> 3).
        const int q = warp - 12;
        const bool producer = (lane == 0);
        int pend[2] = {n_tiles > 0 ? 0 : -1, n_tiles > 0 ? 0 : -1};
        bool ok = true;
        for (int i = 0; i < n_tiles; ++i) {
            const int pos0 = p_begin + i * kTileP;
            const bool page_ok = tile_page(a, pt_row, pos0) >= 0;
#pragma unroll 1
            for (int e = 0; e < 2; ++e) {
                const int r0 = kSubP * (q + 4 * e);          // first position of the sub-tile
                ok = ok && warp_wait(&bar.vfull[q][e], (uint32_t)(i & 1), abort);
                if (producer && ok) pend[e] = -1;
                const int u = kSubTiles * i + q + 4 * e;     // sub-tile index: ring buffer u % 5, its use u / 5
                const int b = u % kVBufs;
                const int k = u / kVBufs;
                if (k >= 1) ok = ok && warp_wait(&bar.v_free[b], (uint32_t)((k - 1) & 1), abort);
                __half* vh = sm.v[b][0];
                const uint8_t* rb = sm.vrec + kRecB * r0;
#pragma unroll 1
                for (int j = 0; j < 4 && FMT == kFmtFp8; ++j) {
                    // 32 dims of one position: 32 E4M3 bytes -> 16 fp16 pairs (exact)
                    const int pl = 8 * (j >> 1) + (lane & 7);
                    const int blk = 4 * (j & 1) + (lane >> 3);
                    uint4 u0 = make_uint4(0u, 0u, 0u, 0u), u1 = u0;
                    if (ok && page_ok && pos0 + r0 + pl < p_end) {
                        const uint4* r = reinterpret_cast<const uint4*>(rb + kRecB * pl + 32 * blk);
                        u0 = r[0];
                        u1 = r[1];
                    }
                    const uint32_t w8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                    uint32_t h16[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) e4m3x4_to_f16(w8[k], h16[2 * k], h16[2 * k + 1]);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(&vh[v_off(32 * blk + 8 * c, pl)]) =
                            make_uint4(h16[4 * c], h16[4 * c + 1], h16[4 * c + 2], h16[4 * c + 3]);
                }
#pragma unroll 1
                for (int j = 0; j < 4 && FMT != kFmtFp8; ++j) {
                    __half* vl = sm.v[b][Fmt<FMT>::kLo ? 1 : 0];

                    const int pl = 8 * (j >> 1) + (lane & 7);
                    const int blk = 4 * (j & 1) + (lane >> 3);
                    uint32_t w3[3];
                    __half s = __ushort_as_half((unsigned short)0);
                    if (ok && page_ok && pos0 + r0 + pl < p_end) {
                        const uint8_t* r = rb + kRecB * pl;
                        const uint32_t* wp = reinterpret_cast<const uint32_t*>(r + 12 * blk);
                        w3[0] = wp[0]; w3[1] = wp[1]; w3[2] = wp[2];
                        s = *reinterpret_cast<const __half*>(r + 96 + 2 * blk);
                        range_bad |= !(__half2float(s) <= kMaxScale);
                    } else {
                        w3[0] = w3[1] = w3[2] = 0u;
                    }
                    uint32_t hi[16], lo[16];
                    dequant_block(w3, s, hi, lo);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int d0 = 32 * blk + 8 * c;
                        *reinterpret_cast<uint4*>(&vh[v_off(d0, pl)]) =
                            make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
                        *reinterpret_cast<uint4*>(&vl[v_off(d0, pl)]) =
                            make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
                    }
                }
                fence_proxy_async();
                __syncwarp();   // this warp's records of the sub-tile are read and its V_hat stored
                if (producer) {
                    mbar_arrive(&bar.v_ready[b]);
                    if (ok && i + 1 < n_tiles && !*abort) {
                        issue_rec_copy<FMT>(a, pt_row, g, 1, pos0 + kTileP, r0, kSubP, sm.vrec + kRecB * r0,
                                              &bar.vfull[q][e]);
                        pend[e] = i + 1;
                    }
                }
            }
        }
        if (producer)
            for (int e = 0; e < 2; ++e)
                if (pend[e] >= 0) mbar_drain(&bar.vfull[q][e], (uint32_t)(pend[e] & 1));
    } else if (warp < 18) {
        // ================================================================ MQa / MQb: QK halves
        const int h = warp - 16;                     // 0: dims 0..127, 1: dims 128..255 (both into S)
        const uint32_t idesc_qk = make_idesc(N, false, false);
        const uint64_t bq_hi = make_desc(smem_u32(sm.qhi) + h * 8 * 256, kQLbo, kQSbo);
        const uint64_t bq_lo = make_desc(smem_u32(sm.qlo) + h * 8 * 256, kQLbo, kQSbo);
        const uint32_t dS = tmem + kColS;
        const uint32_t aK_hi = tmem + kColKHi + 64 * h;
        const uint32_t aK_lo = tmem + kColKLo + 64 * h;
        bool qok = warp_wait(&bar.q_ready, 0u, abort);
        for (int i = 0; qok && i < n_tiles; ++i) {
            if (!warp_wait(&bar.kready[h], (uint32_t)(i & 1), abort)) break;
            // half 0 overwrites S once the softmax has read the previous tile's;
            // half 1 accumulates onto it after half 0's MMAs have completed
            if (h == 0 && i >= 1 && !warp_wait(&bar.s_free, (uint32_t)((i - 1) & 1), abort)) break;
            if (h == 1 && !warp_wait(&bar.qk_done[0], (uint32_t)(i & 1), abort)) break;
            tc_fence_after();
            // descriptors are formed by the whole (converged) warp, so they stay
            // warp-uniform; one elected lane issues
#pragma unroll
            for (int j = 0; j < 8; ++j) {   // descriptor start address is in 16-byte units
                const uint64_t ko = (uint64_t)(16 * j);
                if (elect_one()) {
                    mma_ts(dS, aK_hi + 8 * j, bq_hi + ko, idesc_qk, (h == 0 && j == 0) ? 0u : 1u);
                    mma_ts(dS, aK_hi + 8 * j, bq_lo + ko, idesc_qk, 1u);
                    if (Fmt<FMT>::kLo) mma_ts(dS, aK_lo + 8 * j, bq_hi + ko, idesc_qk, 1u);
                }
                __syncwarp();
            }
            if (elect_one()) mma_commit(&bar.qk_done[h]);
            __syncwarp();
        }
        if (lane == 0) mma_commit(&bar.drain[h]);
        __syncwarp();
        mbar_drain(&bar.drain[h], 0);
        if (h == 0 && !qok && lane == 0) mbar_drain(&bar.q_ready, 0);   // the Q copy, after a timeout
    } else {
        // ================================================================ MP0 / MP1: PV halves
        const int h = warp - 18;                     // O^T dims 128h .. 128h + 127
        const uint32_t idesc_pv = make_idesc(N, true, true);
        const uint32_t dO = tmem + (h ? kColO1 : kColO0);
        const uint64_t bp_hi0 = make_desc(smem_u32(sm.phi[0]), kPLbo, kPSbo);
        const uint64_t bp_lo0 = make_desc(smem_u32(sm.plo[0]), kPLbo, kPSbo);
        const uint64_t pbuf = (uint64_t)(sizeof(sm.phi[0]) >> 4);    // one P^T buffer, 16-byte units
        const uint64_t av_hi0 = make_desc(smem_u32(sm.v[0][0]) + (uint32_t)(16 * h) * kVSbo, kVLbo, kVSbo);
        const uint64_t av_lo0 =
            make_desc(smem_u32(sm.v[0][Fmt<FMT>::kLo ? 1 : 0]) + (uint32_t)(16 * h) * kVSbo, kVLbo, kVSbo);
        const uint64_t vbuf = (uint64_t)(sizeof(sm.v[0]) >> 4);      // one V buffer, 16-byte units
        for (int jt = 0; jt < n_tiles; ++jt) {
            const int pb = jt & 1;
            if (!warp_wait(&bar.p_ready[pb], (uint32_t)((jt >> 1) & 1), abort)) break;
            bool ok = true;
#pragma unroll 1
            for (int sub = 0; sub < kSubTiles; ++sub) {
                // sub-tile u = 8 jt + sub sits in buffer u % 5, that buffer's use u / 5
                const int u = kSubTiles * jt + sub;
                const int b = u % kVBufs;
                ok = warp_wait(&bar.v_ready[b], (uint32_t)((u / kVBufs) & 1), abort);
                if (!ok) break;
                tc_fence_after();
                // descriptors formed by the whole warp (warp-uniform); one elected lane issues
                const uint64_t bfo = (uint64_t)b * vbuf;
                const uint64_t koff = (uint64_t)pb * pbuf + (uint64_t)(16 * sub);   // 2 sub x 128 bytes along K
                const uint32_t acc0 = (jt > 0 || sub > 0) ? 1u : 0u;
                const uint64_t avh = av_hi0 + bfo, avl = av_lo0 + bfo, bph = bp_hi0 + koff, bpl = bp_lo0 + koff;
                if (elect_one()) {
                    mma_ss(dO, avh, bph, idesc_pv, acc0);
                    if (Fmt<FMT>::kLo) mma_ss(dO, avl, bph, idesc_pv, 1u);
                    mma_ss(dO, avh, bpl, idesc_pv, 1u);
                    mma_commit(&bar.v_free[b]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) mma_commit(&bar.pv_done[pb]);
            __syncwarp();
        }
        if (lane == 0) mma_commit(&bar.drain[2 + h]);
        __syncwarp();
        mbar_drain(&bar.drain[2 + h], 0);
    }

    if (range_bad && a.status) atomicOr(a.status, Q3KV_STATUS_RANGE);
    tc_fence_before();
    __syncthreads();
    if (warp == 16) tmem_dealloc(tmem, kTmemCols);
    if (*abort) {
        if (tid == 0 && a.status) atomicOr(a.status, Q3KV_STATUS_TIMEOUT);
        return;
    }
    if (n_splits == 1) {
        // whole rows: H back (rotated format) and 1/16, one warp per row, from
        // registers straight to the output
        constexpr float kOutScale = Fmt<FMT>::kRot ? 0.0625f : 1.0f;   // unnormalised H: 1/16
        for (int r = warp; r < Rc; r += kWarps) {
            const float4* src = reinterpret_cast<const float4*>(outs + r * kHeadDim + 8 * lane);
            const float4 u0 = src[0], u1 = src[1];
            float y[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            if (Fmt<FMT>::kRot) rotate_row_regs(y);
            const int ra = row0 + r;
            float4* o4 = reinterpret_cast<float4*>(a.out + ((q_base + ra / kGroup) * Hq + g * kGroup + ra % kGroup) * kHeadDim +
                                                   8 * lane);
            o4[0] = make_float4(y[0] * kOutScale, y[1] * kOutScale, y[2] * kOutScale, y[3] * kOutScale);
            o4[1] = make_float4(y[4] * kOutScale, y[5] * kOutScale, y[6] * kOutScale, y[7] * kOutScale);
        }
    }
}

template <typename TIn, int FMT>
cudaError_t launch_typed(const VerifyArgs& a, cudaStream_t stream, std::atomic<bool>& attr_set) {
    const size_t smem = sizeof(MmaSmem<FMT>);
    if (!attr_set.load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(verify_mma_kernel<TIn, FMT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set.store(true, std::memory_order_release);
    }
    const unsigned units = (unsigned)(a.num_slots * a.num_kv_heads * a.row_chunks);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(units, kRows / 8);
        qc.blockDim = dim3(256);
        qc.stream = stream;
        qc.attrs = attr;
        qc.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&qc, qprep_kernel<TIn, Fmt<FMT>::kRot>, a);
        if (e != cudaSuccess) return e;
    }
    // the verify grid may start while the query kernel runs: only its QK
    // issuer waits (griddepcontrol.wait) for the queries
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units, (unsigned)a.num_splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_mma_kernel<TIn, FMT>, a);
}

}  // namespace

cudaError_t launch_verify_mma(const VerifyArgs& a, cudaStream_t stream) {
    // the shared-memory opt-in is a per-device function attribute: one flag per
    // (device, instantiation)
    constexpr int kMaxDevices = 64;
    static std::atomic<bool> flags[kMaxDevices][6];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::atomic<bool>* attr_set = flags[dev];
    const bool f32 = a.dtype == Q3KV_F32;
    if (a.fmt == kFmtFp8)
        return f32 ? launch_typed<float, kFmtFp8>(a, stream, attr_set[2])
                   : launch_typed<__nv_bfloat16, kFmtFp8>(a, stream, attr_set[3]);
    if (a.fmt == kFmtT5k)
        return f32 ? launch_typed<float, kFmtT5k>(a, stream, attr_set[4])
                   : launch_typed<__nv_bfloat16, kFmtT5k>(a, stream, attr_set[5]);
    return f32 ? launch_typed<float, kFmtQ3>(a, stream, attr_set[0])
               : launch_typed<__nv_bfloat16, kFmtQ3>(a, stream, attr_set[1]);
}

size_t verify_mma_smem_bytes() { return sizeof(MmaSmem<kFmtQ3>); }

}  // namespace q3kv
