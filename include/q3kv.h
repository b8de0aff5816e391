/*
 * q3kv -- speculative-verify attention over a 3-bit, Walsh-Hadamard-rotated,
 * paged KV cache.  C ABI of the shared library libq3kv.so (sm_103a).
 *
 * Source of the method: the "Quasar" (q27) engine wiki --
 *   - "turbo3 3-bit KV cache" bullet and the "KV cache" stack bullet: K and V
 *     are WHT-rotated and stored as 3-bit codes in fixed-size blocks,
 *     symmetric for K and V, per slot;
 *   - "Self-speculation as the whole design": all drafted tokens of a step are
 *     checked in one shared-KV verify pass;
 *   - "Width-12 verify": up to 12 tokens per step (this library takes up to 16);
 *   - "Continuous batching": several slots go through one fused round.
 * The pages give no bit-level codec and no kernel for this GPU.  The codec
 * here is this library's own (head_dim 256; y = H x in float32 with H the
 * orthonormal Sylvester-Hadamard matrix; 8 blocks of 32; per block an fp16
 * scale s = absmax/3.5 and codes q = clamp(rint(y/s + 3.5), 0, 7); value
 * (q - 3.5) s; 112 bytes per vector).  Queries are rotated by the same H; the
 * output is rotated back, so callers see ordinary attention outputs.
 *
 * Conventions for every call:
 *   - Return value: Q3KV_OK (0) or a negative Q3KV_ERR_* code.  Nothing is
 *     launched when an argument check fails.
 *   - Device-side problems (a page id outside [0, num_pages), a length beyond
 *     the slot's page table, a non-finite input, an fp16 scale overflow) never
 *     trap: the kernel ORs a Q3KV_STATUS_* bit into *d_status and skips the
 *     offending unit.  d_status may be NULL to ignore them.
 *   - All device work is asynchronous on the given stream.  Pointers prefixed
 *     d_ are device pointers; h_ are host pointers.  The library allocates no
 *     device memory: the caller owns the pool, page tables, lengths, inputs,
 *     outputs, workspace and status word.
 *   - Lengths are owned by the caller.  Rolling back rejected drafts is a
 *     smaller length on the next call; stale records are overwritten by the
 *     next append.
 */
#ifndef Q3KV_H
#define Q3KV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define Q3KV_API __attribute__((visibility("default")))
#else
#define Q3KV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define Q3KV_FORMAT_VERSION 1   /* bumps when the record or page layout changes */

/* error codes (return values) */
#define Q3KV_OK                      0
#define Q3KV_ERR_INVALID_ARG        -1
#define Q3KV_ERR_UNSUPPORTED        -2
#define Q3KV_ERR_OUT_OF_PAGES       -3
#define Q3KV_ERR_WORKSPACE_TOO_SMALL -4
#define Q3KV_ERR_CUDA               -5
#define Q3KV_ERR_SLOT_RANGE         -6
#define Q3KV_ERR_HOST_MEMORY        -7   /* host allocation of the page allocator failed */

/* device status bits (*d_status) */
#define Q3KV_STATUS_NONFINITE_INPUT  1
#define Q3KV_STATUS_SCALE_OVERFLOW   2
#define Q3KV_STATUS_BAD_PAGE         4
#define Q3KV_STATUS_BAD_LENGTH       8
#define Q3KV_STATUS_TIMEOUT         16   /* a bounded wait inside a kernel gave up */
#define Q3KV_STATUS_RANGE           32   /* tensor-core leg: a block scale above 5458
                                            (its exact fp16 dequantisation needs
                                            12 s in fp16 range) */

/* input dtypes */
#define Q3KV_F32   0
#define Q3KV_BF16  1

/* verify implementations */
#define Q3KV_IMPL_AUTO  0   /* the fastest one that supports the shape          */
#define Q3KV_IMPL_FMA   1   /* CUDA-core fp32 FMA flash-decode (reference leg)   */
#define Q3KV_IMPL_MMA   2   /* tcgen05 tensor-core leg (fp16 hi/lo operand pairs,
                               fp32 accumulation); needs block scales <= 5458   */

/* Shape of one cache pool.  Supported: head_dim 256, page_size 256,
 * num_q_heads = 8 * num_kv_heads (GQA group of 8), num_kv_heads >= 1. */
typedef struct q3kv_cache_desc {
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t head_dim;    /* 256 */
    int32_t page_size;   /* 256 */
    int32_t num_pages;
} q3kv_cache_desc;

/* Library and layout versions. */
Q3KV_API int q3kv_version(void);
Q3KV_API int q3kv_format_version(void);

/* Text of an error code (static string, never NULL). */
Q3KV_API const char* q3kv_strerror(int err);

/* Text of the last CUDA failure behind a Q3KV_ERR_CUDA return on the calling
 * host thread (static string, never NULL). */
Q3KV_API const char* q3kv_last_cuda_error(void);

/* Bytes of a pool for desc:
 *   num_pages * num_layers * num_kv_heads * 2 * page_size * 112.
 * Pool layout: the 112-byte record of (page, layer, kv_head, kv in {0:K, 1:V},
 * row = position % 256) starts at
 *   ((((page*num_layers + layer)*num_kv_heads + kv_head)*2 + kv)*256 + row)*112.
 * Record: 24 little-endian uint32 code words (three per 32-element block; in
 * block b, element e < 30 is pair m = e/2, half = e%2, in word 3b + m/5 at bit
 * 16*half + 3*(m%5); element 30 keeps code bit k in bit 15 of word 3b+k and
 * element 31 in bit 31), then 8 fp16 scales.  The pool must be 16-byte aligned. */
Q3KV_API int q3kv_pool_bytes(const q3kv_cache_desc* desc, size_t* bytes);

/* ---- host page allocator (no device work) --------------------------------
 * Source: per-slot KV of the "turbo3 3-bit KV cache" bullet, and the
 * PagedAttention paragraph of the prefix-reuse section (a pool of fixed-size
 * blocks).  Pages are 256 positions.  The allocator owns only host state. */
typedef struct q3kv_allocator q3kv_allocator;

/* Create an allocator over page ids [0, num_pages) for num_slots slots whose
 * page-table rows hold max_pages_per_slot entries.  *out receives the handle.
 * Q3KV_ERR_HOST_MEMORY if its host arrays cannot be allocated (no C++
 * exception leaves any call of this library). */
Q3KV_API int q3kv_allocator_create(int32_t num_pages, int32_t num_slots, int32_t max_pages_per_slot,
                          q3kv_allocator** out);
Q3KV_API void q3kv_allocator_destroy(q3kv_allocator* a);

/* Make slot hold pages for n_positions positions (ceil(n/256) pages), taking
 * new pages from the free list.  Writes the slot's page ids into the caller's
 * host row h_page_table_row[0 .. *n_pages_out) (length max_pages_per_slot;
 * entries past the count are set to -1).  Never shrinks.  All or nothing: on
 * Q3KV_ERR_OUT_OF_PAGES or Q3KV_ERR_HOST_MEMORY nothing changes. */
Q3KV_API int q3kv_alloc_pages(q3kv_allocator* a, int32_t slot, int64_t n_positions,
                     int32_t* h_page_table_row, int32_t* n_pages_out);

/* Return all pages of slot to the free list. */
Q3KV_API int q3kv_free_slot(q3kv_allocator* a, int32_t slot);

/* Free pages left. */
Q3KV_API int q3kv_free_pages(const q3kv_allocator* a, int32_t* n_free);

/* ---- quantise-append --------------------------------------------------------
 * Source: the "turbo3 3-bit KV cache" bullet of the "Quasar" (q27) wiki (each
 * step's K and V are WHT-rotated and stored as 3-bit blocks in the slot's
 * cache) and the PagedAttention paragraph of its prefix-reuse section (the
 * attention KV is an append-only log addressed by position).
 * Encodes new raw K and V head vectors and writes their records.  Slot b
 * appends d_n_new[b] tokens at positions [d_slot_len[b], d_slot_len[b] +
 * d_n_new[b]); token t of slot b is input row d_row_offsets[b] + t.
 *   k, v           device, [rows, num_kv_heads, 256], dtype f32 or bf16,
 *                  unrotated; rows = d_row_offsets[num_slots]
 *   d_page_table   device int32 [num_slots, max_pages_per_slot]
 *   d_slot_len     device int32 [num_slots], positions before the append
 *   d_n_new        device int32 [num_slots], 0 allowed
 *   d_row_offsets  device int32 [num_slots + 1]
 *   max_n_new      host bound on d_n_new[b] (sizes the launch; larger device
 *                  values set Q3KV_STATUS_BAD_LENGTH and are skipped)
 * A record whose page id is out of range is skipped with Q3KV_STATUS_BAD_PAGE. */
Q3KV_API int q3kv_append(void* stream, const q3kv_cache_desc* desc, void* d_pool,
                const int32_t* d_page_table, int32_t max_pages_per_slot,
                const int32_t* d_slot_len, const int32_t* d_n_new, const int32_t* d_row_offsets,
                int32_t num_slots, int32_t max_n_new, int32_t layer,
                const void* k, const void* v, int32_t dtype, int32_t* d_status);

/* ---- verify attention ------------------------------------------------------
 * Source: "Self-speculation as the whole design" (the step's drafts are
 * checked in one pass over the shared KV, causal among themselves), "Width-12
 * verify" (a few to a dozen query tokens per slot) and "Continuous batching"
 * (ragged slots in one launch) of the "Quasar" (q27) wiki.
 * For slot b with L_b = d_ctx_len[b] positions already in the cache (the new
 * tokens appended) and T_b = d_n_q[b] query tokens, query token t in [0, T_b)
 * of q head h attends to positions [0, L_b - T_b + t] of kv head h / 8:
 *   out = H softmax((H q) . k_hat / 16) v_hat        (float32 output)
 *   q      device [rows, num_q_heads, 256], f32 or bf16, unrotated;
 *          token t of slot b is row d_q_offsets[b] + t
 *   out    device float32, same indexing as q
 *   max_ctx_len, max_n_q   host bounds of d_ctx_len and d_n_q (size the
 *          launch); max_n_q <= 16
 *   impl   Q3KV_IMPL_*;  split_positions: positions per split-K unit
 *          (multiple of 256; 0 = chosen from the shape and the GPU)
 *   workspace, workspace_bytes: device scratch of at least
 *          q3kv_workspace_bytes(...) bytes for the same arguments (split
 *          partials and, for the tensor-core leg, the rotated queries; no
 *          initial contents needed).  Calls that share one
 *          workspace must not overlap on the GPU.
 * Slots with T_b == 0 produce nothing.  T_b > L_b or L_b beyond the slot's
 * page table sets Q3KV_STATUS_BAD_LENGTH and the slot's rows are left as they
 * were. */
Q3KV_API int q3kv_workspace_bytes(const q3kv_cache_desc* desc, int32_t num_slots, int64_t max_ctx_len,
                         int32_t max_n_q, int32_t impl, int32_t split_positions, size_t* bytes);

Q3KV_API int q3kv_verify_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                     const int32_t* d_page_table, int32_t max_pages_per_slot,
                     const int32_t* d_ctx_len, const int32_t* d_n_q, const int32_t* d_q_offsets,
                     int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q, int32_t layer,
                     const void* q, int32_t dtype, float* out,
                     int32_t impl, int32_t split_positions,
                     void* d_workspace, size_t workspace_bytes, int32_t* d_status);

/* ---- verify attention with fixed scratch (no workspace argument) -----------
 * The pages have no counterpart to this call; it exists for callers that
 * cannot provide a device workspace (another allocator owns all device memory,
 * a serving loop that must not allocate once running, a binding that only
 * receives device pointers).  Same arguments and results as q3kv_verify_attn,
 * minus the workspace: the split-K scratch comes from one array of
 * Q3KV_NOALLOC_SCRATCH_BYTES in the library's own device memory, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing.
 *   - A call that needs more scratch than the limit (q3kv_workspace_bytes for
 *     the same arguments) returns Q3KV_ERR_WORKSPACE_TOO_SMALL and launches
 *     nothing.
 *   - The first call on a device looks up the array's device address for that
 *     device (cudaGetSymbolAddress, with that device current) and caches it;
 *     make that first call before any stream capture.  The cached address is
 *     kept for the life of the process: do not use this call on a device
 *     after cudaDeviceReset, which may reload the library's device memory at
 *     another address.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and may return wrong results.  The
 *     array keeps the last call's contents; the call needs no initial
 *     contents. */
#define Q3KV_NOALLOC_SCRATCH_BYTES (16u << 20)
Q3KV_API int q3kv_verify_attn_noalloc(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                     const int32_t* d_page_table, int32_t max_pages_per_slot,
                     const int32_t* d_ctx_len, const int32_t* d_n_q, const int32_t* d_q_offsets,
                     int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q, int32_t layer,
                     const void* q, int32_t dtype, float* out,
                     int32_t impl, int32_t split_positions, int32_t* d_status);

/* ---- prefill attention over the 3-bit cache --------------------------------------
 * Source: the "turbo3 3-bit KV cache" bullet of the "Quasar" (q27) wiki (the
 * cache serves decode, verify and batched prefill) and the prefill follow-ons
 * bullet (a prefill-attention kernel).  A prefill is the verify step with many
 * new tokens: append them with q3kv_append, then q3kv_prefill_attn computes
 * the same causal attention as q3kv_verify_attn (new token t of slot b sees
 * positions [0, ctx_len - n_new + t]) for up to 8192 new tokens per slot.
 * Arguments, layout, workspace contract, errors and status bits are those of
 * q3kv_verify_attn, with d_n_new / max_n_new in place of d_n_q / max_n_q and
 * the workspace sized by q3kv_prefill_workspace_bytes.  Each CTA of the
 * tensor-core leg reads only the positions its rows can see. */
Q3KV_API int q3kv_prefill_workspace_bytes(const q3kv_cache_desc* desc, int32_t num_slots, int64_t max_ctx_len,
                         int32_t max_n_new, int32_t impl, int32_t split_positions, size_t* bytes);
Q3KV_API int q3kv_prefill_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                     const int32_t* d_page_table, int32_t max_pages_per_slot,
                     const int32_t* d_ctx_len, const int32_t* d_n_new, const int32_t* d_q_offsets,
                     int32_t num_slots, int64_t max_ctx_len, int32_t max_n_new, int32_t layer,
                     const void* q, int32_t dtype, float* out,
                     int32_t impl, int32_t split_positions,
                     void* d_workspace, size_t workspace_bytes, int32_t* d_status);

/* ---- fp8 E4M3 comparison cache ------------------------------------------------
 * The format the pages' server uses by default ("KV cache" stack bullet of the
 * "Quasar" (q27) wiki): K and V stored as fp8 E4M3 with a scale-free,
 * saturating conversion and no rotation.  It exists here to measure what the
 * 3-bit cache buys: 512 bytes per (position, kv head) against 224.
 *   - Record: 256 E4M3 bytes (dims in order) per head vector; pages, page
 *     tables, lengths and allocator exactly as the 3-bit cache, with 256-byte
 *     records in place of 112-byte ones.
 *   - Conversion: round to nearest (ties to even mantissa); magnitudes above
 *     448 and infinities to +-448; NaN stays NaN and, like an infinity, sets
 *     Q3KV_STATUS_NONFINITE_INPUT.
 *   - Verify: out = softmax(q . k / 16) v over the decoded values (no
 *     rotation), on the tensor-core leg only (impl AUTO or MMA; FMA returns
 *     Q3KV_ERR_UNSUPPORTED).  Its workspace is q3kv_workspace_bytes(...) with
 *     the same arguments.
 * Arguments, ownership, errors and status bits are those of q3kv_pool_bytes,
 * q3kv_append and q3kv_verify_attn. */
Q3KV_API int q3kv_fp8_pool_bytes(const q3kv_cache_desc* desc, size_t* bytes);
Q3KV_API int q3kv_fp8_append(void* stream, const q3kv_cache_desc* desc, void* d_pool, const int32_t* d_page_table,
                    int32_t max_pages_per_slot, const int32_t* d_slot_len, const int32_t* d_n_new,
                    const int32_t* d_row_offsets, int32_t num_slots, int32_t max_n_new, int32_t layer,
                    const void* k, const void* v, int32_t dtype, int32_t* d_status);
Q3KV_API int q3kv_fp8_verify_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                     const int32_t* d_page_table, int32_t max_pages_per_slot,
                     const int32_t* d_ctx_len, const int32_t* d_n_q, const int32_t* d_q_offsets,
                     int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q, int32_t layer,
                     const void* q, int32_t dtype, float* out,
                     int32_t impl, int32_t split_positions,
                     void* d_workspace, size_t workspace_bytes, int32_t* d_status);

/* ---- turbo5k-style cache: 5-bit Lloyd-Max K, 3-bit V ----------------------------
 * Source: the turbo5k bullet of the "Quasar" (q27) wiki's stack list: 5-bit K
 * with 32 Lloyd-Max centroids over the same WHT rotation, 82-byte K blocks per
 * 128 dims, and the 3-bit V -- the pages' fix for the 3-bit cache's tail
 * errors.  This library's reading:
 *   - K: y = H x (the 3-bit codec's rotation); per 128-dim half an fp16 scale
 *     s = root mean square of y (float32 squares summed within each run of 8
 *     elements from its first, then over runs pairwise); v = y / s (IEEE
 *     float32), code = the number of the 31 float32 midpoints of the float32
 *     Lloyd-Max centroids of N(0, 1) below v (s == 0: code 16); value c_code s.
 *   - K record, 164 bytes: bytes 0..127 the low nibbles of the 256 codes (two
 *     per byte, even element low), 128..159 their 5th bits (element d at bit
 *     d % 8 of byte 128 + d / 8), 160..163 the two fp16 scales.
 *   - V record: the 3-bit codec's 112 bytes.
 *   - Pool: per (page, layer, kv head) 256 K records then 256 V records:
 *     ((page * L + layer) * H + head) * 70,656 + row * 164 (K), or
 *     + 41,984 + row * 112 (V).  Pages, page tables, lengths, allocator as the
 *     3-bit cache.
 *   - Verify: both legs (impl AUTO = the tensor-core leg, which reads K_hat =
 *     centroid * s rounded to float32 and split into fp16 hi/lo, within 2^-22
 *     of the exact value, and flags Q3KV_STATUS_RANGE for a K scale above
 *     20,000); the workspace is q3kv_workspace_bytes(...) with the same impl.
 * Arguments, ownership, errors and status bits as q3kv_pool_bytes,
 * q3kv_append and q3kv_verify_attn. */
Q3KV_API int q3kv_t5k_pool_bytes(const q3kv_cache_desc* desc, size_t* bytes);
Q3KV_API int q3kv_t5k_append(void* stream, const q3kv_cache_desc* desc, void* d_pool, const int32_t* d_page_table,
                    int32_t max_pages_per_slot, const int32_t* d_slot_len, const int32_t* d_n_new,
                    const int32_t* d_row_offsets, int32_t num_slots, int32_t max_n_new, int32_t layer,
                    const void* k, const void* v, int32_t dtype, int32_t* d_status);
Q3KV_API int q3kv_t5k_verify_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                     const int32_t* d_page_table, int32_t max_pages_per_slot,
                     const int32_t* d_ctx_len, const int32_t* d_n_q, const int32_t* d_q_offsets,
                     int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q, int32_t layer,
                     const void* q, int32_t dtype, float* out,
                     int32_t impl, int32_t split_positions,
                     void* d_workspace, size_t workspace_bytes, int32_t* d_status);

/* ---- greedy acceptance and commit ------------------------------------------
 * Source: "Quasar" (q27) wiki -- the sampler paragraph of "Serving" and the
 * "Model tool protocol" bullet (greedy speculative decode is the default), and
 * the prefix-cache discussion (attention rows below the point where the drafts
 * diverge are append-only and stay valid in place: a rejected draft is undone
 * by shortening the length, and the next append overwrites its rows).
 *
 * Slot b's verify step had T_b = d_n_q[b] query tokens: t_0 (the last committed
 * token) then drafts d_1 .. d_{T_b - 1}, at rows d_q_offsets[b] + j of logits
 * and d_tokens (the same row indexing as q3kv_verify_attn); logits row j
 * predicts the token after query token j.  With g_j the argmax of row j (the
 * lowest vocabulary index among equal maxima):
 *   a    = number of leading drafts with d_{j+1} == g_j      (0 <= a <= T_b - 1)
 *   next = g_a                     (the correction, or the bonus token if a = T_b - 1)
 *   committed = ctx_len - (T_b - 1 - a)   (keeps t_0 and the accepted drafts)
 * Outputs per slot: d_n_accepted[b] = a, d_next_token[b] = next,
 * d_committed_len[b] = committed.  A slot with T_b == 0 gets (0, -1, ctx_len).
 *   logits   device [num_rows, vocab], f32 or bf16 (dtype); num_rows bounds
 *            the rows of all slots (sizes the launch; rows past the slots'
 *            rows are read but unused)
 *   d_ctx_len   cache length of each slot after the step's append; may be the
 *            same array as d_committed_len (in-place commit)
 *   workspace   device scratch of at least q3kv_accept_workspace_bytes(num_rows,
 *            vocab) bytes, 8-byte aligned, no initial contents needed; calls
 *            sharing it must not overlap on the GPU
 * Errors: Q3KV_ERR_INVALID_ARG / _UNSUPPORTED (num_rows > 65535, max_n_q > 16)
 * / _WORKSPACE_TOO_SMALL before any launch.  On the device, T_b > max_n_q,
 * T_b > ctx_len or rows past num_rows set Q3KV_STATUS_BAD_LENGTH and give the
 * slot (0, -1, ctx_len); a NaN logit sets Q3KV_STATUS_NONFINITE_INPUT (its
 * row's argmax is then unspecified).  Asynchronous on the stream. */
Q3KV_API int q3kv_accept_workspace_bytes(int32_t num_rows, int32_t vocab, size_t* bytes);   /* either call */
Q3KV_API int q3kv_accept_greedy(void* stream, const void* logits, int32_t dtype, int32_t vocab,
                       const int32_t* d_q_offsets, const int32_t* d_n_q, const int32_t* d_tokens,
                       int32_t num_slots, int32_t num_rows, int32_t max_n_q, const int32_t* d_ctx_len,
                       int32_t* d_n_accepted, int32_t* d_next_token, int32_t* d_committed_len,
                       void* d_workspace, size_t workspace_bytes, int32_t* d_status);

/* ---- sampled acceptance ------------------------------------------------------
 * Source: "Quasar" (q27) wiki, "Model tool protocol" bullet: temperature > 0
 * routes to sampled speculative decode with Gumbel-max sampling and
 * rejection-sampled acceptance, seeded and reproducible.  This call's reading
 * (without the top-p nucleus; see q3kv_accept_sample_nucleus): the drafts are point masses
 * (a deterministic drafter), p_j = softmax(logits row j / temperature), and
 *   draft d_{j+1} is accepted iff d_uniforms[row j] < p_j(d_{j+1});
 *   at the first rejected row a, next = argmax over x != d_{a+1} of
 *     logits_a[x] / temperature + G(row, x)   (a sample of p_a without the
 *     rejected token, i.e. the residual of the rejection rule);
 *   if every draft is accepted, next = the same argmax over all x of the last
 *     row (the bonus token);
 *   G(row, x) = -log(-log U), U = ((z >> 41) + 0.5) / 2^23, z = output number
 *     row * 2^32 + x of the SplitMix64 stream seeded with `seed` (rows are
 *     global logits rows).
 * Same arguments, outputs, workspace and errors as q3kv_accept_greedy, plus:
 *   temperature  > 0 and finite (else Q3KV_ERR_INVALID_ARG)
 *   d_uniforms   device float [num_rows], values in [0, 1): row j's uniform
 *                tests the draft that follows query token j (the caller draws
 *                them; the last row of a slot is unused)
 * The probabilities and keys are computed in float32; results equal the float64
 * definition except where a uniform or a key lies within rounding of a tie. */
Q3KV_API int q3kv_accept_sample(void* stream, const void* logits, int32_t dtype, int32_t vocab,
                       const int32_t* d_q_offsets, const int32_t* d_n_q, const int32_t* d_tokens,
                       int32_t num_slots, int32_t num_rows, int32_t max_n_q, const int32_t* d_ctx_len,
                       float temperature, const float* d_uniforms, uint64_t seed,
                       int32_t* d_n_accepted, int32_t* d_next_token, int32_t* d_committed_len,
                       void* d_workspace, size_t workspace_bytes, int32_t* d_status);

/* ---- sampled acceptance with the top-p nucleus ---------------------------------
 * Source: the same "Model tool protocol" bullet (sampled speculative decode
 * filters with a top-p nucleus before the Gumbel-max draw and the rejection
 * test) and the sampler paragraph of "Serving" (the nucleus is taken on the
 * temperature-scaled distribution).  Reading: the nucleus of row j is
 * {x : logits_j[x] >= l*}, l* the largest logit of the row whose tokens at or
 * above it carry at least top_p of p_j = softmax(logits_j / temperature) (all
 * tokens tied with the cut are kept); q_j = p_j restricted to the nucleus and
 * renormalised.  Then exactly q3kv_accept_sample's rule with q_j for p_j: draft
 * d_{j+1} is accepted iff d_uniforms[row j] < q_j(d_{j+1}) (0 outside the
 * nucleus), and the residual / bonus argmax of logits / temperature + G runs
 * over the nucleus only (without the rejected token).
 *   top_p   in (0, 1]; 1 gives q3kv_accept_sample's result (else
 *           Q3KV_ERR_INVALID_ARG)
 * The cut is found by a radix select over the logits' order (masses summed
 * in 2^-40 fixed point, so the search is deterministic); results equal the
 * float64 definition except where top_p, a uniform or a key lies within
 * rounding of a tie.  Same arguments, outputs, workspace and errors as
 * q3kv_accept_sample. */
Q3KV_API int q3kv_accept_sample_nucleus(void* stream, const void* logits, int32_t dtype, int32_t vocab,
                       const int32_t* d_q_offsets, const int32_t* d_n_q, const int32_t* d_tokens,
                       int32_t num_slots, int32_t num_rows, int32_t max_n_q, const int32_t* d_ctx_len,
                       float temperature, float top_p, const float* d_uniforms, uint64_t seed,
                       int32_t* d_n_accepted, int32_t* d_next_token, int32_t* d_committed_len,
                       void* d_workspace, size_t workspace_bytes, int32_t* d_status);

#ifdef __cplusplus
}
#endif
#endif /* Q3KV_H */
