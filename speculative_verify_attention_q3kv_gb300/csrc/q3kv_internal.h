// Internal declarations shared by the host entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/q3kv.h"

namespace q3kv {

constexpr int kHeadDim = 256;
constexpr int kPageSize = 256;
constexpr int kGroup = 8;            // q heads per kv head
constexpr int kRecordBytes = 112;    // one coded vector
constexpr int kCodeWords = 24;       // 96 bytes of codes
constexpr int kMaxNq = 16;           // query tokens per slot and step
constexpr int kMaxPrefillNq = 8192;  // new tokens per slot of one prefill call
constexpr int kMaxRows = kGroup * kMaxNq;

constexpr int kFp8RecordBytes = 256;  // fp8 E4M3 comparison format: one byte per element

// Cache formats: the 3-bit rotated codec, the fp8 E4M3 comparison format, and
// the turbo5k-style format (5-bit Lloyd-Max K, 3-bit V).
constexpr int kFmtQ3 = 0;
constexpr int kFmtFp8 = 1;
constexpr int kFmtT5k = 2;

// turbo5k layout: per (page, layer, kv head) 256 K records of 164 bytes
// (128 bytes of low code nibbles, 32 bytes of 5th code bits, 2 fp16 scales)
// then 256 V records of the 3-bit codec's 112 bytes.
constexpr int kT5kKRecordBytes = 164;
constexpr size_t kT5kChunkBytes = (size_t)kPageSize * (kT5kKRecordBytes + kRecordBytes);
__host__ __device__ inline size_t t5k_offset(int num_layers, int num_kv_heads, int64_t page, int layer,
                                             int kv_head, int kv, int row) {
    const size_t base = (size_t)((page * num_layers + layer) * num_kv_heads + kv_head) * kT5kChunkBytes;
    return kv == 0 ? base + (size_t)row * kT5kKRecordBytes
                   : base + (size_t)kPageSize * kT5kKRecordBytes + (size_t)row * kRecordBytes;
}

// The 32 float32 Lloyd-Max centroids of N(0, 1) and the 31 float32 midpoints
// between neighbours (turbo5k K codes), computed once on the host.
struct T5kTable {
    float c[32];
    float b[31];
};
const T5kTable& t5k_table();

// Byte offset of a record inside the pool (see q3kv_pool_bytes); records of
// rec_bytes bytes (112 for the 3-bit codec, 256 for fp8).
__host__ __device__ inline size_t record_offset(int num_layers, int num_kv_heads, int64_t page,
                                                int layer, int kv_head, int kv, int row,
                                                int rec_bytes = kRecordBytes) {
    return (size_t)((((page * num_layers + layer) * num_kv_heads + kv_head) * 2 + kv) * kPageSize + row) *
           rec_bytes;
}

// Everything a verify launch needs, resolved on the host.
struct VerifyArgs {
    const uint8_t* pool;
    const int32_t* page_table;
    int32_t max_pages_per_slot;
    const int32_t* ctx_len;
    const int32_t* n_q;
    const int32_t* q_offsets;
    int32_t num_slots;
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t num_pages;
    int32_t layer;
    const void* q;
    int32_t dtype;
    float* out;
    int32_t max_n_q;
    int32_t split_pages;       // pages per split-K unit (a fixed size; unused when split_auto)
    int32_t num_splits;        // split slots per unit in the grid and the workspace (an upper bound)
    int32_t split_auto;        // 1: the kernels size splits from the slots' own lengths (split_pages_of)
    int32_t split_target;      // automatic policy: (slot, row chunk, split) CTAs per kv head to aim for
    int32_t row_chunks;        // CTAs along the query rows of one kv head
    float* part_o;             // [slots, kv_heads, row_chunks, splits, rows_per_chunk, 256]
    float* part_ml;            // [slots, kv_heads, row_chunks, splits, rows_per_chunk, 2]
    void* q_prep;              // tensor-core leg: [unit][hi|lo][64 x 256] fp16 (rotated) queries
    int32_t fmt;               // kFmtQ3, kFmtFp8 or kFmtT5k
    int32_t* status;
    T5kTable t5k;              // turbo5k only
};

struct AppendArgs {
    uint8_t* pool;
    const int32_t* page_table;
    int32_t max_pages_per_slot;
    const int32_t* slot_len;
    const int32_t* n_new;
    const int32_t* row_offsets;
    int32_t num_slots;
    int32_t max_n_new;
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t num_pages;
    int32_t layer;
    const void* k;
    const void* v;
    int32_t dtype;
    int32_t* status;
    int32_t fmt;               // kFmtQ3 or kFmtT5k (fp8 has its own kernel)
    T5kTable t5k;              // turbo5k only
};

// Greedy acceptance of a verify step (argmax kernel + acceptance kernel).
struct AcceptArgs {
    const void* logits;        // [num_rows, vocab] f32 or bf16
    int32_t dtype;
    int32_t vocab;
    int64_t chunk_elems;       // vocabulary entries per argmax CTA (a multiple of 8)
    int32_t num_chunks;
    int32_t vec_ok;            // rows are 16-byte aligned: 16-byte loads
    const int32_t* q_offsets;
    const int32_t* n_q;
    const int32_t* tokens;     // [num_rows] query tokens (t_0, drafts)
    int32_t num_slots;
    int32_t num_rows;
    int32_t max_n_q;
    const int32_t* ctx_len;
    int32_t* n_accepted;
    int32_t* next_token;
    int32_t* committed_len;
    void* partial;             // [num_rows, num_chunks] per-chunk results
    int32_t* status;
    // sampled acceptance only
    float inv_tau;             // 1 / temperature
    const float* uniforms;     // [num_rows] draft-test uniforms
    uint64_t seed;             // Gumbel noise stream
    // top-p nucleus only
    float top_p;
    void* nucleus;             // [num_rows] NucleusRow, then [num_rows][256] u64 histograms
};
// Per-row scratch of the nucleus search (workspace, after the chunk partials).
constexpr size_t kNucleusRowBytes = 64;
constexpr size_t kNucleusHistBytes = 256 * 8;
constexpr size_t kAcceptPartialBytes = 24;   // largest per-chunk record (sampled acceptance)
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t stream);
cudaError_t launch_accept_sample(const AcceptArgs& a, cudaStream_t stream);
cudaError_t launch_accept_nucleus(const AcceptArgs& a, cudaStream_t stream);

// FMA (CUDA-core) leg: rows per CTA, and its workspace/launch.
constexpr int kFmaRows = 64;
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_append_fp8(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_verify_fma(const VerifyArgs& a, cudaStream_t stream);
// tcgen05 leg: 64 rows per CTA, one CTA per SM (shared memory bound); the
// rotated fp16 hi/lo queries of one unit, as the kernel's B operand of QK.
constexpr int kMmaRows = 64;
constexpr size_t kQPrepBytes = 2 * (size_t)kMmaRows * kHeadDim * 2;
cudaError_t launch_verify_mma(const VerifyArgs& a, cudaStream_t stream);
// Split-K combine + inverse rotation (after either leg when num_splits > 1).
cudaError_t launch_merge(const VerifyArgs& a, int rows_per_chunk, bool log2_units, cudaStream_t stream);

}  // namespace q3kv
