// Host side of the C ABI: argument checks, the page allocator, workspace
// sizing, split-K policy and kernel dispatch.  No device memory is allocated
// here; every device buffer belongs to the caller.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <memory>
#include <new>
#include <vector>

#include "q3kv_internal.h"

using namespace q3kv;

namespace {

constexpr int kVersion = 1;
thread_local cudaError_t g_last_cuda = cudaSuccess;   // last CUDA failure seen by this host thread

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return Q3KV_OK;
    g_last_cuda = e;
    return Q3KV_ERR_CUDA;
}

int check_desc(const q3kv_cache_desc* d) {
    if (!d) return Q3KV_ERR_INVALID_ARG;
    if (d->num_layers <= 0 || d->num_kv_heads <= 0 || d->num_pages <= 0 || d->num_q_heads <= 0)
        return Q3KV_ERR_INVALID_ARG;
    if (d->head_dim != kHeadDim || d->page_size != kPageSize) return Q3KV_ERR_UNSUPPORTED;
    if (d->num_q_heads != kGroup * d->num_kv_heads) return Q3KV_ERR_UNSUPPORTED;
    if (d->num_kv_heads > 64) return Q3KV_ERR_UNSUPPORTED;
    return Q3KV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count(int* sms) {
    int dev = 0;
    int e = cuda_status(cudaGetDevice(&dev));
    if (e != Q3KV_OK) return e;
    return cuda_status(cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev));
}

struct Plan {
    int impl;
    int rows_per_chunk;
    int row_chunks;
    int split_pages;
    int num_splits;
    int split_auto;
    int split_target;
    size_t part_o_bytes;
    size_t part_ml_bytes;
    size_t q_prep_bytes;
    size_t total() const { return part_o_bytes + part_ml_bytes + q_prep_bytes; }
};

// Split-K policy.  A caller-fixed split size (split_positions) is used as
// given.  Otherwise, when the (slot, kv head, row chunk) units alone do not
// fill the GPU (tensor-core leg: one CTA per SM; CUDA-core leg: about two),
// the kernels size the splits from the slots' own lengths (split_pages_of).
// The host only knows the longest context and the slot count, so it sizes
// the grid and the workspace for up to twice an even share of the target
// CTAs per unit (and no more splits than the longest context has pages); the
// kernels never split a slot more finely than that.  A single slot (whose
// length is the longest), more than 32 slots, or units that fill the GPU on
// their own (many slots, long prefills) take the split size from the longest
// context on the host instead, an even share of the target CTAs per unit.
int make_plan(const q3kv_cache_desc* d, int32_t num_slots, int64_t max_ctx, int32_t max_n_q, int32_t impl,
              int32_t split_positions, Plan* p, int32_t max_tokens = kMaxNq) {
    if (num_slots < 0 || max_ctx < 0 || max_n_q < 0 || max_n_q > max_tokens) return Q3KV_ERR_INVALID_ARG;
    if (split_positions < 0 || split_positions % kPageSize != 0) return Q3KV_ERR_INVALID_ARG;
    if (max_ctx > (int64_t)INT32_MAX - kPageSize) return Q3KV_ERR_INVALID_ARG;
    if (impl == Q3KV_IMPL_AUTO) impl = Q3KV_IMPL_MMA;
    if (impl != Q3KV_IMPL_FMA && impl != Q3KV_IMPL_MMA) return Q3KV_ERR_INVALID_ARG;
    p->impl = impl;
    p->rows_per_chunk = (impl == Q3KV_IMPL_MMA) ? kMmaRows : kFmaRows;
    const int rows = kGroup * std::max<int32_t>(max_n_q, 1);
    p->row_chunks = (rows + p->rows_per_chunk - 1) / p->rows_per_chunk;
    const int64_t pages = std::max<int64_t>(1, (max_ctx + kPageSize - 1) / kPageSize);
    p->split_auto = 0;
    p->split_target = 0;
    if (split_positions > 0) {
        p->split_pages = split_positions / kPageSize;
        p->num_splits = (int)((pages + p->split_pages - 1) / p->split_pages);
    } else {
        int sms = 0;
        int e = device_sm_count(&sms);
        if (e != Q3KV_OK) return e;
        const int64_t target = (impl == Q3KV_IMPL_MMA) ? (int64_t)sms : 2 * (int64_t)sms;
        const int64_t units_max = (int64_t)std::max(num_slots, 1) * d->num_kv_heads * p->row_chunks;
        if (num_slots <= 1 || num_slots > 32 || units_max >= target) {
            // one slot (its length is the longest), many slots, or units that fill the
            // GPU alone: splits from the longest context, sized on the host
            const int64_t ts = std::max<int64_t>(1, target / units_max);
            p->split_pages = (int)((pages + ts - 1) / ts);
            p->num_splits = (int)((pages + p->split_pages - 1) / p->split_pages);
        } else {
            p->split_auto = 1;
            p->split_target = (int)std::max<int64_t>(1, target / d->num_kv_heads);
            p->split_pages = 0;
            p->num_splits = (int)std::min<int64_t>(pages, (2 * target + units_max - 1) / units_max);
        }
    }
    const int64_t units = (int64_t)std::max(num_slots, 1) * d->num_kv_heads * p->row_chunks;
    p->part_o_bytes = (size_t)(units * p->num_splits * p->rows_per_chunk * kHeadDim) * sizeof(float);
    p->part_ml_bytes = (size_t)(units * p->num_splits * p->rows_per_chunk * 2) * sizeof(float);
    if (p->num_splits == 1) p->part_o_bytes = p->part_ml_bytes = 0;
    p->q_prep_bytes = (impl == Q3KV_IMPL_MMA) ? (size_t)units * kQPrepBytes : 0;
    return Q3KV_OK;
}

}  // namespace

struct q3kv_allocator {
    int32_t num_pages;
    int32_t num_slots;
    int32_t max_pages_per_slot;
    std::vector<int32_t> free_list;              // stack; back() is handed out next
    std::vector<std::vector<int32_t>> owned;     // per-slot page ids in position order
};

extern "C" {

int q3kv_version(void) { return kVersion; }

const char* q3kv_last_cuda_error(void) {
    return g_last_cuda == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda);
}
int q3kv_format_version(void) { return Q3KV_FORMAT_VERSION; }

const char* q3kv_strerror(int err) {
    switch (err) {
        case Q3KV_OK: return "ok";
        case Q3KV_ERR_INVALID_ARG: return "invalid argument";
        case Q3KV_ERR_UNSUPPORTED: return "unsupported shape or option";
        case Q3KV_ERR_OUT_OF_PAGES: return "out of cache pages";
        case Q3KV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case Q3KV_ERR_CUDA: return "CUDA error";
        case Q3KV_ERR_SLOT_RANGE: return "slot index out of range";
        case Q3KV_ERR_HOST_MEMORY: return "host memory allocation failed";
        default: return "unknown error";
    }
}

int q3kv_pool_bytes(const q3kv_cache_desc* desc, size_t* bytes) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (!bytes) return Q3KV_ERR_INVALID_ARG;
    *bytes = (size_t)desc->num_pages * desc->num_layers * desc->num_kv_heads * 2 * kPageSize * kRecordBytes;
    return Q3KV_OK;
}

// No C++ exception leaves these functions: a failed host allocation is
// returned as Q3KV_ERR_HOST_MEMORY with the allocator unchanged.
int q3kv_allocator_create(int32_t num_pages, int32_t num_slots, int32_t max_pages_per_slot, q3kv_allocator** out) {
    if (!out || num_pages <= 0 || num_slots <= 0 || max_pages_per_slot <= 0) return Q3KV_ERR_INVALID_ARG;
    try {
        std::unique_ptr<q3kv_allocator> a(new q3kv_allocator());
        a->num_pages = num_pages;
        a->num_slots = num_slots;
        a->max_pages_per_slot = max_pages_per_slot;
        // capacity num_pages from here on: returning pages never reallocates
        a->free_list.resize(num_pages);
        for (int32_t i = 0; i < num_pages; ++i) a->free_list[i] = num_pages - 1 - i;   // page 0 first
        a->owned.resize(num_slots);
        *out = a.release();
    } catch (...) {
        return Q3KV_ERR_HOST_MEMORY;
    }
    return Q3KV_OK;
}

void q3kv_allocator_destroy(q3kv_allocator* a) { delete a; }

int q3kv_alloc_pages(q3kv_allocator* a, int32_t slot, int64_t n_positions, int32_t* h_page_table_row,
                     int32_t* n_pages_out) {
    if (!a || !h_page_table_row || n_positions < 0) return Q3KV_ERR_INVALID_ARG;
    if (slot < 0 || slot >= a->num_slots) return Q3KV_ERR_SLOT_RANGE;
    const int64_t need = (n_positions + kPageSize - 1) / kPageSize;
    if (need > a->max_pages_per_slot) return Q3KV_ERR_OUT_OF_PAGES;
    std::vector<int32_t>& mine = a->owned[slot];
    const int64_t extra = need - (int64_t)mine.size();
    if (extra > (int64_t)a->free_list.size()) return Q3KV_ERR_OUT_OF_PAGES;
    if (extra > 0) {
        try {
            mine.reserve((size_t)need);   // the only allocation: before anything changes
        } catch (...) {
            return Q3KV_ERR_HOST_MEMORY;
        }
    }
    for (int64_t i = 0; i < extra; ++i) {
        mine.push_back(a->free_list.back());
        a->free_list.pop_back();
    }
    for (int32_t i = 0; i < a->max_pages_per_slot; ++i)
        h_page_table_row[i] = (i < (int32_t)mine.size()) ? mine[i] : -1;
    if (n_pages_out) *n_pages_out = (int32_t)mine.size();
    return Q3KV_OK;
}

int q3kv_free_slot(q3kv_allocator* a, int32_t slot) {
    if (!a) return Q3KV_ERR_INVALID_ARG;
    if (slot < 0 || slot >= a->num_slots) return Q3KV_ERR_SLOT_RANGE;
    std::vector<int32_t>& mine = a->owned[slot];
    for (auto it = mine.rbegin(); it != mine.rend(); ++it) a->free_list.push_back(*it);
    mine.clear();
    return Q3KV_OK;
}

int q3kv_free_pages(const q3kv_allocator* a, int32_t* n_free) {
    if (!a || !n_free) return Q3KV_ERR_INVALID_ARG;
    *n_free = (int32_t)a->free_list.size();
    return Q3KV_OK;
}

}  // extern "C"

namespace {

int append_impl(int fmt, void* stream, const q3kv_cache_desc* desc, void* d_pool, const int32_t* d_page_table,
                int32_t max_pages_per_slot, const int32_t* d_slot_len, const int32_t* d_n_new,
                const int32_t* d_row_offsets, int32_t num_slots, int32_t max_n_new, int32_t layer, const void* k,
                const void* v, int32_t dtype, int32_t* d_status) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (num_slots < 0 || max_n_new < 0 || max_pages_per_slot <= 0) return Q3KV_ERR_INVALID_ARG;
    if (num_slots > 65535) return Q3KV_ERR_UNSUPPORTED;
    if (layer < 0 || layer >= desc->num_layers) return Q3KV_ERR_INVALID_ARG;
    if (dtype != Q3KV_F32 && dtype != Q3KV_BF16) return Q3KV_ERR_INVALID_ARG;
    if (num_slots == 0 || max_n_new == 0) return Q3KV_OK;
    if (!d_pool || !d_page_table || !d_slot_len || !d_n_new || !d_row_offsets || !k || !v) return Q3KV_ERR_INVALID_ARG;
    if (!aligned16(d_pool) || !aligned16(k) || !aligned16(v)) return Q3KV_ERR_INVALID_ARG;
    AppendArgs a{};
    a.pool = static_cast<uint8_t*>(d_pool);
    a.page_table = d_page_table;
    a.max_pages_per_slot = max_pages_per_slot;
    a.slot_len = d_slot_len;
    a.n_new = d_n_new;
    a.row_offsets = d_row_offsets;
    a.num_slots = num_slots;
    a.max_n_new = max_n_new;
    a.num_layers = desc->num_layers;
    a.num_kv_heads = desc->num_kv_heads;
    a.num_pages = desc->num_pages;
    a.layer = layer;
    a.k = k;
    a.v = v;
    a.dtype = dtype;
    a.status = d_status;
    a.fmt = fmt;
    if (fmt == kFmtT5k) a.t5k = t5k_table();
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(fmt == kFmtFp8 ? launch_append_fp8(a, st) : launch_append(a, st));
}

int verify_impl(int fmt, void* stream, const q3kv_cache_desc* desc, const void* d_pool, const int32_t* d_page_table,
                int32_t max_pages_per_slot, const int32_t* d_ctx_len, const int32_t* d_n_q,
                const int32_t* d_q_offsets, int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q,
                int32_t layer, const void* q, int32_t dtype, float* out, int32_t impl,
                int32_t split_positions, void* d_workspace, size_t workspace_bytes, int32_t* d_status,
                int32_t max_tokens = kMaxNq) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (num_slots < 0 || max_pages_per_slot <= 0 || layer < 0 || layer >= desc->num_layers)
        return Q3KV_ERR_INVALID_ARG;
    if (num_slots > 65535) return Q3KV_ERR_UNSUPPORTED;
    if (dtype != Q3KV_F32 && dtype != Q3KV_BF16) return Q3KV_ERR_INVALID_ARG;
    if (max_n_q > max_tokens) return Q3KV_ERR_UNSUPPORTED;
    if (impl < Q3KV_IMPL_AUTO || impl > Q3KV_IMPL_MMA) return Q3KV_ERR_INVALID_ARG;
    if (fmt == kFmtFp8 && impl == Q3KV_IMPL_FMA) return Q3KV_ERR_UNSUPPORTED;   // tensor-core leg only
    Plan p;
    e = make_plan(desc, num_slots, max_ctx_len, max_n_q, impl, split_positions, &p, max_tokens);
    if (e != Q3KV_OK) return e;
    if (num_slots == 0 || max_n_q == 0 || max_ctx_len == 0) return Q3KV_OK;
    if ((int64_t)num_slots * desc->num_kv_heads * p.row_chunks > INT32_MAX) return Q3KV_ERR_UNSUPPORTED;   // grid.x
    if (!d_pool || !d_page_table || !d_ctx_len || !d_n_q || !d_q_offsets || !q || !out) return Q3KV_ERR_INVALID_ARG;
    if (!aligned16(d_pool) || !aligned16(q) || !aligned16(out)) return Q3KV_ERR_INVALID_ARG;
    if (workspace_bytes < p.total() || (p.total() > 0 && !d_workspace)) return Q3KV_ERR_WORKSPACE_TOO_SMALL;
    if (p.num_splits > 1 && p.rows_per_chunk * (size_t)num_slots * desc->num_kv_heads * p.row_chunks > 0 &&
        (size_t)num_slots * desc->num_kv_heads * p.row_chunks > 65535)
        return Q3KV_ERR_UNSUPPORTED;
    if (d_workspace && !aligned16(d_workspace)) return Q3KV_ERR_INVALID_ARG;
    if ((int64_t)p.num_splits > 65535) return Q3KV_ERR_UNSUPPORTED;

    VerifyArgs a{};
    a.pool = static_cast<const uint8_t*>(d_pool);
    a.page_table = d_page_table;
    a.max_pages_per_slot = max_pages_per_slot;
    a.ctx_len = d_ctx_len;
    a.n_q = d_n_q;
    a.q_offsets = d_q_offsets;
    a.num_slots = num_slots;
    a.num_layers = desc->num_layers;
    a.num_kv_heads = desc->num_kv_heads;
    a.num_pages = desc->num_pages;
    a.layer = layer;
    a.q = q;
    a.dtype = dtype;
    a.out = out;
    a.max_n_q = max_n_q;
    a.split_pages = p.split_pages;
    a.num_splits = p.num_splits;
    a.split_auto = p.split_auto;
    a.split_target = p.split_target;
    a.row_chunks = p.row_chunks;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    a.part_o = p.part_o_bytes ? reinterpret_cast<float*>(ws) : nullptr;
    a.part_ml = p.part_ml_bytes ? reinterpret_cast<float*>(ws + p.part_o_bytes) : nullptr;
    a.q_prep = p.q_prep_bytes ? static_cast<void*>(ws + p.part_o_bytes + p.part_ml_bytes) : nullptr;
    a.fmt = fmt;
    if (fmt == kFmtT5k) a.t5k = t5k_table();
    a.status = d_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool mma = (p.impl == Q3KV_IMPL_MMA);
    cudaError_t ce = mma ? launch_verify_mma(a, st) : launch_verify_fma(a, st);
    if (ce == cudaSuccess) ce = launch_merge(a, p.rows_per_chunk, mma, st);
    return cuda_status(ce);
}

}  // namespace

extern "C" {

int q3kv_append(void* stream, const q3kv_cache_desc* desc, void* d_pool, const int32_t* d_page_table,
                int32_t max_pages_per_slot, const int32_t* d_slot_len, const int32_t* d_n_new,
                const int32_t* d_row_offsets, int32_t num_slots, int32_t max_n_new, int32_t layer, const void* k,
                const void* v, int32_t dtype, int32_t* d_status) {
    return append_impl(kFmtQ3, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_slot_len, d_n_new,
                       d_row_offsets, num_slots, max_n_new, layer, k, v, dtype, d_status);
}

int q3kv_verify_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool, const int32_t* d_page_table,
                     int32_t max_pages_per_slot, const int32_t* d_ctx_len, const int32_t* d_n_q,
                     const int32_t* d_q_offsets, int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q,
                     int32_t layer, const void* q, int32_t dtype, float* out, int32_t impl,
                     int32_t split_positions, void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    return verify_impl(kFmtQ3, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_ctx_len, d_n_q,
                       d_q_offsets, num_slots, max_ctx_len, max_n_q, layer, q, dtype, out, impl, split_positions,
                       d_workspace, workspace_bytes, d_status);
}

int q3kv_workspace_bytes(const q3kv_cache_desc* desc, int32_t num_slots, int64_t max_ctx_len, int32_t max_n_q,
                         int32_t impl, int32_t split_positions, size_t* bytes) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (!bytes) return Q3KV_ERR_INVALID_ARG;
    Plan p;
    e = make_plan(desc, num_slots, max_ctx_len, max_n_q, impl, split_positions, &p);
    if (e != Q3KV_OK) return e;
    *bytes = p.total();
    return Q3KV_OK;
}

int q3kv_fp8_pool_bytes(const q3kv_cache_desc* desc, size_t* bytes) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (!bytes) return Q3KV_ERR_INVALID_ARG;
    *bytes = (size_t)desc->num_pages * desc->num_layers * desc->num_kv_heads * 2 * kPageSize * kFp8RecordBytes;
    return Q3KV_OK;
}

int q3kv_fp8_append(void* stream, const q3kv_cache_desc* desc, void* d_pool, const int32_t* d_page_table,
                    int32_t max_pages_per_slot, const int32_t* d_slot_len, const int32_t* d_n_new,
                    const int32_t* d_row_offsets, int32_t num_slots, int32_t max_n_new, int32_t layer,
                    const void* k, const void* v, int32_t dtype, int32_t* d_status) {
    return append_impl(kFmtFp8, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_slot_len, d_n_new,
                       d_row_offsets, num_slots, max_n_new, layer, k, v, dtype, d_status);
}

int q3kv_fp8_verify_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                         const int32_t* d_page_table, int32_t max_pages_per_slot, const int32_t* d_ctx_len,
                         const int32_t* d_n_q, const int32_t* d_q_offsets, int32_t num_slots, int64_t max_ctx_len,
                         int32_t max_n_q, int32_t layer, const void* q, int32_t dtype, float* out, int32_t impl,
                         int32_t split_positions, void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    return verify_impl(kFmtFp8, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_ctx_len, d_n_q,
                       d_q_offsets, num_slots, max_ctx_len, max_n_q, layer, q, dtype, out, impl, split_positions,
                       d_workspace, workspace_bytes, d_status);
}

int q3kv_t5k_pool_bytes(const q3kv_cache_desc* desc, size_t* bytes) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (!bytes) return Q3KV_ERR_INVALID_ARG;
    *bytes = (size_t)desc->num_pages * desc->num_layers * desc->num_kv_heads * kT5kChunkBytes;
    return Q3KV_OK;
}

int q3kv_t5k_append(void* stream, const q3kv_cache_desc* desc, void* d_pool, const int32_t* d_page_table,
                    int32_t max_pages_per_slot, const int32_t* d_slot_len, const int32_t* d_n_new,
                    const int32_t* d_row_offsets, int32_t num_slots, int32_t max_n_new, int32_t layer,
                    const void* k, const void* v, int32_t dtype, int32_t* d_status) {
    return append_impl(kFmtT5k, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_slot_len, d_n_new,
                       d_row_offsets, num_slots, max_n_new, layer, k, v, dtype, d_status);
}

int q3kv_t5k_verify_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                         const int32_t* d_page_table, int32_t max_pages_per_slot, const int32_t* d_ctx_len,
                         const int32_t* d_n_q, const int32_t* d_q_offsets, int32_t num_slots, int64_t max_ctx_len,
                         int32_t max_n_q, int32_t layer, const void* q, int32_t dtype, float* out, int32_t impl,
                         int32_t split_positions, void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    return verify_impl(kFmtT5k, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_ctx_len, d_n_q,
                       d_q_offsets, num_slots, max_ctx_len, max_n_q, layer, q, dtype, out, impl, split_positions,
                       d_workspace, workspace_bytes, d_status);
}

int q3kv_prefill_workspace_bytes(const q3kv_cache_desc* desc, int32_t num_slots, int64_t max_ctx_len,
                                 int32_t max_n_new, int32_t impl, int32_t split_positions, size_t* bytes) {
    int e = check_desc(desc);
    if (e != Q3KV_OK) return e;
    if (!bytes) return Q3KV_ERR_INVALID_ARG;
    Plan p;
    e = make_plan(desc, num_slots, max_ctx_len, max_n_new, impl, split_positions, &p, kMaxPrefillNq);
    if (e != Q3KV_OK) return e;
    *bytes = p.total();
    return Q3KV_OK;
}

int q3kv_prefill_attn(void* stream, const q3kv_cache_desc* desc, const void* d_pool, const int32_t* d_page_table,
                      int32_t max_pages_per_slot, const int32_t* d_ctx_len, const int32_t* d_n_new,
                      const int32_t* d_q_offsets, int32_t num_slots, int64_t max_ctx_len, int32_t max_n_new,
                      int32_t layer, const void* q, int32_t dtype, float* out, int32_t impl,
                      int32_t split_positions, void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    return verify_impl(kFmtQ3, stream, desc, d_pool, d_page_table, max_pages_per_slot, d_ctx_len, d_n_new,
                       d_q_offsets, num_slots, max_ctx_len, max_n_new, layer, q, dtype, out, impl, split_positions,
                       d_workspace, workspace_bytes, d_status, kMaxPrefillNq);
}

}  // extern "C"

// ---- greedy acceptance
namespace {
// Vocabulary chunks per row: enough argmax CTAs to cover the GPU about twice,
// chunks of at least 2,048 entries, each a multiple of 8 entries.
int accept_plan(int32_t num_rows, int32_t vocab, int32_t* num_chunks, int64_t* chunk_elems) {
    if (num_rows < 0 || vocab <= 0) return Q3KV_ERR_INVALID_ARG;
    int sms = 0;
    int e = device_sm_count(&sms);
    if (e != Q3KV_OK) return e;
    const int64_t target = std::max<int64_t>(1, (2 * (int64_t)sms + std::max(num_rows, 1) - 1) / std::max(num_rows, 1));
    const int64_t most = std::max<int64_t>(1, ((int64_t)vocab + 2047) / 2048);
    const int64_t n = std::min(target, most);
    int64_t chunk = ((int64_t)vocab + n - 1) / n;
    chunk = (chunk + 7) / 8 * 8;
    *chunk_elems = chunk;
    *num_chunks = (int32_t)(((int64_t)vocab + chunk - 1) / chunk);
    return Q3KV_OK;
}
}  // namespace

extern "C" {

int q3kv_accept_workspace_bytes(int32_t num_rows, int32_t vocab, size_t* bytes) {
    if (!bytes) return Q3KV_ERR_INVALID_ARG;
    int32_t nch = 0;
    int64_t chunk = 0;
    int e = accept_plan(num_rows, vocab, &nch, &chunk);
    if (e != Q3KV_OK) return e;
    // the chunk partials, then (top-p nucleus) a row record and a 256-bin histogram per row
    *bytes = (size_t)num_rows * ((size_t)nch * kAcceptPartialBytes + kNucleusRowBytes + kNucleusHistBytes);
    return Q3KV_OK;
}

int q3kv_accept_greedy(void* stream, const void* logits, int32_t dtype, int32_t vocab, const int32_t* d_q_offsets,
                       const int32_t* d_n_q, const int32_t* d_tokens, int32_t num_slots, int32_t num_rows,
                       int32_t max_n_q, const int32_t* d_ctx_len, int32_t* d_n_accepted, int32_t* d_next_token,
                       int32_t* d_committed_len, void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    if (dtype != Q3KV_F32 && dtype != Q3KV_BF16) return Q3KV_ERR_INVALID_ARG;
    if (vocab <= 0 || num_slots < 0 || num_rows < 0 || max_n_q < 0) return Q3KV_ERR_INVALID_ARG;
    if (max_n_q > kMaxNq || num_rows > 65535 || num_slots > (1 << 30)) return Q3KV_ERR_UNSUPPORTED;
    int32_t nch = 0;
    int64_t chunk = 0;
    int e = accept_plan(num_rows, vocab, &nch, &chunk);
    if (e != Q3KV_OK) return e;
    if (num_slots == 0) return Q3KV_OK;
    if (!d_q_offsets || !d_n_q || !d_tokens || !d_ctx_len || !d_n_accepted || !d_next_token || !d_committed_len)
        return Q3KV_ERR_INVALID_ARG;
    if (num_rows > 0 && !logits) return Q3KV_ERR_INVALID_ARG;
    const size_t need = (size_t)num_rows * (size_t)nch * 8;
    if (workspace_bytes < need || (need > 0 && !d_workspace)) return Q3KV_ERR_WORKSPACE_TOO_SMALL;
    if (d_workspace && (reinterpret_cast<uintptr_t>(d_workspace) & 7u)) return Q3KV_ERR_INVALID_ARG;
    AcceptArgs a{};
    a.logits = logits;
    a.dtype = dtype;
    a.vocab = vocab;
    a.chunk_elems = chunk;
    a.num_chunks = nch;
    const size_t esize = dtype == Q3KV_F32 ? 4 : 2;
    a.vec_ok = (aligned16(logits) && ((size_t)vocab * esize) % 16 == 0) ? 1 : 0;
    a.q_offsets = d_q_offsets;
    a.n_q = d_n_q;
    a.tokens = d_tokens;
    a.num_slots = num_slots;
    a.num_rows = num_rows;
    a.max_n_q = max_n_q;
    a.ctx_len = d_ctx_len;
    a.n_accepted = d_n_accepted;
    a.next_token = d_next_token;
    a.committed_len = d_committed_len;
    a.partial = d_workspace;
    a.status = d_status;
    return cuda_status(launch_accept(a, static_cast<cudaStream_t>(stream)));
}

int q3kv_accept_sample(void* stream, const void* logits, int32_t dtype, int32_t vocab, const int32_t* d_q_offsets,
                       const int32_t* d_n_q, const int32_t* d_tokens, int32_t num_slots, int32_t num_rows,
                       int32_t max_n_q, const int32_t* d_ctx_len, float temperature, const float* d_uniforms,
                       uint64_t seed, int32_t* d_n_accepted, int32_t* d_next_token, int32_t* d_committed_len,
                       void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    if (dtype != Q3KV_F32 && dtype != Q3KV_BF16) return Q3KV_ERR_INVALID_ARG;
    if (vocab <= 0 || num_slots < 0 || num_rows < 0 || max_n_q < 0) return Q3KV_ERR_INVALID_ARG;
    if (!(temperature > 0.0f) || !(temperature < 3.0e38f)) return Q3KV_ERR_INVALID_ARG;
    if (max_n_q > kMaxNq || num_rows > 65535 || num_slots > (1 << 30)) return Q3KV_ERR_UNSUPPORTED;
    int32_t nch = 0;
    int64_t chunk = 0;
    int e = accept_plan(num_rows, vocab, &nch, &chunk);
    if (e != Q3KV_OK) return e;
    if (num_slots == 0) return Q3KV_OK;
    if (!d_q_offsets || !d_n_q || !d_tokens || !d_ctx_len || !d_n_accepted || !d_next_token || !d_committed_len)
        return Q3KV_ERR_INVALID_ARG;
    if (num_rows > 0 && (!logits || !d_uniforms)) return Q3KV_ERR_INVALID_ARG;
    const size_t need = (size_t)num_rows * (size_t)nch * kAcceptPartialBytes;
    if (workspace_bytes < need || (need > 0 && !d_workspace)) return Q3KV_ERR_WORKSPACE_TOO_SMALL;
    if (d_workspace && (reinterpret_cast<uintptr_t>(d_workspace) & 7u)) return Q3KV_ERR_INVALID_ARG;
    AcceptArgs a{};
    a.logits = logits;
    a.dtype = dtype;
    a.vocab = vocab;
    a.chunk_elems = chunk;
    a.num_chunks = nch;
    a.vec_ok = (aligned16(logits) && ((size_t)vocab * (dtype == Q3KV_F32 ? 4 : 2)) % 16 == 0) ? 1 : 0;
    a.q_offsets = d_q_offsets;
    a.n_q = d_n_q;
    a.tokens = d_tokens;
    a.num_slots = num_slots;
    a.num_rows = num_rows;
    a.max_n_q = max_n_q;
    a.ctx_len = d_ctx_len;
    a.n_accepted = d_n_accepted;
    a.next_token = d_next_token;
    a.committed_len = d_committed_len;
    a.partial = d_workspace;
    a.status = d_status;
    a.inv_tau = 1.0f / temperature;
    a.uniforms = d_uniforms;
    a.seed = seed;
    return cuda_status(launch_accept_sample(a, static_cast<cudaStream_t>(stream)));
}

int q3kv_accept_sample_nucleus(void* stream, const void* logits, int32_t dtype, int32_t vocab,
                               const int32_t* d_q_offsets, const int32_t* d_n_q, const int32_t* d_tokens,
                               int32_t num_slots, int32_t num_rows, int32_t max_n_q, const int32_t* d_ctx_len,
                               float temperature, float top_p, const float* d_uniforms, uint64_t seed,
                               int32_t* d_n_accepted, int32_t* d_next_token, int32_t* d_committed_len,
                               void* d_workspace, size_t workspace_bytes, int32_t* d_status) {
    if (!(top_p > 0.0f) || !(top_p <= 1.0f)) return Q3KV_ERR_INVALID_ARG;
    if (top_p >= 1.0f)   // the nucleus is the whole vocabulary
        return q3kv_accept_sample(stream, logits, dtype, vocab, d_q_offsets, d_n_q, d_tokens, num_slots, num_rows,
                                  max_n_q, d_ctx_len, temperature, d_uniforms, seed, d_n_accepted, d_next_token,
                                  d_committed_len, d_workspace, workspace_bytes, d_status);
    if (dtype != Q3KV_F32 && dtype != Q3KV_BF16) return Q3KV_ERR_INVALID_ARG;
    if (vocab <= 0 || num_slots < 0 || num_rows < 0 || max_n_q < 0) return Q3KV_ERR_INVALID_ARG;
    if (!(temperature > 0.0f) || !(temperature < 3.0e38f)) return Q3KV_ERR_INVALID_ARG;
    if (max_n_q > kMaxNq || num_rows > 65535 || num_slots > (1 << 30)) return Q3KV_ERR_UNSUPPORTED;
    int32_t nch = 0;
    int64_t chunk = 0;
    int e = accept_plan(num_rows, vocab, &nch, &chunk);
    if (e != Q3KV_OK) return e;
    if (num_slots == 0) return Q3KV_OK;
    if (!d_q_offsets || !d_n_q || !d_tokens || !d_ctx_len || !d_n_accepted || !d_next_token || !d_committed_len)
        return Q3KV_ERR_INVALID_ARG;
    if (num_rows > 0 && (!logits || !d_uniforms)) return Q3KV_ERR_INVALID_ARG;
    const size_t part = (size_t)num_rows * (size_t)nch * kAcceptPartialBytes;
    const size_t need = part + (size_t)num_rows * (kNucleusRowBytes + kNucleusHistBytes);
    if (workspace_bytes < need || (need > 0 && !d_workspace)) return Q3KV_ERR_WORKSPACE_TOO_SMALL;
    if (d_workspace && (reinterpret_cast<uintptr_t>(d_workspace) & 7u)) return Q3KV_ERR_INVALID_ARG;
    AcceptArgs a{};
    a.logits = logits;
    a.dtype = dtype;
    a.vocab = vocab;
    a.chunk_elems = chunk;
    a.num_chunks = nch;
    a.vec_ok = (aligned16(logits) && ((size_t)vocab * (dtype == Q3KV_F32 ? 4 : 2)) % 16 == 0) ? 1 : 0;
    a.q_offsets = d_q_offsets;
    a.n_q = d_n_q;
    a.tokens = d_tokens;
    a.num_slots = num_slots;
    a.num_rows = num_rows;
    a.max_n_q = max_n_q;
    a.ctx_len = d_ctx_len;
    a.n_accepted = d_n_accepted;
    a.next_token = d_next_token;
    a.committed_len = d_committed_len;
    a.partial = d_workspace;
    a.status = d_status;
    a.inv_tau = 1.0f / temperature;
    a.uniforms = d_uniforms;
    a.seed = seed;
    a.top_p = top_p;
    a.nucleus = d_workspace ? static_cast<void*>(static_cast<uint8_t*>(d_workspace) + part) : nullptr;
    return cuda_status(launch_accept_nucleus(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
