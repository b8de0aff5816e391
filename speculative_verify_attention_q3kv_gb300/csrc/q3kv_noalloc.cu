// Verify attention without a caller-supplied workspace.
//
// Some callers cannot hand this library a device workspace: code that runs
// where another allocator owns all device memory and must not be bypassed,
// serving loops that may not allocate once they are running, or bindings
// that only ever receive device pointers from elsewhere.  For them,
// q3kv_verify_attn_noalloc takes its split-K scratch from one fixed array that
// lives in the library's own device memory (every GPU that loads the library
// holds Q3KV_NOALLOC_SCRATCH_BYTES of it until the process exits).  The call
// itself allocates nothing: no cudaMalloc, no cudaFree, no allocating library
// routine.
//
// In host code the array's name is only a stand-in for the device symbol, so
// its device address is looked up with cudaGetSymbolAddress, once per device,
// the first time the entry point runs with that device current, and cached.
#include <cuda_runtime.h>

#include <atomic>

#include "q3kv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[Q3KV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (set-up on first use).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q3KV_ERR_CUDA;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return Q3KV_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return Q3KV_OK;
}

}  // namespace

extern "C" int q3kv_verify_attn_noalloc(void* stream, const q3kv_cache_desc* desc, const void* d_pool,
                                        const int32_t* d_page_table, int32_t max_pages_per_slot,
                                        const int32_t* d_ctx_len, const int32_t* d_n_q,
                                        const int32_t* d_q_offsets, int32_t num_slots, int64_t max_ctx_len,
                                        int32_t max_n_q, int32_t layer, const void* q, int32_t dtype, float* out,
                                        int32_t impl, int32_t split_positions, int32_t* d_status) {
    size_t need = 0;
    int e = q3kv_workspace_bytes(desc, num_slots, max_ctx_len, max_n_q, impl, split_positions, &need);
    if (e != Q3KV_OK) return e;
    if (need > (size_t)Q3KV_NOALLOC_SCRATCH_BYTES) return Q3KV_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    e = scratch_address(&scratch);
    if (e != Q3KV_OK) return e;
    // The split partials are written before they are read within the call, so
    // whatever an earlier call left in the array needs no clearing.
    return q3kv_verify_attn(stream, desc, d_pool, d_page_table, max_pages_per_slot, d_ctx_len, d_n_q, d_q_offsets,
                            num_slots, max_ctx_len, max_n_q, layer, q, dtype, out, impl, split_positions, scratch,
                            (size_t)Q3KV_NOALLOC_SCRATCH_BYTES, d_status);
}
