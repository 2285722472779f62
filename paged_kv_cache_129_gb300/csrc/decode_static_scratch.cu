// pa_decode_static_scratch: pa_decode with its split-KV scratch taken from a
// fixed array compiled into the library, for callers that cannot allocate
// device memory around the call (see include/pa.h for who and why).
//
// The array lives in this translation unit alone, so under lazy module loading
// (the CUDA default) only a process that calls this entry point pays its
// PA_STATIC_SCRATCH_BYTES of device memory.
#include <cstddef>
#include <mutex>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace {

// The scratch: split-KV partial records of one pa_decode call.  Nothing in it
// needs to start at zero: every record a merge reads is written earlier in the
// same call (and a static __device__ array starts zeroed anyway).
static __device__ __align__(256) unsigned char g_pa_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device; resolved once per
// device (with that device current) and cached.
int scratch_address(void** out) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return pa::fail(PA_ERR_CUDA, "pa_decode_static_scratch: cudaGetDevice: %s", cudaGetErrorString(e));
    if (device < 0 || device >= kMaxDevices)
        return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_static_scratch: device index %d", device);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress((void**)&p, g_pa_static_scratch);
        if (e != cudaSuccess)
            return pa::fail(PA_ERR_CUDA, "pa_decode_static_scratch: cudaGetSymbolAddress(scratch): %s (%s)",
                            cudaGetErrorName(e), cudaGetErrorString(e));
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_static_scratch(void* out, const void* query, const void* key_cache, const void* value_cache,
                                        const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                        int num_heads, int num_kv_heads, int head_dim, int block_size,
                                        int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                        void* stream) {
    pa::clear_error();
    if (num_seqs < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_static_scratch: num_seqs=%d", num_seqs);
    void* scratch = nullptr;
    int st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    // The scratch pa_decode's own plan wants for these sizes (0: one pass, none).
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                 max_blocks_per_seq, dtype);
    if (need > (size_t)PA_STATIC_SCRATCH_BYTES)
        return pa::fail(PA_ERR_UNSUPPORTED,
                        "pa_decode_static_scratch: these sizes need %zu bytes of scratch, more than the %zu bytes "
                        "(PA_STATIC_SCRATCH_BYTES) built into the library; call pa_decode with a workspace of "
                        "pa_decode_workspace_size() bytes instead",
                        need, (size_t)PA_STATIC_SCRATCH_BYTES);
    // Same plan as pa_decode given a workspace of exactly `need` bytes.
    return pa_decode(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                     need ? scratch : nullptr, need, stream);
}
