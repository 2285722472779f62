// C-ABI entry points: argument checks, the split-KV plan, TMA descriptors, the
// device error word and the thread-local error message.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>
#include <random>
#include <string>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "decode_launch.h"
#include "kv_ops.h"
#include "pa.h"
#include "pa_common.cuh"
#include "pa_internal.h"

// One error word per device, set by kernels with atomicOr (see pa_common.cuh).
__device__ unsigned int g_pa_device_error_word;

namespace pa {

namespace {
thread_local std::string g_message;
constexpr int kMaxDevices = 64;
std::atomic<int> g_force_restart{0};  // pa_diag_force_restart
}  // namespace

// An NVTX range around a C-ABI call, so that profilers show each call by name (a no-op when no
// tool is attached).
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_message = buf;
    return code;
}

void clear_error() { g_message.clear(); }

bool decode_kernel_info(int dtype, int head_dim, int block_size, int kind, int gmax, int num_seqs, KernelInfo* info) {
    switch (dtype) {
        case PA_F32: return decode_kernel_info_f32(head_dim, block_size, kind, gmax, num_seqs, info);
        case PA_F16: return decode_kernel_info_f16(head_dim, block_size, kind, gmax, num_seqs, info);
        case PA_BF16: return decode_kernel_info_bf16(head_dim, block_size, kind, gmax, num_seqs, info);
        default: return false;
    }
}

cudaError_t decode_launch(int dtype, int head_dim, int block_size, int kind, int gmax, int schedule,
                          const CUtensorMap& k, const CUtensorMap& v, const DecodeArgs& a, int grid, int num_seqs,
                          cudaStream_t s) {
    switch (dtype) {
        case PA_F32: return decode_launch_f32(head_dim, block_size, kind, gmax, schedule, k, v, a, grid, num_seqs, s);
        case PA_F16: return decode_launch_f16(head_dim, block_size, kind, gmax, schedule, k, v, a, grid, num_seqs, s);
        case PA_BF16: return decode_launch_bf16(head_dim, block_size, kind, gmax, schedule, k, v, a, grid, num_seqs, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t merge_launch(int dtype, int head_dim, const MergeArgs& a, cudaStream_t s) {
    switch (dtype) {
        case PA_F32: return merge_launch_f32(head_dim, a, s);
        case PA_F16: return merge_launch_f16(head_dim, a, s);
        case PA_BF16: return merge_launch_bf16(head_dim, a, s);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

// Internal element code of an FP8 (E4M3) cache, for the tensor-map cache (not a public dtype).
constexpr int kCacheE4M3 = 16;

int elem_bytes(int dtype) { return dtype == PA_F32 ? 4 : (dtype == kCacheE4M3 || dtype == PA_E4M3) ? 1 : 2; }
// element types the byte movers (block copy, swap) accept
bool bytes_dtype_ok(int dtype) { return dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16 || dtype == PA_E4M3; }
bool dtype_ok(int dtype) { return dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A value for DecodeArgs::epoch that no earlier call of this process has used, and
// that a workspace left by another process (or holding any other data) is most
// unlikely to contain: a 64-bit counter that starts at a random value, never 0.
unsigned long long next_epoch() {
    static std::atomic<unsigned long long> counter{[] {
        std::random_device rd;
        const unsigned long long t =
            (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
        return (((unsigned long long)rd() << 32) ^ (unsigned long long)rd()) ^ (t * 0x9E3779B97F4A7C15ull);
    }()};
    unsigned long long e = 0;
    while (e == 0) e = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    return e;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceState {
    unsigned* error_word = nullptr;
    int num_sms = 0;
};

std::mutex g_dev_mutex;
DeviceState g_dev[kMaxDevices];

int current_device_state(DeviceState** out) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (device < 0 || device >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device index %d", device);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState& st = g_dev[device];
    if (!st.error_word) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pa_device_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        st.error_word = static_cast<unsigned*>(p);
    }
    *out = &st;
    return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of a cache: rows = num_blocks * H_kv * bs (one row per slot and head), columns = d.
// The box is 128 bytes of d by bs rows, loaded with the 128-byte swizzle.
// interleave = 2: an FP8 cache holding K then V of every (block, kv head) ([N, H_kv, 2, bs, d]): twice
// the rows, and a box of 2 * bs rows that brings a page's K and V in one copy.
int encode_cache_map_uncached(CUtensorMap* map, const void* base, int dtype, int num_blocks, int num_kv_heads,
                              int block_size, int head_dim, int interleave = 1) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int eb = elem_bytes(dtype);
    const CUtensorMapDataType type = dtype == PA_F32       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : dtype == PA_F16     ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                     : dtype == kCacheE4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)num_blocks * num_kv_heads * block_size * interleave};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * eb};
    cuuint32_t box[2] = {(cuuint32_t)(128 / eb), (cuuint32_t)(block_size * interleave)};
    cuuint32_t estrides[2] = {1, 1};
    CUresult r = encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estrides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return PA_OK;
}

// The same caches are described again on every call of a decode loop: keep the last few
// descriptors of this thread (a descriptor is a pure function of these arguments).
int encode_cache_map(CUtensorMap* map, const void* base, int dtype, int num_blocks, int num_kv_heads,
                     int block_size, int head_dim, int interleave = 1) {
    struct Entry {
        const void* base;
        int dtype, num_blocks, num_kv_heads, block_size, head_dim, interleave;
        CUtensorMap map;
    };
    constexpr int kEntries = 8;
    thread_local Entry entries[kEntries] = {};
    thread_local int next = 0;
    for (const Entry& e : entries)
        if (e.base == base && e.base && e.dtype == dtype && e.num_blocks == num_blocks &&
            e.num_kv_heads == num_kv_heads && e.block_size == block_size && e.head_dim == head_dim &&
            e.interleave == interleave) {
            *map = e.map;
            return PA_OK;
        }
    const int st =
        encode_cache_map_uncached(map, base, dtype, num_blocks, num_kv_heads, block_size, head_dim, interleave);
    if (st != PA_OK) return st;
    entries[next] = Entry{base, dtype, num_blocks, num_kv_heads, block_size, head_dim, interleave, *map};
    next = (next + 1) % kEntries;
    return PA_OK;
}

struct Plan {
    int kind = 0;
    int dkind = 0;  // the kernel instantiation: kind, or 3 for the tensor-core kernel with causal bounds
    bool row_split = false;  // one CTA per partition takes all of a kv head's row chunks, a warp each
    int schedule = kScheduleGrid;
    int gmax = 8;
    int head_chunks = 1;
    int units = 0;
    int partition_pages = 1;
    int max_parts = 1;
    long long grid = 0;
    size_t ws_bytes = 0;
    size_t off_m = 0, off_l = 0, off_o = 0;  // partitioned grid: offsets of m, l and o~
    size_t off_part = 0;                     // lean: warp partial records
    size_t off_flag = 0;                     // lean: one flag per record
    KernelInfo ki{};
};

void workspace_layout(int num_seqs, int num_heads, int head_dim, int max_parts, Plan* p) {
    if (max_parts <= 1) {
        p->ws_bytes = p->off_m = p->off_l = p->off_o = 0;
        return;
    }
    const size_t rows = (size_t)num_seqs * num_heads * max_parts;
    p->off_m = 0;
    p->off_l = p->off_m + align256(rows * sizeof(float));
    p->off_o = p->off_l + align256(rows * sizeof(float));
    p->ws_bytes = p->off_o + align256(rows * head_dim * sizeof(float));
}

// has_ws: false means no workspace is usable (single pass forced).
// q_len > 1: multi-query decode; a kv head then serves q_len * group query rows.
int make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks, int dtype,
              bool has_ws, size_t ws_avail, int max_context_len, int partition_pages, int kernel, Plan* plan,
              int q_len = 1, bool fp8 = false) {
    if (!dtype_ok(dtype)) return fail(PA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_heads=%d must be a positive multiple of num_kv_heads=%d", num_heads,
                    num_kv_heads);
    if (head_dim <= 0 || block_size <= 0 || max_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "head_dim=%d block_size=%d max_blocks_per_seq=%d", head_dim, block_size,
                    max_blocks);
    if ((long long)max_blocks * block_size >= (1ll << 31))
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq * block_size must be < 2^31");
    if (q_len < 1 || (long long)q_len * num_heads >= (1 << 24))
        return fail(PA_ERR_INVALID_ARG, "q_len=%d must be positive (and q_len * num_heads < 2^24)", q_len);
    Plan p;
    const int rows = q_len * (num_heads / num_kv_heads);  // query rows per kv head
    if (fp8) {
        // FP8 caches: the lean schedule with the FP8 tensor-core consumer, single-query decode.
        if (dtype != PA_F16 && dtype != PA_BF16)
            return fail(PA_ERR_UNSUPPORTED, "FP8 decode needs f16 or bf16 queries");
        if (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_MMA)
            return fail(PA_ERR_UNSUPPORTED, "FP8 decode has only the tensor-core kernel");
        if (q_len != 1) return fail(PA_ERR_UNSUPPORTED, "FP8 decode is single-query");
        if (partition_pages != 0)
            return fail(PA_ERR_UNSUPPORTED, "FP8 decode has only the lean schedule (partition_pages must be 0)");
        p.kind = PA_KERNEL_MMA;
        p.dkind = 4;
        if (!decode_kernel_info_fp8(dtype, head_dim, block_size, num_seqs, &p.ki))
            return fail(PA_ERR_UNSUPPORTED, "no FP8 decode kernel for dtype=%d head_dim=%d block_size=%d", dtype,
                        head_dim, block_size);
        p.head_chunks = (rows + p.ki.heads_per_cta - 1) / p.ki.heads_per_cta;
        p.units = num_seqs * num_kv_heads * p.head_chunks;
        if (num_seqs > p.ki.lean_max_seqs)
            return fail(PA_ERR_UNSUPPORTED, "FP8 decode: num_seqs=%d > %d", num_seqs, p.ki.lean_max_seqs);
        if ((long long)num_seqs * max_blocks * num_kv_heads * p.head_chunks >= (1ll << 31))
            return fail(PA_ERR_UNSUPPORTED, "FP8 decode: num_seqs * max_blocks * units is too large");
        DeviceState* dev = nullptr;
        int st = current_device_state(&dev);
        if (st != PA_OK) return st;
        const long long ctas = (long long)dev->num_sms * p.ki.lean_ctas_per_sm;
        const size_t records = (size_t)ctas * p.ki.lean_warps_per_cta * 2;
        const size_t off_flag = align256(records * (size_t)p.ki.lean_record_floats * sizeof(float));
        const size_t need = off_flag + align256(records * sizeof(unsigned long long));
        if (!has_ws || need > ws_avail)
            return fail(PA_ERR_INVALID_ARG, "FP8 decode needs a workspace of %zu bytes (%zu given)", need,
                        has_ws ? ws_avail : (size_t)0);
        p.schedule = kScheduleLean;
        p.partition_pages = 0;
        p.max_parts = 0;
        p.grid = ctas;
        p.ws_bytes = need;
        p.off_part = 0;
        p.off_flag = off_flag;
        *plan = p;
        return PA_OK;
    }
    if (kernel == PA_KERNEL_AUTO) {
        p.kind = dtype == PA_F32 ? PA_KERNEL_SIMT : PA_KERNEL_MMA;
    } else if (kernel == PA_KERNEL_MMA || kernel == PA_KERNEL_SIMT) {
        p.kind = kernel;
    } else {
        return fail(PA_ERR_INVALID_ARG, "unknown kernel choice %d", kernel);
    }
    if (p.kind == PA_KERNEL_MMA && dtype == PA_F32)
        return fail(PA_ERR_UNSUPPORTED, "the tensor-core kernel needs f16 or bf16");
    p.gmax = 8;
    if (p.kind == PA_KERNEL_SIMT) {
        const int g = rows < 8 ? rows : 8;
        p.gmax = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
    }
    p.dkind = (p.kind == PA_KERNEL_MMA && q_len > 1) ? 3 : p.kind;
    if (!decode_kernel_info(dtype, head_dim, block_size, p.dkind, p.gmax, num_seqs, &p.ki))
        return fail(PA_ERR_UNSUPPORTED, "no %s decode kernel for dtype=%d head_dim=%d block_size=%d",
                    p.kind == PA_KERNEL_MMA ? "tensor-core" : "CUDA-core", dtype, head_dim, block_size);
    p.head_chunks = (rows + p.ki.heads_per_cta - 1) / p.ki.heads_per_cta;
    // Multi-query rows of a kv head in 2..4 chunks: row split on the partitioned grid, so that
    // every page is loaded once for all the chunks (as separate units each chunk would stream
    // the pages again).
    if (p.dkind == 3 && p.head_chunks >= 2 && p.head_chunks <= p.ki.lean_warps_per_cta) {
        p.row_split = true;
        p.head_chunks = 1;
    }
    p.units = num_seqs * num_kv_heads * p.head_chunks;

    long long max_ctx = (long long)max_blocks * block_size;
    if (max_context_len > 0 && max_context_len < max_ctx) max_ctx = max_context_len;
    int nblk_max = (int)((max_ctx + block_size - 1) / block_size);
    if (nblk_max < 1) nblk_max = 1;

    DeviceState* dev = nullptr;
    int st = current_device_state(&dev);
    if (st != PA_OK) return st;
    const long long slots = (long long)dev->num_sms * p.ki.ctas_per_sm;

    // Lean schedule: one persistent wave; every consumer warp streams an equal share of all pages.
    // (Worth it when there are fewer units than consumer warps: then units must be split
    // to keep every SM streaming, and equal shares balance them.  With more units than
    // that, whole-unit CTAs already balance and need no merge.  So a 16/32-bit lean plan always
    // merges with one CTA per unit; the merge grid by share boundary serves FP8 plans alone.)
    const long long lean_ctas = (long long)dev->num_sms * p.ki.lean_ctas_per_sm;
    if (partition_pages == 0 && has_ws && !p.row_split && num_seqs <= p.ki.lean_max_seqs &&
        (long long)p.units < lean_ctas * p.ki.lean_warps_per_cta &&
        (long long)num_seqs * max_blocks * num_kv_heads * p.head_chunks < (1ll << 31)) {
        const long long ctas = lean_ctas;
        const size_t records = (size_t)ctas * p.ki.lean_warps_per_cta * 2;  // two per consumer warp
        const size_t rec_bytes = (size_t)p.ki.lean_record_floats * sizeof(float);
        const size_t off_flag = align256(records * rec_bytes);
        const size_t need = off_flag + align256(records * sizeof(unsigned long long));
        if (need <= ws_avail) {
            p.schedule = kScheduleLean;
            p.partition_pages = 0;
            p.max_parts = 0;
            p.grid = ctas;
            p.ws_bytes = need;
            p.off_part = 0;
            p.off_flag = off_flag;
            *plan = p;
            return PA_OK;
        }
    }

    // Row split (multi-query decode, 2..4 row chunks per kv head): one persistent wave, every CTA an
    // equal share of all pages, each page read once for all of its kv head's rows.
    if (p.row_split && partition_pages == 0 && has_ws && p.ki.rs_ctas_per_sm > 0 && num_seqs <= p.ki.lean_max_seqs &&
        (long long)num_seqs * max_blocks * num_kv_heads < (1ll << 31)) {
        const long long ctas = (long long)dev->num_sms * p.ki.rs_ctas_per_sm;
        const size_t need = align256((size_t)ctas * 2 * 4 * p.ki.rs_record_floats * sizeof(float));
        if (need <= ws_avail) {
            p.schedule = kScheduleRowSplit;
            p.partition_pages = 0;
            p.max_parts = 0;
            p.grid = ctas;
            p.ws_bytes = need;
            p.off_part = 0;
            *plan = p;
            return PA_OK;
        }
    }

    int pp;
    if (partition_pages < 0 || !has_ws) {
        if (partition_pages > 0 && partition_pages < nblk_max)
            return fail(PA_ERR_INVALID_ARG, "partition_pages=%d splits contexts but no workspace was given",
                        partition_pages);
        pp = nblk_max;
    } else if (partition_pages > 0) {
        pp = partition_pages < nblk_max ? partition_pages : nblk_max;
    } else {
        if ((long long)p.units >= 4 * slots) {
            pp = nblk_max;  // whole contexts: at least four waves of CTAs already
        } else {
            // About 512 tokens per partition; shorter when that leaves fewer than two waves of CTAs.
            pp = 512 / block_size > 8 ? 512 / block_size : 8;
            while (pp > 8 && (long long)p.units * ((nblk_max + pp - 1) / pp) < 2 * slots) pp /= 2;
            if (pp > nblk_max) pp = nblk_max;
        }
    }
    for (;;) {
        p.partition_pages = pp;
        p.max_parts = (nblk_max + pp - 1) / pp;
        workspace_layout(num_seqs, num_heads * q_len, head_dim, p.max_parts, &p);
        const bool fits = p.max_parts == 1 || (p.ws_bytes <= ws_avail && p.max_parts <= p.ki.merge_parts_cap);
        if (fits) break;
        if (partition_pages > 0)
            return fail(PA_ERR_INVALID_ARG,
                        "workspace of %zu bytes is too small for partition_pages=%d (needs %zu, or too many parts)",
                        ws_avail, partition_pages, p.ws_bytes);
        pp = pp * 2 < nblk_max ? pp * 2 : nblk_max;
    }
    p.grid = (long long)p.max_parts * p.units;
    if (p.grid >= (1ll << 31)) return fail(PA_ERR_UNSUPPORTED, "grid of %lld CTAs is too large", p.grid);
    *plan = p;
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_last_error_string(void) { return g_message.c_str(); }

const char* pa_version(void) { return "paged_kv_cache_129_gb300 0.1.0 (sm_103a)"; }

int pa_check_error(void* stream) {
    clear_error();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    DeviceState* dev = nullptr;
    int st = current_device_state(&dev);
    if (st != PA_OK) return st;
    unsigned word = 0;
    e = cudaMemcpy(&word, dev->error_word, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word == 0) return PA_OK;
    const unsigned zero = 0;
    e = cudaMemcpy(dev->error_word, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    if (word & kErrBadTable) return fail(PA_ERR_BAD_TABLE, "a kernel met a block id outside the pool (word 0x%x)", word);
    if (word & kErrBadSlot) return fail(PA_ERR_BAD_SLOT, "a kernel met a slot past the pool (word 0x%x)", word);
    if (word & kErrBadContext)
        return fail(PA_ERR_BAD_CONTEXT, "a context length was negative or longer than its table (word 0x%x)", word);
    return fail(PA_ERR_TIMEOUT, "a kernel-internal wait gave up (word 0x%x)", word);
}

int pa_write_kv(const void* key, const void* value, void* key_cache, void* value_cache, const int64_t* slot_mapping,
                int num_tokens, int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                void* stream) {
    CallRange nvtx_range("pa_write_kv");
    clear_error();
    if (!dtype_ok(dtype)) return fail(PA_ERR_INVALID_ARG, "pa_write_kv: unknown dtype %d", dtype);
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: bad sizes");
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: NULL pointer");
    if (!aligned(slot_mapping, 8)) return fail(PA_ERR_INVALID_ARG, "pa_write_kv: slot_mapping must be 8-byte aligned");
    const int eb = elem_bytes(dtype);
    if (!aligned(key, eb) || !aligned(value, eb) || !aligned(key_cache, eb) || !aligned(value_cache, eb))
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: buffers must be aligned to the element size");
    DeviceState* dev = nullptr;
    int st = current_device_state(&dev);
    if (st != PA_OK) return st;
    WriteArgs a{key, value, key_cache, value_cache, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                num_blocks, eb, dev->error_word};
    cudaError_t e = write_kv_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_write_kv launch");
    return PA_OK;
}

int pa_copy_blocks(void* key_cache, void* value_cache, const int64_t* src_dst_pairs, int num_pairs, int num_kv_heads,
                   int head_dim, int block_size, int num_blocks, int dtype, void* stream) {
    CallRange nvtx_range("pa_copy_blocks");
    clear_error();
    if (!bytes_dtype_ok(dtype)) return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: unknown dtype %d", dtype);
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: bad sizes");
    if (num_pairs == 0) return PA_OK;
    if (!key_cache || !src_dst_pairs) return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: NULL pointer");
    // value_cache NULL: one cache of [N, H_kv, 2, bs, d] records (interleaved FP8), each copied whole
    const bool single = value_cache == nullptr;
    if (!aligned(src_dst_pairs, 8)) return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: pairs must be 8-byte aligned");
    const int eb = elem_bytes(dtype);
    if (!aligned(key_cache, eb) || !aligned(value_cache, eb))
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: caches must be aligned to the element size");
    DeviceState* dev = nullptr;
    int st = current_device_state(&dev);
    if (st != PA_OK) return st;
    CopyArgs a{key_cache, single ? key_cache : value_cache, src_dst_pairs, num_pairs,
               single ? 2 * num_kv_heads : num_kv_heads, head_dim, block_size, num_blocks, eb, single ? 1 : 0,
               dev->error_word};
    cudaError_t e = copy_blocks_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_copy_blocks launch");
    return PA_OK;
}

namespace {

// The address at which the current device reaches p: device memory of that device as is,
// page-locked host memory through its device mapping.  Pageable host memory and memory of
// another device are refused.
int device_address(const void* p, int device, const char* what, const void** out) {
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PA_ERR_INVALID_ARG, "%s is not memory the CUDA runtime knows (%s)", what,
                    cudaGetErrorName(e));
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
            if (at.device != device)
                return fail(PA_ERR_INVALID_ARG, "%s is memory of device %d, not of the current %d",
                            what, at.device, device);
            *out = p;
            return PA_OK;
        case cudaMemoryTypeManaged:
            *out = p;
            return PA_OK;
        case cudaMemoryTypeHost:
            if (!at.devicePointer)
                return fail(PA_ERR_INVALID_ARG, "%s is page-locked but not mapped for the device", what);
            *out = at.devicePointer;
            return PA_OK;
        default:
            return fail(PA_ERR_INVALID_ARG,
                        "%s is pageable host memory; page-lock it (cudaHostAlloc, cudaHostRegister)",
                        what);
    }
}

}  // namespace

static_assert(PA_MAX_LAYERS == kMaxLayers, "the header's layer limit is the kernel's");

int pa_write_kv_layers(const void* const* keys, const void* const* values, void* const* key_caches,
                       void* const* value_caches, int num_layers, const int64_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype, void* stream) {
    CallRange nvtx_range("pa_write_kv_layers");
    clear_error();
    if (!dtype_ok(dtype)) return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: unknown dtype %d", dtype);
    if (num_layers < 1 || num_layers > kMaxLayers)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: num_layers=%d outside [1, %d]", num_layers, kMaxLayers);
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: bad sizes");
    if (!keys || !values || !key_caches || !value_caches)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: NULL pointer array");
    if (num_tokens == 0) return PA_OK;
    if (!slot_mapping || !aligned(slot_mapping, 8))
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: slot_mapping must be non-NULL and 8-byte aligned");
    const int eb = elem_bytes(dtype);
    LayerPtrs ptrs;
    for (int l = 0; l < num_layers; ++l) {
        if (!keys[l] || !values[l] || !key_caches[l] || !value_caches[l])
            return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: NULL pointer for layer %d", l);
        if (!aligned(keys[l], eb) || !aligned(values[l], eb) || !aligned(key_caches[l], eb) ||
            !aligned(value_caches[l], eb))
            return fail(PA_ERR_INVALID_ARG, "pa_write_kv_layers: layer %d buffers not aligned to the element size", l);
        ptrs.key[l] = keys[l];
        ptrs.value[l] = values[l];
        ptrs.key_cache[l] = key_caches[l];
        ptrs.value_cache[l] = value_caches[l];
    }
    DeviceState* dev = nullptr;
    int st = current_device_state(&dev);
    if (st != PA_OK) return st;
    WriteLayersArgs a{&ptrs, num_layers, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, num_blocks, eb,
                      dev->error_word};
    cudaError_t e = write_kv_layers_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_write_kv_layers launch");
    return PA_OK;
}

int pa_apply_table_deltas(int32_t* block_tables, int num_rows, int max_blocks_per_seq, const int32_t* deltas,
                          int num_deltas, void* stream) {
    CallRange nvtx_range("pa_apply_table_deltas");
    clear_error();
    if (num_rows < 0 || max_blocks_per_seq < 0 || num_deltas < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_apply_table_deltas: bad sizes");
    if (num_deltas == 0) return PA_OK;
    if (!block_tables || !deltas) return fail(PA_ERR_INVALID_ARG, "pa_apply_table_deltas: NULL pointer");
    if (!aligned(block_tables, 4) || !aligned(deltas, 4))
        return fail(PA_ERR_INVALID_ARG, "pa_apply_table_deltas: tables and deltas must be 4-byte aligned");
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const void* dd = nullptr;
    const void* tt = nullptr;
    int st = device_address(deltas, device, "deltas", &dd);
    if (st == PA_OK) st = device_address(block_tables, device, "block_tables", &tt);
    if (st != PA_OK) return st;
    DeviceState* dev = nullptr;
    st = current_device_state(&dev);
    if (st != PA_OK) return st;
    DeltaArgs a{static_cast<int32_t*>(const_cast<void*>(tt)), num_rows, max_blocks_per_seq,
                static_cast<const int32_t*>(dd), num_deltas, dev->error_word};
    e = apply_table_deltas_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_apply_table_deltas launch");
    return PA_OK;
}

int pa_swap_blocks(void* dst_key_cache, void* dst_value_cache, const void* src_key_cache, const void* src_value_cache,
                   const int64_t* block_pairs, int num_pairs, int num_kv_heads, int head_dim, int block_size,
                   int src_num_blocks, int dst_num_blocks, int dtype, void* stream) {
    CallRange nvtx_range("pa_swap_blocks");
    clear_error();
    if (!bytes_dtype_ok(dtype)) return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: unknown dtype %d", dtype);
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || src_num_blocks < 0 ||
        dst_num_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: bad sizes");
    if (num_pairs == 0) return PA_OK;
    if (!dst_key_cache || !src_key_cache || !block_pairs || (!dst_value_cache != !src_value_cache))
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: NULL pointer (value caches: both or neither)");
    // both value caches NULL: [N, H_kv, 2, bs, d] records (interleaved FP8), each copied whole
    const bool single = dst_value_cache == nullptr;
    if (!aligned(block_pairs, 8)) return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: pairs must be 8-byte aligned");
    const int eb = elem_bytes(dtype);
    if (!aligned(dst_key_cache, eb) || !aligned(dst_value_cache, eb) || !aligned(src_key_cache, eb) ||
        !aligned(src_value_cache, eb))
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: caches must be aligned to the element size");
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const void* dk = nullptr;
    const void* dv = nullptr;
    const void* sk = nullptr;
    const void* sv = nullptr;
    const void* pr = nullptr;
    int st = device_address(dst_key_cache, device, "dst_key_cache", &dk);
    if (st == PA_OK && !single) st = device_address(dst_value_cache, device, "dst_value_cache", &dv);
    if (st == PA_OK) st = device_address(src_key_cache, device, "src_key_cache", &sk);
    if (st == PA_OK && !single) st = device_address(src_value_cache, device, "src_value_cache", &sv);
    if (single) {
        dv = dk;
        sv = sk;
    }
    if (st == PA_OK) st = device_address(block_pairs, device, "block_pairs", &pr);
    if (st != PA_OK) return st;
    DeviceState* dev = nullptr;
    st = current_device_state(&dev);
    if (st != PA_OK) return st;
    SwapArgs a{const_cast<void*>(dk), const_cast<void*>(dv), sk, sv, static_cast<const int64_t*>(pr), num_pairs,
               single ? 2 * num_kv_heads : num_kv_heads, head_dim, block_size, src_num_blocks, dst_num_blocks, eb,
               dev->num_sms, single ? 1 : 0, dev->error_word};
    e = swap_blocks_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_swap_blocks launch");
    return PA_OK;
}

int pa_decode_make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                        int max_blocks_per_seq, int dtype, size_t workspace_bytes, int max_context_len,
                        int partition_pages, int kernel, pa_decode_plan* out) {
    clear_error();
    if (!out) return fail(PA_ERR_INVALID_ARG, "pa_decode_make_plan: out is NULL");
    Plan p;
    int st = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype,
                       workspace_bytes > 0, workspace_bytes, max_context_len, partition_pages, kernel, &p);
    if (st != PA_OK) return st;
    out->kernel = p.kind;
    out->schedule = p.schedule;
    out->partition_pages = p.partition_pages;
    out->max_parts = p.max_parts;
    out->heads_per_cta = p.ki.heads_per_cta;
    out->grid_ctas = (int)p.grid;
    out->threads_per_cta = p.ki.threads;
    out->smem_bytes = p.schedule == kScheduleRowSplit ? p.ki.rs_smem_bytes
                      : p.schedule == kScheduleLean   ? p.ki.lean_smem_bytes
                                                      : p.ki.smem_bytes;
    out->workspace_bytes = p.ws_bytes;
    return PA_OK;
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks_per_seq, int dtype) {
    Plan p;
    if (make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype, true,
                  (size_t)-1, 0, 0, PA_KERNEL_AUTO, &p) != PA_OK)
        return 0;
    return p.ws_bytes;
}

}  // extern "C"

namespace pa {
namespace {

// pa_decode_ex, and pa_decode_append when new_key != nullptr.
int decode_impl(void* out, const void* query, const void* new_key, const void* new_value, const void* key_cache,
                const void* value_cache, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes, int max_context_len,
                int partition_pages, int kernel, void* stream, int q_len = 1, const float* k_scale = nullptr,
                const float* v_scale = nullptr) {
    CallRange nvtx_range("pa_decode");
    clear_error();
    const bool fp8 = k_scale != nullptr;
    if (fp8 && (!v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4)))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_fp8: k_scale/v_scale must be non-NULL and 4-byte aligned");
    if (fp8 && (!aligned(query, 16) || !aligned(out, 16)))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_fp8: query and out must be 16-byte aligned");
    if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "pa_decode: num_seqs=%d", num_seqs);
    if (new_key && (!new_value || !aligned(new_key, 16) || !aligned(new_value, 16)))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_append: new_key/new_value must be non-NULL and 16-byte aligned");
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !key_cache || (!value_cache && !fp8) || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "pa_decode: NULL pointer");
    if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "pa_decode: num_blocks=%d", num_blocks);
    if (num_kv_heads <= 0 || (long long)num_blocks * num_kv_heads * block_size >= (1ll << 31))
        return fail(PA_ERR_INVALID_ARG, "pa_decode: num_blocks * num_kv_heads * block_size must be < 2^31");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "pa_decode: scale is not finite");
    if (!aligned(key_cache, 16) || !aligned(value_cache, 16))  // (a NULL value cache is aligned)
        return fail(PA_ERR_INVALID_ARG, "pa_decode: caches must be 16-byte aligned");
    if (!aligned(query, 4) || !aligned(out, 4) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return fail(PA_ERR_INVALID_ARG, "pa_decode: query/out/tables/lens must be 4-byte aligned");
    if (workspace && !aligned(workspace, 256))
        return fail(PA_ERR_INVALID_ARG, "pa_decode: workspace must be 256-byte aligned");
    Plan p;
    int st = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype,
                       workspace != nullptr && workspace_bytes > 0, workspace ? workspace_bytes : 0, max_context_len,
                       partition_pages, kernel, &p, q_len, fp8);
    if (st != PA_OK) return st;
    DeviceState* dev = nullptr;
    st = current_device_state(&dev);
    if (st != PA_OK) return st;

    CUtensorMap tk, tv;
    const int cache_type = fp8 ? kCacheE4M3 : dtype;
    const bool interleaved = fp8 && value_cache == nullptr;  // K and V of a (block, head) in one record
    st = encode_cache_map(&tk, key_cache, cache_type, num_blocks, num_kv_heads, block_size, head_dim,
                          interleaved ? 2 : 1);
    if (st != PA_OK) return st;
    if (interleaved) {
        tv = tk;
    } else {
        st = encode_cache_map(&tv, value_cache, cache_type, num_blocks, num_kv_heads, block_size, head_dim);
        if (st != PA_OK) return st;
    }

    DecodeArgs a{};
    a.out = out;
    a.q = query;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    char* ws = static_cast<char*>(workspace);
    const bool grid_split = p.schedule == kScheduleGrid && p.max_parts > 1;
    a.ws_m = grid_split ? reinterpret_cast<float*>(ws + p.off_m) : nullptr;
    a.ws_l = grid_split ? reinterpret_cast<float*>(ws + p.off_l) : nullptr;
    a.ws_o = grid_split ? reinterpret_cast<float*>(ws + p.off_o) : nullptr;
    a.ws_part = (p.schedule == kScheduleLean || p.schedule == kScheduleRowSplit)
                    ? reinterpret_cast<float*>(ws + p.off_part)
                    : nullptr;
    a.ws_flag = p.schedule == kScheduleLean ? reinterpret_cast<unsigned long long*>(ws + p.off_flag) : nullptr;
    a.epoch = p.schedule == kScheduleLean ? next_epoch() : 0;
    a.wait_ns = kWaitLimitNs;
    a.force_restart = g_force_restart.load(std::memory_order_relaxed);
    a.new_key = new_key;
    a.new_value = new_key ? new_value : nullptr;
    a.key_cache = new_key ? const_cast<void*>(key_cache) : nullptr;
    a.value_cache = new_key ? const_cast<void*>(value_cache) : nullptr;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.kv_interleaved = interleaved ? 1 : 0;
    a.lean_warps_per_cta = p.ki.lean_warps_per_cta;
    a.err = dev->error_word;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_heads / num_kv_heads;
    a.q_len = q_len;
    a.rows = q_len * a.group;
    a.head_chunks = p.head_chunks;
    a.row_split = p.row_split ? 1 : 0;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.partition_pages = p.partition_pages;
    a.max_parts = p.max_parts;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);  // log2(e)
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = fp8 ? decode_launch_fp8(dtype, head_dim, block_size, tk, tv, a, (int)p.grid, num_seqs, s)
                        : decode_launch(dtype, head_dim, block_size, p.dkind, p.gmax, p.schedule, tk, tv, a,
                                        (int)p.grid, num_seqs, s);
    if (e != cudaSuccess) return cuda_fail(e, "pa_decode: decode kernel launch");
    if (grid_split) {
        MergeArgs m{out, context_lens, a.ws_m, a.ws_l, a.ws_o, num_seqs, num_heads, block_size, max_blocks_per_seq,
                    p.partition_pages, p.max_parts, num_kv_heads, a.group, q_len, a.rows};
        e = merge_launch(dtype, head_dim, m, s);
        if (e != cudaSuccess) return cuda_fail(e, "pa_decode: merge kernel launch");
    }
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" {

int pa_decode_ex(void* out, const void* query, const void* key_cache, const void* value_cache,
                 const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads,
                 int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                 int dtype, void* workspace, size_t workspace_bytes, int max_context_len, int partition_pages,
                 int kernel, void* stream) {
    return decode_impl(out, query, nullptr, nullptr, key_cache, value_cache, block_tables, context_lens, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                       workspace, workspace_bytes, max_context_len, partition_pages, kernel, stream);
}

int pa_decode_append(void* out, const void* query, const void* new_key, const void* new_value, void* key_cache,
                     void* value_cache, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                     int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
                     int max_context_len, int partition_pages, int kernel, void* stream) {
    if (!new_key) {
        clear_error();
        return fail(PA_ERR_INVALID_ARG, "pa_decode_append: new_key is NULL");
    }
    return decode_impl(out, query, new_key, new_value, key_cache, value_cache, block_tables, context_lens, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                       workspace, workspace_bytes, max_context_len, partition_pages, kernel, stream);
}

int pa_decode_multi(void* out, const void* query, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int q_len, int num_heads,
                    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                    float scale, int dtype, void* workspace, size_t workspace_bytes, int max_context_len,
                    int partition_pages, int kernel, void* stream) {
    return decode_impl(out, query, nullptr, nullptr, key_cache, value_cache, block_tables, context_lens, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                       workspace, workspace_bytes, max_context_len, partition_pages, kernel, stream, q_len);
}

int pa_decode_multi_make_plan(int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int dtype, size_t workspace_bytes, int max_context_len,
                              int partition_pages, int kernel, pa_decode_plan* out) {
    clear_error();
    if (!out) return fail(PA_ERR_INVALID_ARG, "pa_decode_multi_make_plan: out is NULL");
    Plan p;
    int st = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype,
                       workspace_bytes > 0, workspace_bytes, max_context_len, partition_pages, kernel, &p, q_len);
    if (st != PA_OK) return st;
    out->kernel = p.kind;
    out->schedule = p.schedule;
    out->partition_pages = p.partition_pages;
    out->max_parts = p.max_parts;
    out->heads_per_cta = p.ki.heads_per_cta;
    out->grid_ctas = (int)p.grid;
    out->threads_per_cta = p.ki.threads;
    out->smem_bytes = p.schedule == kScheduleRowSplit ? p.ki.rs_smem_bytes
                      : p.schedule == kScheduleLean   ? p.ki.lean_smem_bytes
                                                      : p.ki.smem_bytes;
    out->workspace_bytes = p.ws_bytes;
    return PA_OK;
}

size_t pa_decode_multi_workspace_size(int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int max_blocks_per_seq, int dtype) {
    Plan p;
    if (make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype, true,
                  (size_t)-1, 0, 0, PA_KERNEL_AUTO, &p, q_len) != PA_OK)
        return 0;
    return p.ws_bytes;
}

int pa_decode_fp8(void* out, const void* query, const void* key_cache, const void* value_cache, const float* k_scale,
                  const float* v_scale, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                  int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                  int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (!k_scale) {
        clear_error();
        return fail(PA_ERR_INVALID_ARG, "pa_decode_fp8: k_scale is NULL");
    }
    return decode_impl(out, query, nullptr, nullptr, key_cache, value_cache, block_tables, context_lens, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                       workspace, workspace_bytes, 0, 0, PA_KERNEL_AUTO, stream, 1, k_scale, v_scale);
}

int pa_decode_fp8_append(void* out, const void* query, const void* new_key, const void* new_value, void* key_cache,
                         void* value_cache, const float* k_scale, const float* v_scale, const int32_t* block_tables,
                         const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (!k_scale || !new_key) {
        clear_error();
        return fail(PA_ERR_INVALID_ARG, "pa_decode_fp8_append: k_scale or new_key is NULL");
    }
    return decode_impl(out, query, new_key, new_value, key_cache, value_cache, block_tables, context_lens, num_seqs,
                       num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                       workspace, workspace_bytes, 0, 0, PA_KERNEL_AUTO, stream, 1, k_scale, v_scale);
}

size_t pa_decode_fp8_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int dtype) {
    Plan p;
    if (make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype, true,
                  (size_t)-1, 0, 0, PA_KERNEL_AUTO, &p, 1, true) != PA_OK)
        return 0;
    return p.ws_bytes;
}

int pa_write_kv_fp8(const void* key, const void* value, void* key_cache, void* value_cache, const float* k_scale,
                    const float* v_scale, const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int dtype, void* stream) {
    CallRange nvtx_range("pa_write_kv_fp8");
    clear_error();
    if (!dtype_ok(dtype)) return fail(PA_ERR_INVALID_ARG, "pa_write_kv_fp8: unknown source dtype %d", dtype);
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 4 != 0 || block_size <= 0 ||
        num_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_fp8: bad sizes (head_dim must be a multiple of 4)");
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !k_scale || !v_scale || !slot_mapping)  // value_cache NULL: interleaved
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_fp8: NULL pointer");
    const int eb = elem_bytes(dtype);
    if (!aligned(slot_mapping, 8) || !aligned(key, eb) || !aligned(value, eb) || !aligned(key_cache, 4) ||
        !aligned(value_cache, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv_fp8: misaligned buffer");
    DeviceState* dev = nullptr;
    int st = current_device_state(&dev);
    if (st != PA_OK) return st;
    WriteFp8Args a{key, value, static_cast<uint8_t*>(key_cache), static_cast<uint8_t*>(value_cache), k_scale, v_scale,
                   slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, num_blocks, dtype,
                   dev->error_word};
    cudaError_t e = write_kv_fp8_launch(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_write_kv_fp8 launch");
    return PA_OK;
}

void pa_diag_force_restart(int on) { g_force_restart.store(on ? 1 : 0, std::memory_order_relaxed); }

int pa_diag_merge_timeout(void* out, const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                          int head_dim, int block_size, int max_blocks_per_seq, int dtype, void* workspace,
                          size_t workspace_bytes, unsigned long long wait_limit_ns, void* stream) {
    CallRange nvtx_range("pa_diag_merge_timeout");
    clear_error();
    if (num_seqs <= 0 || !out || !context_lens || !workspace)
        return fail(PA_ERR_INVALID_ARG, "pa_diag_merge_timeout: needs num_seqs > 0, out, context_lens, workspace");
    if (!aligned(workspace, 256) || !aligned(out, 4) || !aligned(context_lens, 4))
        return fail(PA_ERR_INVALID_ARG, "pa_diag_merge_timeout: misaligned pointer");
    if (wait_limit_ns == 0 || wait_limit_ns > kWaitLimitNs)
        return fail(PA_ERR_INVALID_ARG, "pa_diag_merge_timeout: wait_limit_ns must be in (0, %llu]", kWaitLimitNs);
    Plan p;
    int st = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, dtype, true,
                       workspace_bytes, 0, 0, PA_KERNEL_AUTO, &p);
    if (st != PA_OK) return st;
    if (p.schedule != kScheduleLean)
        return fail(PA_ERR_INVALID_ARG, "pa_diag_merge_timeout: these sizes do not take the lean schedule");
    DeviceState* dev = nullptr;
    st = current_device_state(&dev);
    if (st != PA_OK) return st;
    DecodeArgs a{};
    a.out = out;
    a.context_lens = context_lens;
    char* ws = static_cast<char*>(workspace);
    a.ws_part = reinterpret_cast<float*>(ws + p.off_part);
    a.ws_flag = reinterpret_cast<unsigned long long*>(ws + p.off_flag);
    a.epoch = next_epoch();  // no decode grid publishes this epoch
    a.wait_ns = wait_limit_ns;
    a.lean_warps_per_cta = p.ki.lean_warps_per_cta;
    a.err = dev->error_word;
    a.num_seqs = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = num_heads / num_kv_heads;
    a.q_len = 1;
    a.rows = a.group;
    a.head_chunks = p.head_chunks;
    a.max_blocks = max_blocks_per_seq;
    a.partition_pages = p.partition_pages;
    CUtensorMap none{};
    cudaError_t e = decode_launch(dtype, head_dim, block_size, p.dkind, p.gmax, kScheduleLeanMergeOnly, none, none, a,
                                  (int)p.grid, num_seqs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pa_diag_merge_timeout: merge kernel launch");
    return PA_OK;
}

int pa_decode(void* out, const void* query, const void* key_cache, const void* value_cache,
              const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
              int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
              void* workspace, size_t workspace_bytes, void* stream) {
    return pa_decode_ex(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs, num_heads,
                        num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, workspace,
                        workspace_bytes, 0, 0, PA_KERNEL_AUTO, stream);
}

}  // extern "C"
