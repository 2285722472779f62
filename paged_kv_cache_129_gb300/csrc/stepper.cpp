// Native step runner: the per-step sequence of copies, waits and library calls of a
// decode loop fed from page-locked host staging (upload -> deltas + decode -> download),
// ordered by events across three streams.  It owns only its events; every buffer is the
// caller's.
#include <cstring>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

struct pa_stepper {
    struct Slot {
        const void* host_in = nullptr;
        void* dev_in = nullptr;
        size_t in_bytes = 0;
        void* host_out = nullptr;
        const void* dev_out = nullptr;
        size_t out_bytes = 0;
        pa_step_call call{};
        bool has_call = false;
        bool used = false;
        cudaEvent_t uploaded = nullptr, decoded = nullptr, downloaded = nullptr;
    };
    cudaStream_t up = nullptr, comp = nullptr, down = nullptr;
    std::vector<Slot> slots;
};

namespace {

int cuda_err(cudaError_t e, const char* what) {
    return pa::fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void destroy_events(pa_stepper* st) {
    for (auto& s : st->slots) {
        if (s.uploaded) cudaEventDestroy(s.uploaded);
        if (s.decoded) cudaEventDestroy(s.decoded);
        if (s.downloaded) cudaEventDestroy(s.downloaded);
        s.uploaded = s.decoded = s.downloaded = nullptr;
    }
}

int run_call(const pa_step_call& c, int num_deltas, cudaStream_t stream) {
    void* sp = static_cast<void*>(stream);
    if (c.deltas && num_deltas > 0) {
        const int st = pa_apply_table_deltas(c.block_tables, c.num_seqs, c.max_blocks_per_seq, c.deltas, num_deltas,
                                             sp);
        if (st != PA_OK) return st;
    }
    switch (c.kind) {
        case PA_STEP_DECODE:
            return pa_decode_ex(c.out, c.query, c.key_cache, c.value_cache, c.block_tables, c.context_lens,
                                c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size,
                                c.max_blocks_per_seq, c.num_blocks, c.scale, c.dtype, c.workspace, c.workspace_bytes,
                                c.max_context_len, c.partition_pages, c.kernel, sp);
        case PA_STEP_APPEND:
            return pa_decode_append(c.out, c.query, c.new_key, c.new_value, c.key_cache, c.value_cache,
                                    c.block_tables, c.context_lens, c.num_seqs, c.num_heads, c.num_kv_heads,
                                    c.head_dim, c.block_size, c.max_blocks_per_seq, c.num_blocks, c.scale, c.dtype,
                                    c.workspace, c.workspace_bytes, c.max_context_len, c.partition_pages, c.kernel,
                                    sp);
        case PA_STEP_FP8_WRITE: {
            const int st = pa_write_kv_fp8(c.new_key, c.new_value, c.key_cache, c.value_cache, c.k_scale, c.v_scale,
                                           c.slots, c.num_seqs, c.num_kv_heads, c.head_dim, c.block_size,
                                           c.num_blocks, c.dtype, sp);
            if (st != PA_OK) return st;
        }
            [[fallthrough]];
        case PA_STEP_FP8:
            return pa_decode_fp8(c.out, c.query, c.key_cache, c.value_cache, c.k_scale, c.v_scale, c.block_tables,
                                 c.context_lens, c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size,
                                 c.max_blocks_per_seq, c.num_blocks, c.scale, c.dtype, c.workspace,
                                 c.workspace_bytes, sp);
        case PA_STEP_FP8_APPEND:
            return pa_decode_fp8_append(c.out, c.query, c.new_key, c.new_value, c.key_cache, c.value_cache, c.k_scale,
                                        c.v_scale, c.block_tables, c.context_lens, c.num_seqs, c.num_heads,
                                        c.num_kv_heads, c.head_dim, c.block_size, c.max_blocks_per_seq, c.num_blocks,
                                        c.scale, c.dtype, c.workspace, c.workspace_bytes, sp);
        default:
            return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper: unknown step kind %d", c.kind);
    }
}

}  // namespace

extern "C" {

int pa_stepper_create(int slots, void* upload_stream, void* compute_stream, void* download_stream,
                      pa_stepper** out) {
    if (!out) return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_create: out is NULL");
    *out = nullptr;
    if (slots < 1 || slots > 64) return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_create: slots=%d", slots);
    pa_stepper* st = new (std::nothrow) pa_stepper();
    if (!st) return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_create: out of host memory");
    st->up = static_cast<cudaStream_t>(upload_stream);
    st->comp = static_cast<cudaStream_t>(compute_stream);
    st->down = static_cast<cudaStream_t>(download_stream);
    st->slots.resize(slots);
    for (auto& s : st->slots) {
        cudaError_t e = cudaEventCreateWithFlags(&s.uploaded, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.decoded, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.downloaded, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            destroy_events(st);
            delete st;
            return cuda_err(e, "pa_stepper_create: cudaEventCreateWithFlags");
        }
    }
    *out = st;
    return PA_OK;
}

void pa_stepper_destroy(pa_stepper* st) {
    if (!st) return;
    destroy_events(st);
    delete st;
}

int pa_stepper_set_slot(pa_stepper* st, int slot, const void* host_in, void* dev_in, size_t in_bytes, void* host_out,
                        const void* dev_out, size_t out_bytes) {
    if (!st || slot < 0 || slot >= (int)st->slots.size())
        return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_set_slot: bad stepper or slot %d", slot);
    if ((in_bytes && (!host_in || !dev_in)) || (out_bytes && (!host_out || !dev_out)))
        return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_set_slot: NULL buffer");
    auto& s = st->slots[slot];
    s.host_in = host_in;
    s.dev_in = dev_in;
    s.in_bytes = in_bytes;
    s.host_out = host_out;
    s.dev_out = dev_out;
    s.out_bytes = out_bytes;
    return PA_OK;
}

int pa_stepper_set_call(pa_stepper* st, int slot, const pa_step_call* call) {
    if (!st || slot < 0 || slot >= (int)st->slots.size() || !call)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_set_call: bad stepper, slot %d or call", slot);
    if (call->kind < PA_STEP_DECODE || call->kind > PA_STEP_FP8_APPEND)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_set_call: unknown step kind %d", call->kind);
    st->slots[slot].call = *call;
    st->slots[slot].has_call = true;
    return PA_OK;
}

int pa_stepper_launch(pa_stepper* st, int step, size_t upload_bytes, int num_deltas) {
    if (!st || step < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_launch: bad stepper or step");
    auto& s = st->slots[step % st->slots.size()];
    if (!s.has_call) return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_launch: slot has no call");
    if (upload_bytes > s.in_bytes || num_deltas < 0)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_launch: upload of %zu bytes > %zu, or num_deltas < 0",
                        upload_bytes, s.in_bytes);
    cudaError_t e = cudaSuccess;
    // upload: after the slot's previous decode has read its inputs
    if (s.used) e = cudaStreamWaitEvent(st->up, s.decoded, 0);
    if (e == cudaSuccess && upload_bytes)
        e = cudaMemcpyAsync(s.dev_in, s.host_in, upload_bytes, cudaMemcpyHostToDevice, st->up);
    if (e == cudaSuccess) e = cudaEventRecord(s.uploaded, st->up);
    // decode: after the upload, and after the slot's previous output has been downloaded
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st->comp, s.uploaded, 0);
    if (e == cudaSuccess && s.used) e = cudaStreamWaitEvent(st->comp, s.downloaded, 0);
    if (e != cudaSuccess) return cuda_err(e, "pa_stepper_launch: upload");
    const int status = run_call(s.call, num_deltas, st->comp);
    if (status != PA_OK) return status;
    e = cudaEventRecord(s.decoded, st->comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st->down, s.decoded, 0);
    if (e == cudaSuccess && s.out_bytes)
        e = cudaMemcpyAsync(s.host_out, s.dev_out, s.out_bytes, cudaMemcpyDeviceToHost, st->down);
    if (e == cudaSuccess) e = cudaEventRecord(s.downloaded, st->down);
    if (e != cudaSuccess) return cuda_err(e, "pa_stepper_launch: download");
    s.used = true;
    return PA_OK;
}

int pa_stepper_wait(pa_stepper* st, int step) {
    if (!st || step < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_stepper_wait: bad stepper or step");
    const cudaError_t e = cudaEventSynchronize(st->slots[step % st->slots.size()].downloaded);
    if (e != cudaSuccess) return cuda_err(e, "pa_stepper_wait");
    return PA_OK;
}

}  // extern "C"
