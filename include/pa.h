/*
 * Paged decode attention on GB300 (sm_103a) — C ABI.
 *
 * The library implements single-step decode attention over a paged KV cache
 * (PagedAttention) and the two cache-maintenance kernels around it, plus a
 * host block pool that produces block tables, slot mappings and copy-on-write
 * pairs.  All signatures use plain C types: device buffers are raw pointers,
 * a stream is a `cudaStream_t` passed as `void*` (NULL = the legacy default
 * stream), sizes are ints.
 *
 * Conventions shared by every call:
 *  - Every call returns an int status (PA_OK = 0, else one of PA_ERR_*);
 *    pa_last_error_string() gives a thread-local message for the last failure.
 *  - Device buffers are owned by the caller; the library never allocates or
 *    frees device memory in these calls.
 *  - Kernel calls are asynchronous on the given stream.  Argument and launch
 *    errors come back synchronously.  Bad data found by a kernel (a block id
 *    outside the pool, a slot past the pool, a context longer than its table)
 *    does not fault: the kernel skips the access and sets a bit in a device
 *    error word, which pa_check_error() reads (it synchronises the stream).
 *  - Cache layout (MiniPaged-Qwen, section 8.2): key_cache and value_cache are
 *    contiguous [num_blocks, num_kv_heads, block_size, head_dim] arrays of the
 *    element type `dtype`; slice [pb, kvh, :, :] of one block and head is
 *    contiguous.  query/out are [num_seqs, num_heads, head_dim], key/value
 *    of the write are [num_tokens, num_kv_heads, head_dim], all contiguous.
 *  - dtype is one of PA_F32, PA_F16, PA_BF16; query, caches and out share it.
 */
#ifndef PAGED_KV_GB300_PA_H
#define PAGED_KV_GB300_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------- */
enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,    /* a null pointer, a bad size, misalignment, ... */
    PA_ERR_UNSUPPORTED = 2,    /* head_dim / block_size / dtype combination not compiled */
    PA_ERR_CUDA = 3,           /* a CUDA runtime call failed */
    PA_ERR_POOL_EXHAUSTED = 4, /* the block pool has no free block (state unchanged) */
    PA_ERR_BAD_TABLE = 5,      /* a block id outside [0, num_blocks) was met */
    PA_ERR_BAD_SLOT = 6,       /* a slot at or past num_blocks * block_size was met */
    PA_ERR_BAD_CONTEXT = 7,    /* a context length < 0 or longer than its block table */
    PA_ERR_TIMEOUT = 8,        /* a kernel-internal wait gave up (should never happen) */
    PA_ERR_NOT_FOUND = 9       /* unknown sequence id, or a block id not in use */
};

/* ---- element types ------------------------------------------------------------------- */
enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_E4M3 = 3 /* one-byte FP8 codes: pa_copy_blocks, pa_swap_blocks */ };

/* ---- decode kernel choice (pa_decode_ex) ---------------------------------------------- */
enum {
    PA_KERNEL_AUTO = 0, /* tensor-core kernel for f16/bf16, CUDA-core kernel for f32 */
    PA_KERNEL_MMA = 1,  /* f16/bf16 only: QK^T and PV on warp-level tensor-core MMA */
    PA_KERNEL_SIMT = 2  /* all dtypes: CUDA-core FMA */
};

/* Thread-local message describing the last non-OK status of this thread. */
const char* pa_last_error_string(void);

/* Library version string. */
const char* pa_version(void);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device.  Returns PA_OK, or the first of PA_ERR_BAD_TABLE,
 * PA_ERR_BAD_SLOT, PA_ERR_BAD_CONTEXT, PA_ERR_TIMEOUT whose bit was set by a
 * kernel since the last check, or PA_ERR_CUDA if the stream failed.
 */
int pa_check_error(void* stream);

/*
 * pa_write_kv — the reshape-and-cache writer (MiniPaged-Qwen, sections 8.1-8.2:
 * append_token returns the token's linear slot; the cache write kernel stores
 * the token's K/V there).
 *
 * For every token t and kv head h:
 *     key_cache  [slot / block_size, h, slot % block_size, :] = key  [t, h, :]
 *     value_cache[slot / block_size, h, slot % block_size, :] = value[t, h, :]
 * where slot = slot_mapping[t] (device int64 array of num_tokens entries).
 * A negative slot means "no write" (padding).  A slot >= num_blocks *
 * block_size is skipped and sets PA_ERR_BAD_SLOT in the device error word.
 * Bit-exact: elements are copied as raw bytes.  Slots of one call must be
 * distinct (duplicate slots race).  num_tokens == 0 is a no-op.
 */
int pa_write_kv(const void* key, const void* value, void* key_cache, void* value_cache,
                const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                int block_size, int num_blocks, int dtype, void* stream);

/*
 * pa_copy_blocks — copy-on-write block copy (vLLM and PagedAttention page,
 * copy-on-write section: a branch that appends to a shared, non-full tail
 * block first copies it into a private block).
 *
 * src_dst_pairs is a device int64 array [num_pairs, 2] of (src, dst) block
 * ids.  For every pair, block dst of key_cache and of value_cache becomes a
 * byte copy of block src (all kv heads, all slots).  The dst ids of one call
 * must be distinct and no dst may be a src of the same call (otherwise the
 * result depends on scheduling).  dtype gives the element size only (PA_E4M3 for
 * FP8 caches); value_cache NULL: the interleaved FP8 layout, key_cache holding
 * [num_blocks, H_kv, 2, block_size, head_dim] and the whole record copied.  An id outside [0, num_blocks) skips the pair
 * and sets PA_ERR_BAD_TABLE in the device error word.  num_pairs == 0 is a
 * no-op.
 */
int pa_copy_blocks(void* key_cache, void* value_cache, const int64_t* src_dst_pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                   void* stream);

/*
 * pa_write_kv_layers — pa_write_kv for every layer of a model in one launch (the
 * same slot_mapping in every layer: a sequence's physical blocks have the same ids
 * in each layer's cache).  keys, values, key_caches, value_caches are HOST arrays
 * of num_layers device pointers (read during the call; the memory they point to
 * must stay valid until the stream has passed the call): layer l's key/value
 * [num_tokens, H_kv, d] go into key_caches[l] / value_caches[l]
 * [num_blocks, H_kv, bs, d] at the slots, exactly as pa_write_kv would.
 * 1 <= num_layers <= PA_MAX_LAYERS.  A negative slot is skipped; a slot at or
 * past num_blocks * block_size sets PA_ERR_BAD_SLOT in the device error word.
 */
#define PA_MAX_LAYERS 256
int pa_write_kv_layers(const void* const* keys, const void* const* values, void* const* key_caches,
                       void* const* value_caches, int num_layers, const int64_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype, void* stream);

/*
 * pa_apply_table_deltas — apply a delta export (pa_pool_table_deltas) to a
 * device block table: block_tables[row * max_blocks_per_seq + j] = block for
 * every (row, j, block) of deltas [num_deltas, 3] int32.  deltas may be device
 * memory or page-locked host memory (read directly, no staging copy).  A row
 * outside [0, num_rows) or j outside [0, max_blocks_per_seq) is skipped and sets
 * PA_ERR_BAD_TABLE in the device error word.  Launch it on the stream of the
 * decode that reads the table: stream order keeps it after the previous decode.
 */
int pa_apply_table_deltas(int32_t* block_tables, int num_rows, int max_blocks_per_seq, const int32_t* deltas,
                          int num_deltas, void* stream);

/*
 * pa_swap_blocks — swap-out / swap-in copy of whole blocks between two caches of
 * the same block geometry (the vLLM and PagedAttention page's preemption; the
 * LLM-inference page's swap of KV blocks to CPU memory and back).  For every
 * (src, dst) row of block_pairs [num_pairs, 2] int64, block dst of dst_key_cache
 * and dst_value_cache becomes a byte copy of block src of src_key_cache and
 * src_value_cache (all kv heads, all slots; dtype gives only the element size, PA_E4M3
 * for FP8 caches).  dst_value_cache and src_value_cache both NULL: the interleaved FP8
 * layout ([num_blocks, H_kv, 2, block_size, head_dim] records, each copied whole).
 *  - each cache and block_pairs may be device memory of the current device or
 *    page-locked host memory the device can address (cudaHostAlloc, cudaHostRegister,
 *    torch pin_memory); the kernel reads and writes host memory directly over
 *    the host link, in one launch for all pairs.  Pageable host memory is
 *    rejected (PA_ERR_INVALID_ARG);
 *  - src ids index [0, src_num_blocks), dst ids [0, dst_num_blocks); a pair with
 *    an id outside its pool is skipped and sets PA_ERR_BAD_TABLE in the device
 *    error word; the dst ids of one call must be distinct;
 *  - asynchronous on `stream`: host memory involved must stay allocated and
 *    untouched by the host until the stream has passed the call.
 * num_pairs == 0 is a no-op.
 */
int pa_swap_blocks(void* dst_key_cache, void* dst_value_cache, const void* src_key_cache,
                   const void* src_value_cache, const int64_t* block_pairs, int num_pairs, int num_kv_heads,
                   int head_dim, int block_size, int src_num_blocks, int dst_num_blocks, int dtype, void* stream);

/*
 * pa_decode — single-step decode attention over the paged cache
 * (MiniPaged-Qwen, section 1 formula, sections 5.1-5.2 and 6.2; GQA mapping of
 * section 9.1).
 *
 * For every sequence b and query head qh, with g = num_heads / num_kv_heads,
 * kvh = qh / g and L = context_lens[b]:
 *     pos -> logical block pos / block_size -> pb = block_tables[b, that block],
 *     k_pos = key_cache[pb, kvh, pos % block_size, :], v_pos likewise,
 *     out[b, qh, :] = sum_pos softmax_pos(scale * <query[b, qh, :], k_pos>) * v_pos
 * with the softmax taken over all L positions (online: running max and
 * running denominator, fp32 accumulation).  L == 0 gives a zero row.
 *
 *  block_tables   device int32 [num_seqs, max_blocks_per_seq]; only the first
 *                 ceil(L / block_size) entries of a row are read.
 *  context_lens   device int32 [num_seqs].
 *  scale          softmax scale, usually 1/sqrt(head_dim).
 *  workspace      device scratch for the split-KV partials, or NULL.  With
 *                 NULL every (sequence, kv head) is done by one CTA in one
 *                 pass.  With at least pa_decode_workspace_size() bytes the
 *                 default (lean) schedule runs: one persistent wave of CTAs
 *                 whose warps each stream an equal share of all pages, and a
 *                 small merge kernel that combines the contexts cut at share
 *                 boundaries.  A smaller workspace selects partitioned
 *                 contexts (a decode kernel plus a merge kernel).  No
 *                 initialisation is needed: the lean merge tells this call's
 *                 partial records from stale ones by a per-call 64-bit epoch,
 *                 and clears every flag it consumed, so a call captured in a
 *                 CUDA graph (which replays one epoch) stays correct on every
 *                 replay.  256-byte aligned.  Calls that share a workspace
 *                 must not overlap on the GPU.
 * Requires num_heads % num_kv_heads == 0, head_dim in {64, 128, 256},
 * block_size in {16, 32} (f32: head_dim in {64, 128}), 16-byte aligned caches,
 * 4-byte aligned query/out, num_blocks * num_kv_heads * block_size < 2^31.
 */
int pa_decode(void* out, const void* query, const void* key_cache, const void* value_cache,
              const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads,
              int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
              float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_ex — pa_decode with explicit planning controls.
 *  max_context_len  an upper bound of context_lens (0 = max_blocks_per_seq *
 *                   block_size); only used to size the partitions.  A context
 *                   longer than this bound sets PA_ERR_BAD_CONTEXT.
 *  partition_pages  0 = default plan (the lean schedule when the workspace
 *                   is large enough and num_seqs <= 4096, else partitions of
 *                   about 512 tokens); > 0 = partitioned contexts of exactly
 *                   this many pages (blocks) per CTA (needs a workspace when
 *                   it splits a context); < 0 = one CTA per context (no
 *                   workspace used).
 *  kernel           PA_KERNEL_AUTO / PA_KERNEL_MMA / PA_KERNEL_SIMT.
 */
int pa_decode_ex(void* out, const void* query, const void* key_cache, const void* value_cache,
                 const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads,
                 int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                 float scale, int dtype, void* workspace, size_t workspace_bytes, int max_context_len,
                 int partition_pages, int kernel, void* stream);

/*
 * pa_decode_append — one decode step with its cache write folded in: the new
 * token of every sequence is appended at position L - 1 and attended to.
 * Equivalent to pa_write_kv with slot_mapping[b] = block_tables[b, (L_b - 1) /
 * block_size] * block_size + (L_b - 1) % block_size for every b with L_b >= 1
 * (sequences with L_b == 0 write nothing), followed by pa_decode_ex; the write
 * is the MiniPaged-Qwen append of section 8.1 (the token's slot from the block
 * table), and the attention reads the new row from the staged page instead of
 * re-reading it.
 *  new_key, new_value  device [num_seqs, num_kv_heads, head_dim] of `dtype`,
 *                      16-byte aligned.
 *  key_cache, value_cache  written: one row per (sequence, kv head).
 * Other arguments as pa_decode_ex.  The page holding position L_b - 1 must not
 * be read by another sequence of the same call (a block pool with copy-on-write
 * guarantees it: an append never writes a shared block).
 */
int pa_decode_append(void* out, const void* query, const void* new_key, const void* new_value, void* key_cache,
                     void* value_cache, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                     int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
                     int max_context_len, int partition_pages, int kernel, void* stream);

/*
 * FP8 KV cache (the LLM-inference page's quantised KV cache, FP8 among the remedies
 * when the pool runs out; the vLLM and PagedAttention page's attention metadata: KV
 * dtype and quantisation scales).  A cache element is an OCP FP8 E4M3 code (bias 7,
 * no infinities, largest finite 448, S.1111.111 = NaN), one byte, in the same layout
 * [num_blocks, H_kv, block_size, head_dim]; k_scale and v_scale are float32
 * [num_blocks, H_kv] (device), one scale per (physical block, kv head), positive and
 * finite.  The value attended is code * scale.  Choosing the scales (e.g. from the
 * block's first tokens, or one per layer) is the caller's policy.
 * Interleaved layout: with value_cache == NULL, key_cache holds [num_blocks, H_kv, 2,
 * block_size, head_dim] bytes, the K rows then the V rows of every (block, kv head),
 * so that the decode brings a page's K and V in one contiguous 2 * block_size * head_dim
 * byte copy (the same layout for pa_write_kv_fp8 and pa_decode_fp8).
 *
 * pa_write_kv_fp8 — pa_write_kv into an FP8 cache: element i of token t, kv head h
 * is stored as e4m3(x / scale[slot / block_size, h]) with x the source element
 * (dtype PA_F32, PA_F16 or PA_BF16) as float32, the division in float32, round to
 * nearest even, magnitudes above 448 saturating to 448, NaN staying NaN.
 * head_dim a multiple of 4.  Slots as pa_write_kv.
 */
int pa_write_kv_fp8(const void* key, const void* value, void* key_cache, void* value_cache, const float* k_scale,
                    const float* v_scale, const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int dtype, void* stream);
/*
 * pa_decode_fp8 — pa_decode over an FP8 cache; query and out in `dtype` (PA_F16 or
 * PA_BF16).  Compiled for head_dim 128, block_size 16 and 32 (PA_ERR_UNSUPPORTED
 * otherwise).  Runs the lean schedule (equal page shares per warp + merge) and
 * needs a workspace of pa_decode_fp8_workspace_size() bytes (PA_ERR_INVALID_ARG
 * without it); query and out 16-byte aligned.  The codes are widened to f16 exactly and multiplied on the tensor
 * cores with fp32 accumulation; the scales are applied in fp32.
 */
int pa_decode_fp8(void* out, const void* query, const void* key_cache, const void* value_cache, const float* k_scale,
                  const float* v_scale, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                  int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                  int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream);
size_t pa_decode_fp8_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int dtype);
/*
 * pa_decode_fp8_append — pa_decode_fp8 with the step's write folded in, as pa_decode_append: the
 * new token of sequence b (new_key / new_value [num_seqs, H_kv, head_dim] in `dtype`, device,
 * 16-byte aligned, read only) is quantised with the scales of the block that receives it and
 * stored at the slot the block table gives position L_b - 1, then attended.  Same cache bytes and
 * output bits as pa_write_kv_fp8 at those slots followed by pa_decode_fp8 with the same workspace.
 * value_cache NULL: interleaved layout.  A sequence with L_b == 0 writes nothing; a block id
 * outside the pool skips the store and sets PA_ERR_BAD_TABLE in the device error word; a NULL or
 * misaligned new_key / new_value, k_scale or v_scale returns PA_ERR_INVALID_ARG.
 */
int pa_decode_fp8_append(void* out, const void* query, const void* new_key, const void* new_value, void* key_cache,
                         void* value_cache, const float* k_scale, const float* v_scale, const int32_t* block_tables,
                         const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_multi — multi-query decode: the verify step of speculative decoding, or
 * the tail of a chunked prefill (vLLM and PagedAttention page, section on how the
 * attention kernel reads paged KV: each sequence's query range and context length,
 * verify semantics, causal mask).  Sequence b has q_len query tokens, at positions
 * L_b - q_len .. L_b - 1 of its context (L_b = context_lens[b]; their K/V are in the
 * cache already, e.g. written with pa_write_kv); query token t attends positions
 * 0 .. L_b - q_len + t, and a token whose bound is negative gets a zero row.
 *  query, out  [num_seqs, q_len, num_heads, head_dim].
 * A kv head serves q_len * g query rows, so each page of the context is read once for
 * all of them.  Other arguments as pa_decode_ex; q_len == 1 is pa_decode_ex.  The
 * workspace for the default plan: pa_decode_multi_workspace_size().
 */
int pa_decode_multi(void* out, const void* query, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int q_len, int num_heads,
                    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                    float scale, int dtype, void* workspace, size_t workspace_bytes, int max_context_len,
                    int partition_pages, int kernel, void* stream);
size_t pa_decode_multi_workspace_size(int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int max_blocks_per_seq, int dtype);
/* The plan pa_decode_multi would use (pa_decode_make_plan with q_len query tokens per sequence). */
struct pa_decode_plan;
int pa_decode_multi_make_plan(int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks_per_seq, int dtype, size_t workspace_bytes, int max_context_len,
                              int partition_pages, int kernel, struct pa_decode_plan* plan);

/* The partition plan pa_decode_ex would use on the current device. */
typedef struct pa_decode_plan {
    int kernel;            /* PA_KERNEL_MMA or PA_KERNEL_SIMT */
    int schedule;          /* 0: partitioned grid (+ merge kernel), 1: lean persistent wave,
                              2: persistent row-split wave (pa_decode_multi with 9..32 query rows
                              per kv head: a warp per chunk of 8 rows, equal page shares per CTA) */
    int partition_pages;   /* pages per CTA partition (grid schedule; 0 otherwise) */
    int max_parts;         /* partitions of the longest context (grid schedule; 0 otherwise) */
    int heads_per_cta;     /* query heads handled by one CTA */
    int grid_ctas;         /* CTAs launched */
    int threads_per_cta;
    int smem_bytes;        /* dynamic shared memory per CTA */
    size_t workspace_bytes; /* workspace this plan needs (0 for a single-pass grid) */
} pa_decode_plan;

int pa_decode_make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                        int max_blocks_per_seq, int dtype, size_t workspace_bytes, int max_context_len,
                        int partition_pages, int kernel, pa_decode_plan* plan);

/*
 * Workspace bytes pa_decode needs to use its own (heuristic) partition plan
 * on the current device, for these sizes.  0 means one pass, no workspace.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int dtype);

/*
 * Diagnostics of the bounded device waits (no counterpart on the pages).  Launches the
 * split-KV merge of the lean schedule on its own, for the plan pa_decode would use with this
 * workspace, as if the decode grid had published none of its partial records: the merge's
 * wait for them can only run out.  Each merge CTA with a cut unit gives up after
 * wait_limit_ns nanoseconds (1 .. 2e9), sets the timeout bit of the device error word
 * (pa_check_error then returns PA_ERR_TIMEOUT) and writes nothing to out; the device stays
 * usable.  Arguments as for pa_decode; PA_ERR_INVALID_ARG when these sizes do not take the
 * lean schedule.  Asynchronous on `stream`.
 */
int pa_diag_merge_timeout(void* out, const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                          int head_dim, int block_size, int max_blocks_per_seq, int dtype, void* workspace,
                          size_t workspace_bytes, unsigned long long wait_limit_ns, void* stream);

/*
 * Diagnostics of the lean schedule's early set-up (no counterpart on the pages).  The lean
 * decode reads the context lengths and the first block-table rows of every warp before it
 * waits for the previous kernel in the stream, issues the first page loads from them as soon
 * as the wait returns, and reads both again to check them; a CTA whose early reads differ
 * (the previous kernel changed them) discards those pages and sets up again.  With on != 0
 * every later lean decode of this process takes that second path in every CTA, so that tests
 * can check it; results are the same either way.  Not for production use.
 */
void pa_diag_force_restart(int on);

/*
 * pa_decode without a caller workspace: the split-KV scratch comes from one
 * fixed array of PA_STATIC_SCRATCH_BYTES compiled into the library (one copy
 * per device).  The method on the pages has no counterpart to this call; it is
 * a library convenience.
 *
 * For callers that cannot allocate device memory around a decode step: a C
 * host or plugin handed only a stream and its tensors, with no allocator to
 * ask; or a serving loop that must not call cudaMalloc/cudaFree on the step
 * path, because those can synchronise the device and fragment memory already
 * sized for the KV cache.  The call itself allocates nothing.
 *
 * Arguments, layout and results are those of pa_decode; the plan is the one
 * pa_decode uses with a workspace of pa_decode_workspace_size() bytes.
 *  - Limit: sizes whose plan needs more than PA_STATIC_SCRATCH_BYTES of scratch
 *    (for example head_dim 256 on a 152-SM GPU) are refused with
 *    PA_ERR_UNSUPPORTED and a message giving the bytes needed; use pa_decode
 *    with a workspace for those.
 *  - Nothing in the scratch has to start at zero, so nothing is cleared.
 *  - The first call on each device does setup (resolves the scratch address,
 *    loads and configures kernels): make it before any stream capture.
 *  - Calls that overlap on the GPU race on the one scratch: calls on one
 *    stream are ordered and safe; calls on different streams of one device
 *    must be ordered by the caller (events), or use pa_decode.
 */
#define PA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

int pa_decode_static_scratch(void* out, const void* query, const void* key_cache, const void* value_cache,
                             const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                             int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int max_blocks_per_seq, int num_blocks, float scale, int dtype, void* stream);

/*
 * pa_stepper — one decode step fed from page-locked host staging, sequenced in native
 * code: per step one host-to-device copy of the step's packed inputs on an upload
 * stream, the block-table deltas (if any) and the decode on a compute stream, one
 * device-to-host copy of the output on a download stream, ordered by events so that
 * with two or more slots the upload of step i + 1 overlaps the decode of step i.
 * (The step of a serving loop: queries, new K/V and lengths arrive from the host
 * every step, the outputs go back; MiniPaged-Qwen's closing notes ask for lower host
 * overhead per step.)  Memory is the caller's: pa_stepper_set_slot gives each slot's
 * host and device staging and output buffers, pa_stepper_set_call the decode call of
 * a slot (pointers into that slot's device staging, the caches, the workspace).  The
 * library creates only its own events.  Not thread-safe; one stepper per loop.
 *
 * kind: PA_STEP_DECODE (pa_decode_ex), PA_STEP_APPEND (pa_decode_append),
 * PA_STEP_FP8 (pa_decode_fp8), PA_STEP_FP8_WRITE (pa_write_kv_fp8 of the new tokens at
 * `slots`, then pa_decode_fp8), PA_STEP_FP8_APPEND (pa_decode_fp8_append).  With
 * deltas != NULL, pa_apply_table_deltas(
 * block_tables, num_seqs, max_blocks_per_seq, deltas, num_deltas) runs first.
 */
enum { PA_STEP_DECODE = 0, PA_STEP_APPEND = 1, PA_STEP_FP8 = 2, PA_STEP_FP8_WRITE = 3, PA_STEP_FP8_APPEND = 4 };
typedef struct pa_step_call {
    int kind;
    void* out;
    const void* query;
    const void* new_key;     /* PA_STEP_APPEND, PA_STEP_FP8_WRITE, PA_STEP_FP8_APPEND */
    const void* new_value;
    const int64_t* slots;    /* PA_STEP_FP8_WRITE: int64 [num_seqs] */
    void* key_cache;
    void* value_cache;
    const float* k_scale;    /* FP8 kinds */
    const float* v_scale;
    int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* deltas;   /* NULL: no table deltas */
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks;
    float scale;
    int dtype;               /* query / output type */
    void* workspace;
    size_t workspace_bytes;
    int max_context_len, partition_pages, kernel;
} pa_step_call;
typedef struct pa_stepper pa_stepper;
int pa_stepper_create(int slots, void* upload_stream, void* compute_stream, void* download_stream,
                      pa_stepper** out);
void pa_stepper_destroy(pa_stepper* st);
int pa_stepper_set_slot(pa_stepper* st, int slot, const void* host_in, void* dev_in, size_t in_bytes,
                        void* host_out, const void* dev_out, size_t out_bytes);
int pa_stepper_set_call(pa_stepper* st, int slot, const pa_step_call* call);
/* Launch step `step` on slot step % slots: upload its first upload_bytes (<= in_bytes), apply
 * num_deltas deltas, decode, download.  Asynchronous; the slot's host staging must not be
 * refilled before pa_stepper_wait of the step that last used the slot. */
int pa_stepper_launch(pa_stepper* st, int step, size_t upload_bytes, int num_deltas);
/* Block the host until the output of `step` has arrived in its slot's host buffer. */
int pa_stepper_wait(pa_stepper* st, int step);

/* ---- host block pool ----------------------------------------------------------------- */
/*
 * Fixed-size block allocator with reference counts, fork and copy-on-write
 * append.  Semantics of the BlockPool simulation on the vLLM and
 * PagedAttention page (section "最小分页与 COW 模拟"):
 *  - allocation takes the LAST id of the free list (LIFO); the list starts as
 *    0..num_blocks-1, or as `free_order` when given;
 *  - append: a fresh block if the sequence has none or its tail block is full
 *    (no copy, even if that full tail is shared); otherwise, if the tail is
 *    shared (refcount > 1), a private block is allocated, the shared tail loses
 *    one reference and the caller must copy src -> dst (cow_src/cow_dst)
 *    before writing the token; otherwise the token goes into the tail in place;
 *  - fork: the child lists the same blocks; each block's refcount + 1;
 *  - release: each block of the sequence loses one reference; a block at zero
 *    goes back to the end of the free list, in table order.
 * Every failing call leaves the pool unchanged (rollback).  Not thread-safe:
 * one pool per thread, or external locking.  Host memory only.
 */
typedef struct pa_pool pa_pool;

int pa_pool_create(int num_blocks, int block_size, const int32_t* free_order, pa_pool** out);
void pa_pool_destroy(pa_pool* pool);
int pa_seq_create(pa_pool* pool, int64_t* seq_id);
/* slot = pb * block_size + offset of the new token; cow_src/cow_dst = -1 when no copy is needed. */
int pa_seq_append(pa_pool* pool, int64_t seq_id, int64_t* slot, int64_t* cow_src, int64_t* cow_dst);
/*
 * Append one token to each of `n` sequences (in order).  slots[n] receive the
 * slots; cow_pairs (capacity n pairs, [n, 2] int64) receives the copy pairs in
 * order and *num_cow their count.  All-or-nothing: on failure nothing changed.
 */
int pa_seq_append_batch(pa_pool* pool, const int64_t* seq_ids, int n, int64_t* slots, int64_t* cow_pairs,
                        int* num_cow);
int pa_seq_fork(pa_pool* pool, int64_t parent_id, int64_t* child_id);
int pa_seq_release(pa_pool* pool, int64_t seq_id);
int pa_seq_length(const pa_pool* pool, int64_t seq_id, int64_t* length);
/*
 * pa_pool_blocks_needed — the reservation check of an iteration-level scheduler (the
 * vLLM and PagedAttention page, continuous batching: before an iteration, the blocks the
 * admitted sequences may grow into must be available): *needed receives the number of
 * free blocks that appending counts[i] tokens to seq_ids[i], for i = 0 .. n-1 in that
 * order, would take — fresh blocks past full tails and copy-on-write copies of shared
 * partial tails, exactly as pa_seq_append would, including a shared tail whose other
 * holders copied away first.  Nothing changes; the appends fit iff *needed <=
 * pa_pool_num_free().  A sequence may appear more than once.
 */
int pa_pool_blocks_needed(const pa_pool* pool, const int64_t* seq_ids, const int32_t* counts, int n,
                          int64_t* needed);
/*
 * pa_seq_swap — move sequence seq_id from pool src to pool dst (preemption: the
 * vLLM and PagedAttention page lets a request's physical blocks be released or
 * migrated while its logical tokens are kept; the LLM-inference page swaps a
 * request's KV blocks out to CPU memory and back in).  Typically one pool
 * indexes the device caches and the other a pinned host copy of the same
 * geometry; the call works either way round.
 *  - every block of the sequence's table, in table order, gets a fresh block of
 *    dst (LIFO) with the same fill; block_pairs [capacity, 2] int64 (host)
 *    receives (src block, dst block) for each, *num_pairs their count;
 *  - the sequence is then released in src (a block it shared stays there for
 *    its other holders); in dst it is *new_seq_id, its blocks private;
 *  - the caller copies the pairs' data with pa_swap_blocks before using either
 *    side again.
 * PA_ERR_POOL_EXHAUSTED (dst has fewer free blocks than the table), or
 * PA_ERR_INVALID_ARG (block sizes differ, same pool, capacity too small):
 * both pools unchanged.  PA_ERR_NOT_FOUND for an unknown id.
 */
int pa_seq_swap(pa_pool* src, pa_pool* dst, int64_t seq_id, int64_t* new_seq_id, int64_t* block_pairs,
                int capacity, int* num_pairs);
/*
 * Host export of block tables: tables [n, max_blocks] int32 (unused entries
 * -1) and lens [n] int32 for the given sequence ids.  PA_ERR_INVALID_ARG if a
 * table is wider than max_blocks.  The caller uploads them.
 */
int pa_pool_block_tables(const pa_pool* pool, const int64_t* seq_ids, int n, int32_t* tables, int max_blocks,
                         int32_t* lens);
/*
 * pa_pool_table_deltas — host export of block-table changes only (MiniPaged-Qwen's
 * closing notes: richer block metadata at lower host overhead).  Row i of a
 * device-resident table holds sequence seq_ids[i]; that table is assumed to have
 * received every earlier delta export of this pool, in order (pa_apply_table_deltas).
 *  - deltas [capacity, 3] int32 (host) receives (row, logical block, physical
 *    block) triples, *num_deltas their count; lens [n] int32 every row's length;
 *  - a sequence exported into the row it held at its last export, with no other
 *    sequence exported into that row since, sends only the entries that changed
 *    (a copy-on-write tail) or were added (a new block); otherwise all its entries;
 *  - entries past a table's end are not touched (the decode never reads them).
 * PA_ERR_INVALID_ARG (the deltas do not fit, a sequence in two rows) or
 * PA_ERR_NOT_FOUND: nothing exported and the pool unchanged.  Capacity
 * n * max_blocks always suffices.
 */
int pa_pool_table_deltas(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* deltas, int capacity,
                         int* num_deltas, int32_t* lens);
int pa_pool_num_free(const pa_pool* pool);
int pa_pool_num_blocks(const pa_pool* pool);
int pa_pool_block_size(const pa_pool* pool);
/* Reference count of `block` (0 if free); -1 if the id is outside the pool. */
int pa_pool_refcount(const pa_pool* pool, int32_t block);
/*
 * Check the pool's invariants (free and used blocks partition the pool,
 * refcount = number of tables holding the block, every table holds
 * ceil(len / block_size) blocks).  PA_OK or PA_ERR_INVALID_ARG with a message.
 */
int pa_pool_check_invariants(const pa_pool* pool);
/*
 * Checkpoint / resume of a pool: pa_pool_save writes the whole state (free list in
 * order, reference counts, fills, every sequence's table and length, the delta-export
 * bookkeeping) as a flat byte image of pa_pool_state_size() bytes; pa_pool_load
 * builds a new pool from an image, which then behaves exactly as the saved pool
 * (same ids, slots, copies and deltas for the same calls).  A truncated, corrupt or
 * inconsistent image is refused (PA_ERR_INVALID_ARG).  Host memory only.
 */
size_t pa_pool_state_size(const pa_pool* pool);
int pa_pool_save(const pa_pool* pool, void* buffer, size_t capacity, size_t* written);
int pa_pool_load(const void* buffer, size_t size, pa_pool** out);
/* Copy the free list (bottom first) into out[capacity]; returns its length or -1. */
int pa_pool_free_list(const pa_pool* pool, int32_t* out, int capacity);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_GB300_PA_H */
