// Interface between the C-ABI layer and the per-dtype decode translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Arguments of the paged decode kernel (plain data, passed by value).
struct DecodeArgs {
    void* out;                   // [B, Hq, D] element type T
    const void* q;               // [B, Hq, D]
    const int32_t* block_tables; // [B, max_blocks]
    const int32_t* context_lens; // [B]
    float* ws_m;                 // [B * Hq, max_parts]   running max (log2 domain) per partition
    float* ws_l;                 // [B * Hq, max_parts]   running denominator per partition
    float* ws_o;                 // [B * Hq, max_parts, D] unnormalised output per partition
    float* ws_part;              // lean schedule: two partial records per consumer warp; row-split: two per CTA and chunk
    unsigned long long* ws_flag; // lean schedule: one flag per record, set to `epoch` when published
    unsigned long long epoch;    // lean schedule: a value no earlier call has used (never 0)
    unsigned long long wait_ns;  // lean merge: bound of its wait for the partial records (ns)
    unsigned* err;               // device error word
    // Append mode (new_key != nullptr): the new token of sequence b, new_key/new_value
    // [B, Hkv, D], sits at position L_b - 1; the kernel copies it into its staged copy of
    // that page and stores it into the cache (raw pointers below) before attending.
    const void* new_key;
    const void* new_value;
    void* key_cache;
    void* value_cache;
    // FP8 caches (E4M3 codes): float32 scales [num_blocks, num_kv_heads] for K and V.
    const float* k_scale;
    const float* v_scale;
    // FP8 cache layout [N, H_kv, 2, bs, D] (K then V of each (block, kv head)), one tensor map whose
    // 2 * bs-row box brings a page's K and V in one copy; 0: separate K and V caches.
    int kv_interleaved;
    int num_seqs, num_heads, num_kv_heads, group, head_chunks;
    // Multi-query decode: q_len query tokens per sequence at positions L - q_len .. L - 1
    // (q_len = 1: single-step decode).  A kv head serves rows = q_len * group query rows,
    // row v = t * group + h being query token t of head kvh * group + h.
    int q_len, rows;
    // Row split (the tensor-core kernel with per-row bounds, a kv head of 2..4 row chunks):
    // each consumer warp of a partition's CTA takes one row chunk and consumes every page,
    // so a page is loaded once for all of the kv head's rows (head_chunks is then 1).
    int row_split;
    int max_blocks, num_blocks;
    int partition_pages, max_parts;
    float scale_log2;            // softmax scale * log2(e)
    int lean_warps_per_cta;      // consumer warps per lean CTA
    int lean_grid;               // CTAs of the lean / row-split decode launch (set for their merge kernels)
    int lean_merge_by_boundary;  // merge grid: one CTA per boundary between warp shares, not per unit
    int lean_share_warps;        // lean schedule: consumer warps the pages are cut for (<= all of them)
    int force_restart;           // lean decode: treat the set-up made before the wait as wrong (tests)
};

// Arguments of the split-KV merge kernel.
struct MergeArgs {
    void* out;
    const int32_t* context_lens;
    const float* ws_m;
    const float* ws_l;
    const float* ws_o;
    int num_seqs, num_heads, block_size, max_blocks, partition_pages, max_parts;
    int num_kv_heads, group, q_len, rows;  // row id = (b * num_kv_heads + kvh) * rows + v
};

struct KernelInfo {
    int threads;          // threads per CTA
    int smem_bytes;       // dynamic shared memory per CTA (partitioned-grid schedule)
    int heads_per_cta;    // query heads one CTA (or warp) serves: the head-chunk width
    int ctas_per_sm;      // resident CTAs per SM, partitioned-grid schedule
    int merge_parts_cap;  // partitions the merge kernel can combine
    int lean_smem_bytes;  // dynamic shared memory per CTA, lean schedule, for the given num_seqs
    int lean_ctas_per_sm; // resident CTAs per SM, lean schedule
    int lean_warps_per_cta;
    int lean_record_floats; // floats of one partial record
    int lean_max_seqs;
    int rs_ctas_per_sm;     // resident CTAs per SM, persistent row-split schedule (0: not compiled)
    int rs_smem_bytes;      // its dynamic shared memory per CTA for the given num_seqs
    int rs_record_floats;   // floats of one of its partial records (8 rows of a chunk)
};

// kScheduleRowSplit: the persistent row-split wave (multi-query decode with 2..4 row chunks per kv
// head) and its merge.  kScheduleLeanMergeOnly: the lean merge kernel alone (diagnostics of its
// bounded wait; never a plan's schedule).
enum Schedule { kScheduleGrid = 0, kScheduleLean = 1, kScheduleRowSplit = 2, kScheduleLeanMergeOnly = 3 };

// kind: 1 = tensor-core (mma) kernel, 2 = CUDA-core kernel, 3 = tensor-core kernel with a causal bound
// per row (multi-query decode; the CUDA-core kernel always has it); gmax: head-chunk width of the
// CUDA-core kernel.
// Return false when the combination is not compiled.
bool decode_kernel_info(int dtype, int head_dim, int block_size, int kind, int gmax, int num_seqs, KernelInfo* info);
cudaError_t decode_launch(int dtype, int head_dim, int block_size, int kind, int gmax, int schedule,
                          const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeArgs& args, int grid,
                          int num_seqs, cudaStream_t stream);
cudaError_t merge_launch(int dtype, int head_dim, const MergeArgs& args, cudaStream_t stream);

// Per-dtype entry points (one translation unit each).
bool decode_kernel_info_f32(int head_dim, int block_size, int kind, int gmax, int num_seqs, KernelInfo* info);
bool decode_kernel_info_f16(int head_dim, int block_size, int kind, int gmax, int num_seqs, KernelInfo* info);
bool decode_kernel_info_bf16(int head_dim, int block_size, int kind, int gmax, int num_seqs, KernelInfo* info);
cudaError_t decode_launch_f32(int head_dim, int block_size, int kind, int gmax, int schedule,
                              const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeArgs& args,
                              int grid, int num_seqs, cudaStream_t stream);
cudaError_t decode_launch_f16(int head_dim, int block_size, int kind, int gmax, int schedule,
                              const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeArgs& args,
                              int grid, int num_seqs, cudaStream_t stream);
cudaError_t decode_launch_bf16(int head_dim, int block_size, int kind, int gmax, int schedule,
                              const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeArgs& args,
                              int grid, int num_seqs, cudaStream_t stream);
// FP8 (E4M3) caches: the lean schedule with the FP8 tensor-core consumer; dtype is the
// query/output type (PA_F16 or PA_BF16).
bool decode_kernel_info_fp8(int dtype, int head_dim, int block_size, int num_seqs, KernelInfo* info);
cudaError_t decode_launch_fp8(int dtype, int head_dim, int block_size, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, const DecodeArgs& args, int grid, int num_seqs,
                              cudaStream_t stream);
cudaError_t merge_launch_f32(int head_dim, const MergeArgs& args, cudaStream_t stream);
cudaError_t merge_launch_f16(int head_dim, const MergeArgs& args, cudaStream_t stream);
cudaError_t merge_launch_bf16(int head_dim, const MergeArgs& args, cudaStream_t stream);

}  // namespace pa
