// Launchers of the write and copy kernels (called by the C-ABI layer).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pa {

struct WriteArgs {
    const void* key;
    const void* value;
    void* key_cache;
    void* value_cache;
    const int64_t* slot_mapping;
    int num_tokens, num_kv_heads, head_dim, block_size, num_blocks, elem_bytes;
    unsigned* err;
};

struct CopyArgs {
    void* key_cache;
    void* value_cache;
    const int64_t* pairs;
    int num_pairs, num_kv_heads, head_dim, block_size, num_blocks, elem_bytes;
    int single;  // 1: one cache (key_cache), its blocks copied whole
    unsigned* err;
};

struct SwapArgs {
    void* dst_key;
    void* dst_value;
    const void* src_key;
    const void* src_value;
    const int64_t* pairs;  // device addresses (host memory through its device mapping)
    int num_pairs, num_kv_heads, head_dim, block_size, src_num_blocks, dst_num_blocks, elem_bytes;
    int num_sms;  // the grid is capped at a few CTAs per SM
    int single;   // 1: one cache per side (dst_key, src_key), its blocks copied whole
    unsigned* err;
};

constexpr int kMaxLayers = 256;

// Per-layer pointers, passed by value as a kernel argument.
struct LayerPtrs {
    const void* key[kMaxLayers];
    const void* value[kMaxLayers];
    void* key_cache[kMaxLayers];
    void* value_cache[kMaxLayers];
};

struct WriteLayersArgs {
    const LayerPtrs* layers;  // host struct, copied into the launch
    int num_layers;
    const int64_t* slot_mapping;
    int num_tokens, num_kv_heads, head_dim, block_size, num_blocks, elem_bytes;
    unsigned* err;
};

struct DeltaArgs {
    int32_t* block_tables;
    int num_rows, max_blocks;
    const int32_t* deltas;  // device address (host memory through its device mapping)
    int num_deltas;
    unsigned* err;
};

struct WriteFp8Args {
    const void* key;
    const void* value;
    uint8_t* key_cache;
    uint8_t* value_cache;
    const float* k_scale;
    const float* v_scale;
    const int64_t* slot_mapping;
    int num_tokens, num_kv_heads, head_dim, block_size, num_blocks;
    int src_dtype;  // PA_F32, PA_F16 or PA_BF16
    unsigned* err;
};

cudaError_t write_kv_launch(const WriteArgs& args, cudaStream_t stream);
cudaError_t copy_blocks_launch(const CopyArgs& args, cudaStream_t stream);
cudaError_t swap_blocks_launch(const SwapArgs& args, cudaStream_t stream);
cudaError_t write_kv_layers_launch(const WriteLayersArgs& args, cudaStream_t stream);
cudaError_t apply_table_deltas_launch(const DeltaArgs& args, cudaStream_t stream);
cudaError_t write_kv_fp8_launch(const WriteFp8Args& args, cudaStream_t stream);

}  // namespace pa
