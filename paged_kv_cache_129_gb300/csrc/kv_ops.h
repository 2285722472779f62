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
    unsigned* err;
};

cudaError_t write_kv_launch(const WriteArgs& args, cudaStream_t stream);
cudaError_t copy_blocks_launch(const CopyArgs& args, cudaStream_t stream);

}  // namespace pa
