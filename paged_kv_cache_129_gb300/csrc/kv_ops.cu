// Cache-maintenance kernels: the paged KV write (reshape-and-cache) and the
// copy-on-write block copy.  Both move raw bytes, so they are bit-exact for
// every element type.
#include <cstdint>

#include "kv_ops.h"
#include "pa_common.cuh"

namespace pa {

// One warp per (token, kv head): the token's row goes to
// cache[slot / bs, h, slot % bs, :] (MiniPaged-Qwen, sections 8.1-8.2).
template <typename V>
__global__ void __launch_bounds__(256) write_kv_kernel(const V* __restrict__ key, const V* __restrict__ value,
                                                       V* __restrict__ key_cache, V* __restrict__ value_cache,
                                                       const int64_t* __restrict__ slots, int num_tokens,
                                                       int num_kv_heads, int row_vecs, int block_size,
                                                       long long num_slots, unsigned* err) {
    griddep_wait();
    griddep_launch_dependents();
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= (long long)num_tokens * num_kv_heads) return;
    const int lane = threadIdx.x & 31;
    const int t = (int)(gw / num_kv_heads);
    const int h = (int)(gw - (long long)t * num_kv_heads);
    const long long slot = __ldg(slots + t);
    if (slot < 0) return;  // padding token: nothing to write
    if (slot >= num_slots) {
        if (lane == 0 && h == 0) atomicOr(err, kErrBadSlot);
        return;
    }
    const long long blk = slot / block_size;
    const long long off = slot - blk * block_size;
    const size_t src = ((size_t)t * num_kv_heads + h) * row_vecs;
    const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) {
        key_cache[dst + i] = __ldg(key + src + i);
        value_cache[dst + i] = __ldg(value + src + i);
    }
}

// Grid (pair, cache, chunk): block dst of one cache becomes a copy of block src.
template <typename V>
__global__ void __launch_bounds__(256) copy_blocks_kernel(V* key_cache, V* value_cache, const int64_t* __restrict__ pairs,
                                                          long long block_vecs, int num_blocks, unsigned* err) {
    griddep_wait();
    griddep_launch_dependents();
    const int pidx = blockIdx.x;
    const long long src = __ldg(pairs + 2 * pidx);
    const long long dst = __ldg(pairs + 2 * pidx + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(err, kErrBadTable);
        return;
    }
    V* cache = blockIdx.y == 0 ? key_cache : value_cache;
    const V* s = cache + src * block_vecs;
    V* d = cache + dst * block_vecs;
    const long long stride = (long long)gridDim.z * blockDim.x;
    for (long long i = (long long)blockIdx.z * blockDim.x + threadIdx.x; i < block_vecs; i += stride) d[i] = s[i];
}

namespace {

// Widest unit (16, 8, 4, 2 or 1 bytes) that divides `bytes` and the alignment of every pointer.
int vector_bytes(long long bytes, const void* const* ptrs, int n) {
    int v = 16;
    while (v > 1) {
        bool ok = bytes % v == 0;
        for (int i = 0; i < n && ok; ++i) ok = (reinterpret_cast<uintptr_t>(ptrs[i]) % v) == 0;
        if (ok) break;
        v >>= 1;
    }
    return v;
}

template <typename V>
cudaError_t write_typed(const WriteArgs& a, long long row_bytes, cudaStream_t stream) {
    const int row_vecs = (int)(row_bytes / sizeof(V));
    const long long warps = (long long)a.num_tokens * a.num_kv_heads;
    const int threads = 256;
    const long long grid = (warps + (threads / 32) - 1) / (threads / 32);
    return launch_pdl(write_kv_kernel<V>, dim3((unsigned)grid), dim3(threads), 0, stream, static_cast<const V*>(a.key),
                      static_cast<const V*>(a.value), static_cast<V*>(a.key_cache), static_cast<V*>(a.value_cache),
                      a.slot_mapping, a.num_tokens, a.num_kv_heads, row_vecs, a.block_size,
                      (long long)a.num_blocks * a.block_size, a.err);
}

template <typename V>
cudaError_t copy_typed(const CopyArgs& a, long long block_bytes, cudaStream_t stream) {
    const long long block_vecs = block_bytes / (long long)sizeof(V);
    const int threads = 256;
    long long chunks = (block_vecs + threads * 4 - 1) / (threads * 4);
    if (chunks > 65535) chunks = 65535;
    dim3 grid((unsigned)a.num_pairs, 2, (unsigned)chunks);
    return launch_pdl(copy_blocks_kernel<V>, grid, dim3(threads), 0, stream, static_cast<V*>(a.key_cache),
                      static_cast<V*>(a.value_cache), a.pairs, block_vecs, a.num_blocks, a.err);
}

}  // namespace

cudaError_t write_kv_launch(const WriteArgs& a, cudaStream_t stream) {
    const long long row_bytes = (long long)a.head_dim * a.elem_bytes;
    const void* ptrs[4] = {a.key, a.value, a.key_cache, a.value_cache};
    switch (vector_bytes(row_bytes, ptrs, 4)) {
        case 16: return write_typed<uint4>(a, row_bytes, stream);
        case 8: return write_typed<uint2>(a, row_bytes, stream);
        case 4: return write_typed<uint32_t>(a, row_bytes, stream);
        case 2: return write_typed<uint16_t>(a, row_bytes, stream);
        default: return write_typed<uint8_t>(a, row_bytes, stream);
    }
}

cudaError_t copy_blocks_launch(const CopyArgs& a, cudaStream_t stream) {
    const long long block_bytes = (long long)a.num_kv_heads * a.block_size * a.head_dim * a.elem_bytes;
    const void* ptrs[2] = {a.key_cache, a.value_cache};
    switch (vector_bytes(block_bytes, ptrs, 2)) {
        case 16: return copy_typed<uint4>(a, block_bytes, stream);
        case 8: return copy_typed<uint2>(a, block_bytes, stream);
        case 4: return copy_typed<uint32_t>(a, block_bytes, stream);
        case 2: return copy_typed<uint16_t>(a, block_bytes, stream);
        default: return copy_typed<uint8_t>(a, block_bytes, stream);
    }
}

}  // namespace pa
