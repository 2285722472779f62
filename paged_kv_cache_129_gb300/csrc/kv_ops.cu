// Cache-maintenance kernels: the paged KV write (reshape-and-cache), the
// copy-on-write block copy and the swap copy between two pools.  All move raw
// bytes, so they are bit-exact for every element type.
#include <algorithm>
#include <cstdint>

#include <cuda_fp8.h>

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

// The write of every layer in one launch: grid.y = layer, then as write_kv_kernel.  The
// pointers of all layers travel in the kernel's parameter block.
template <typename V>
__global__ void __launch_bounds__(256) write_kv_layers_kernel(const LayerPtrs layers, const int64_t* __restrict__ slots,
                                                              int num_tokens, int num_kv_heads, int row_vecs,
                                                              int block_size, long long num_slots, unsigned* err) {
    griddep_wait();
    griddep_launch_dependents();
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= (long long)num_tokens * num_kv_heads) return;
    const int layer = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int t = (int)(gw / num_kv_heads);
    const int h = (int)(gw - (long long)t * num_kv_heads);
    const long long slot = __ldg(slots + t);
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && h == 0 && layer == 0) atomicOr(err, kErrBadSlot);
        return;
    }
    const V* key = static_cast<const V*>(layers.key[layer]);
    const V* value = static_cast<const V*>(layers.value[layer]);
    V* key_cache = static_cast<V*>(layers.key_cache[layer]);
    V* value_cache = static_cast<V*>(layers.value_cache[layer]);
    const long long blk = slot / block_size;
    const long long off = slot - blk * block_size;
    const size_t src = ((size_t)t * num_kv_heads + h) * row_vecs;
    const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) {
        key_cache[dst + i] = __ldg(key + src + i);
        value_cache[dst + i] = __ldg(value + src + i);
    }
}

// Paged write into an FP8 (E4M3) cache: one warp per (token, kv head); element i of the row
// becomes e4m3(x / scale[block, head]) (the division in float32, round to nearest even,
// saturating to +-448, NaN kept), four elements per lane and step.
template <typename S>
__global__ void __launch_bounds__(256) write_kv_fp8_kernel(const S* __restrict__ key, const S* __restrict__ value,
                                                           uint8_t* __restrict__ key_cache,
                                                           uint8_t* __restrict__ value_cache,
                                                           const float* __restrict__ k_scale,
                                                           const float* __restrict__ v_scale,
                                                           const int64_t* __restrict__ slots, int num_tokens,
                                                           int num_kv_heads, int head_dim, int block_size,
                                                           long long num_slots, int interleaved, unsigned* err) {
    griddep_wait();
    griddep_launch_dependents();
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= (long long)num_tokens * num_kv_heads) return;
    const int lane = threadIdx.x & 31;
    const int t = (int)(gw / num_kv_heads);
    const int h = (int)(gw - (long long)t * num_kv_heads);
    const long long slot = __ldg(slots + t);
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && h == 0) atomicOr(err, kErrBadSlot);
        return;
    }
    const long long blk = slot / block_size;
    const long long off = slot - blk * block_size;
    const float ks = __ldg(k_scale + blk * num_kv_heads + h);
    const float vs = __ldg(v_scale + blk * num_kv_heads + h);
    const size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
    // separate caches: row (blk, h, off) of each; interleaved ([N, H_kv, 2, bs, d] in key_cache):
    // the K row, and the V row bs rows further
    const size_t rec = (size_t)blk * num_kv_heads + h;
    const size_t dst = interleaved ? (rec * 2 * block_size + off) * head_dim : (rec * block_size + off) * head_dim;
    const size_t dst_v = interleaved ? dst + (size_t)block_size * head_dim : dst;
    for (int i = 4 * lane; i < head_dim; i += 128) {
        float xk[4], xv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            xk[e] = to_float(key[src + i + e]) / ks;
            xv[e] = to_float(value[src + i + e]) / vs;
        }
        const uint32_t ck = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(xk[0], xk[1]), __NV_SATFINITE, __NV_E4M3) |
                            ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(xk[2], xk[3]), __NV_SATFINITE, __NV_E4M3)
                             << 16);
        const uint32_t cv = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(xv[0], xv[1]), __NV_SATFINITE, __NV_E4M3) |
                            ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(xv[2], xv[3]), __NV_SATFINITE, __NV_E4M3)
                             << 16);
        *reinterpret_cast<uint32_t*>(key_cache + dst + i) = ck;
        *reinterpret_cast<uint32_t*>(value_cache + dst_v + i) = cv;
    }
}

// One thread per (row, logical block, physical block) delta of a block table.
__global__ void __launch_bounds__(256) apply_table_deltas_kernel(int32_t* __restrict__ tables, int num_rows,
                                                                 int max_blocks, const int32_t* deltas,
                                                                 int num_deltas, unsigned* err) {
    griddep_wait();
    griddep_launch_dependents();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= num_deltas) return;
    // the deltas may live in host memory: plain loads
    const int row = deltas[3 * i];
    const int j = deltas[3 * i + 1];
    const int block = deltas[3 * i + 2];
    if (row < 0 || row >= num_rows || j < 0 || j >= max_blocks) {
        atomicOr(err, kErrBadTable);
        return;
    }
    tables[(size_t)row * max_blocks + j] = block;
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

// Swap copy between two pools.  Work unit (pair, cache, chunk): kSwapUnroll * 256 vectors of
// one block, all loads of a thread issued before its stores, so that enough requests are in
// flight to cover the latency of host memory on the other side of the link.  The grid is
// capped at kSwapCtasPerSm per SM and strides over the units, so that a swap-out and a
// swap-in launched on two streams are resident together and use both directions of the link.
constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;
constexpr int kSwapCtasPerSm = 3;

template <typename V>
__global__ void __launch_bounds__(kSwapThreads) swap_blocks_kernel(V* dst_key, V* dst_value, const V* src_key,
                                                                   const V* src_value, const int64_t* pairs,
                                                                   long long block_vecs, int chunks, long long units,
                                                                   int src_blocks, int dst_blocks, int caches,
                                                                   unsigned* err) {
    griddep_wait();
    griddep_launch_dependents();
    for (long long u0 = blockIdx.x; u0 < units; u0 += gridDim.x) {
        const int chunk = (int)(u0 % chunks);
        const long long pc = u0 / chunks;
        const int cache = (int)(pc % caches);  // caches: 2 (K, V) or 1 (one cache)
        const long long pidx = pc / caches;
        // the pairs may live in host memory: plain loads
        const long long src = pairs[2 * pidx];
        const long long dst = pairs[2 * pidx + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
            if (threadIdx.x == 0 && chunk == 0 && cache == 0) atomicOr(err, kErrBadTable);
            continue;
        }
        const V* s = (cache ? src_value : src_key) + src * block_vecs;
        V* d = (cache ? dst_value : dst_key) + dst * block_vecs;
        const long long base = (long long)chunk * kSwapThreads * kSwapUnroll + threadIdx.x;
        V r[kSwapUnroll];
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const long long i = base + (long long)u * kSwapThreads;
            if (i < block_vecs) r[u] = s[i];
        }
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const long long i = base + (long long)u * kSwapThreads;
            if (i < block_vecs) d[i] = r[u];
        }
    }
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
    dim3 grid((unsigned)a.num_pairs, a.single ? 1u : 2u, (unsigned)chunks);
    return launch_pdl(copy_blocks_kernel<V>, grid, dim3(threads), 0, stream, static_cast<V*>(a.key_cache),
                      static_cast<V*>(a.value_cache), a.pairs, block_vecs, a.num_blocks, a.err);
}

template <typename V>
cudaError_t swap_typed(const SwapArgs& a, long long block_bytes, cudaStream_t stream) {
    const long long block_vecs = block_bytes / (long long)sizeof(V);
    const long long per_cta = (long long)kSwapThreads * kSwapUnroll;
    const long long chunks = (block_vecs + per_cta - 1) / per_cta;
    if (chunks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int caches = a.single ? 1 : 2;
    const long long units = (long long)a.num_pairs * caches * chunks;
    const long long grid = std::min<long long>(units, (long long)kSwapCtasPerSm * std::max(a.num_sms, 1));
    return launch_pdl(swap_blocks_kernel<V>, dim3((unsigned)grid), dim3(kSwapThreads), 0, stream,
                      static_cast<V*>(a.dst_key), static_cast<V*>(a.dst_value), static_cast<const V*>(a.src_key),
                      static_cast<const V*>(a.src_value), a.pairs, block_vecs, (int)chunks, units, a.src_num_blocks,
                      a.dst_num_blocks, caches, a.err);
}

template <typename V>
cudaError_t write_layers_typed(const WriteLayersArgs& a, long long row_bytes, cudaStream_t stream) {
    const int row_vecs = (int)(row_bytes / sizeof(V));
    const long long warps = (long long)a.num_tokens * a.num_kv_heads;
    const int threads = 256;
    const long long grid = (warps + (threads / 32) - 1) / (threads / 32);
    return launch_pdl(write_kv_layers_kernel<V>, dim3((unsigned)grid, (unsigned)a.num_layers), dim3(threads), 0,
                      stream, *a.layers, a.slot_mapping, a.num_tokens, a.num_kv_heads, row_vecs, a.block_size,
                      (long long)a.num_blocks * a.block_size, a.err);
}

}  // namespace

cudaError_t write_kv_layers_launch(const WriteLayersArgs& a, cudaStream_t stream) {
    const long long row_bytes = (long long)a.head_dim * a.elem_bytes;
    int v = 16;
    for (int l = 0; l < a.num_layers; ++l) {
        const void* ptrs[4] = {a.layers->key[l], a.layers->value[l], a.layers->key_cache[l], a.layers->value_cache[l]};
        v = std::min(v, vector_bytes(row_bytes, ptrs, 4));
    }
    switch (v) {
        case 16: return write_layers_typed<uint4>(a, row_bytes, stream);
        case 8: return write_layers_typed<uint2>(a, row_bytes, stream);
        case 4: return write_layers_typed<uint32_t>(a, row_bytes, stream);
        case 2: return write_layers_typed<uint16_t>(a, row_bytes, stream);
        default: return write_layers_typed<uint8_t>(a, row_bytes, stream);
    }
}

cudaError_t write_kv_fp8_launch(const WriteFp8Args& a, cudaStream_t stream) {
    const long long warps = (long long)a.num_tokens * a.num_kv_heads;
    const int threads = 256;
    const long long grid = (warps + (threads / 32) - 1) / (threads / 32);
    const long long num_slots = (long long)a.num_blocks * a.block_size;
    const int interleaved = a.value_cache == nullptr ? 1 : 0;
    uint8_t* vc = interleaved ? a.key_cache : a.value_cache;
    switch (a.src_dtype) {
        case 0:
            return launch_pdl(write_kv_fp8_kernel<float>, dim3((unsigned)grid), dim3(threads), 0, stream,
                              static_cast<const float*>(a.key), static_cast<const float*>(a.value), a.key_cache,
                              vc, a.k_scale, a.v_scale, a.slot_mapping, a.num_tokens, a.num_kv_heads,
                              a.head_dim, a.block_size, num_slots, interleaved, a.err);
        case 1:
            return launch_pdl(write_kv_fp8_kernel<__half>, dim3((unsigned)grid), dim3(threads), 0, stream,
                              static_cast<const __half*>(a.key), static_cast<const __half*>(a.value), a.key_cache,
                              vc, a.k_scale, a.v_scale, a.slot_mapping, a.num_tokens, a.num_kv_heads,
                              a.head_dim, a.block_size, num_slots, interleaved, a.err);
        case 2:
            return launch_pdl(write_kv_fp8_kernel<__nv_bfloat16>, dim3((unsigned)grid), dim3(threads), 0, stream,
                              static_cast<const __nv_bfloat16*>(a.key), static_cast<const __nv_bfloat16*>(a.value),
                              a.key_cache, vc, a.k_scale, a.v_scale, a.slot_mapping, a.num_tokens,
                              a.num_kv_heads, a.head_dim, a.block_size, num_slots, interleaved, a.err);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t apply_table_deltas_launch(const DeltaArgs& a, cudaStream_t stream) {
    const int threads = 256;
    const int grid = (a.num_deltas + threads - 1) / threads;
    return launch_pdl(apply_table_deltas_kernel, dim3((unsigned)grid), dim3(threads), 0, stream, a.block_tables,
                      a.num_rows, a.max_blocks, a.deltas, a.num_deltas, a.err);
}

cudaError_t swap_blocks_launch(const SwapArgs& a, cudaStream_t stream) {
    const long long block_bytes = (long long)a.num_kv_heads * a.block_size * a.head_dim * a.elem_bytes;
    const void* ptrs[4] = {a.dst_key, a.dst_value, a.src_key, a.src_value};
    switch (vector_bytes(block_bytes, ptrs, 4)) {
        case 16: return swap_typed<uint4>(a, block_bytes, stream);
        case 8: return swap_typed<uint2>(a, block_bytes, stream);
        case 4: return swap_typed<uint32_t>(a, block_bytes, stream);
        case 2: return swap_typed<uint16_t>(a, block_bytes, stream);
        default: return swap_typed<uint8_t>(a, block_bytes, stream);
    }
}

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
