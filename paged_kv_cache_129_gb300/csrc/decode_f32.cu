// Decode kernels for fp32 caches: explicit instantiations and dispatch.
#include "decode_kernel.cuh"

namespace pa {
namespace {

using T = float;

template <typename F>
bool dispatch(int d, int bs, int kind, int gmax, F&& f) {
    if (kind == 2) {
        if (d == 64 && bs == 16 && gmax == 1) return f(DecodeKernel<T, 64, 16, false, 1, false>{}), true;
        if (d == 64 && bs == 16 && gmax == 2) return f(DecodeKernel<T, 64, 16, false, 2, false>{}), true;
        if (d == 64 && bs == 16 && gmax == 4) return f(DecodeKernel<T, 64, 16, false, 4, false>{}), true;
        if (d == 64 && bs == 16 && gmax == 8) return f(DecodeKernel<T, 64, 16, false, 8, false>{}), true;
        if (d == 64 && bs == 32 && gmax == 1) return f(DecodeKernel<T, 64, 32, false, 1, false>{}), true;
        if (d == 64 && bs == 32 && gmax == 2) return f(DecodeKernel<T, 64, 32, false, 2, false>{}), true;
        if (d == 64 && bs == 32 && gmax == 4) return f(DecodeKernel<T, 64, 32, false, 4, false>{}), true;
        if (d == 64 && bs == 32 && gmax == 8) return f(DecodeKernel<T, 64, 32, false, 8, false>{}), true;
        if (d == 128 && bs == 16 && gmax == 1) return f(DecodeKernel<T, 128, 16, false, 1, false>{}), true;
        if (d == 128 && bs == 16 && gmax == 2) return f(DecodeKernel<T, 128, 16, false, 2, false>{}), true;
        if (d == 128 && bs == 16 && gmax == 4) return f(DecodeKernel<T, 128, 16, false, 4, false>{}), true;
        if (d == 128 && bs == 16 && gmax == 8) return f(DecodeKernel<T, 128, 16, false, 8, false>{}), true;
        if (d == 128 && bs == 32 && gmax == 1) return f(DecodeKernel<T, 128, 32, false, 1, false>{}), true;
        if (d == 128 && bs == 32 && gmax == 2) return f(DecodeKernel<T, 128, 32, false, 2, false>{}), true;
        if (d == 128 && bs == 32 && gmax == 4) return f(DecodeKernel<T, 128, 32, false, 4, false>{}), true;
        if (d == 128 && bs == 32 && gmax == 8) return f(DecodeKernel<T, 128, 32, false, 8, false>{}), true;
    }
    return false;
}

}  // namespace

bool decode_kernel_info_f32(int head_dim, int block_size, int kind, int gmax, int num_seqs, KernelInfo* info) {
    bool ok = false;
    const bool found =
        dispatch(head_dim, block_size, kind, gmax, [&](auto k) { ok = decltype(k)::info(num_seqs, info); });
    return found && ok;
}

cudaError_t decode_launch_f32(int head_dim, int block_size, int kind, int gmax, int schedule,
                              const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, const DecodeArgs& args,
                              int grid, int num_seqs, cudaStream_t stream) {
    cudaError_t err = cudaErrorInvalidValue;
    dispatch(head_dim, block_size, kind, gmax, [&](auto k) {
        err = decltype(k)::launch(schedule, tmap_k, tmap_v, args, grid, num_seqs, stream);
    });
    return err;
}

cudaError_t merge_launch_f32(int head_dim, const MergeArgs& args, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_merge<T, 64>(args, stream);
        case 128: return launch_merge<T, 128>(args, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
