// Decode kernels for FP8 (E4M3) caches: explicit instantiations and dispatch by the
// query/output type, head_dim and block size.
#include "decode_kernel.cuh"
#include "pa.h"

namespace pa {
namespace {

template <typename F>
bool dispatch(int dtype, int d, int bs, F&& f) {
    if (d != 128) return false;
    if (dtype == PA_BF16 && bs == 16) return f(DecodeKernelF8<__nv_bfloat16, 128, 16>{}), true;
    if (dtype == PA_BF16 && bs == 32) return f(DecodeKernelF8<__nv_bfloat16, 128, 32>{}), true;
    if (dtype == PA_F16 && bs == 16) return f(DecodeKernelF8<__half, 128, 16>{}), true;
    if (dtype == PA_F16 && bs == 32) return f(DecodeKernelF8<__half, 128, 32>{}), true;
    return false;
}

}  // namespace

bool decode_kernel_info_fp8(int dtype, int head_dim, int block_size, int num_seqs, KernelInfo* info) {
    bool ok = false;
    const bool found = dispatch(dtype, head_dim, block_size, [&](auto k) { ok = decltype(k)::info(num_seqs, info); });
    return found && ok;
}

cudaError_t decode_launch_fp8(int dtype, int head_dim, int block_size, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, const DecodeArgs& args, int grid, int num_seqs,
                              cudaStream_t stream) {
    cudaError_t err = cudaErrorInvalidValue;
    dispatch(dtype, head_dim, block_size,
             [&](auto k) { err = decltype(k)::launch(tmap_k, tmap_v, args, grid, num_seqs, stream); });
    return err;
}

}  // namespace pa
