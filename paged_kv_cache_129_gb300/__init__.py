"""Paged decode attention (PagedAttention) for GB300, behind a C ABI.

The compute path is the CUDA library built from ``csrc/`` (see
``include/pa.h``); this package only marshals torch tensors into it.
"""
from .binding import (  # noqa: F401
    KERNELS,
    STATIC_SCRATCH_BYTES,
    LIB_PATH,
    BlockPool,
    apply_table_deltas,
    DecodePlan,
    PAError,
    PoolExhausted,
    check_error,
    copy_blocks,
    decode,
    decode_append,
    decode_fp8,
    decode_fp8_append,
    decode_fp8_workspace_size,
    decode_multi,
    decode_multi_workspace_size,
    decode_plan,
    decode_static_scratch,
    decode_workspace_size,
    diag_force_restart,
    diag_merge_timeout,
    library,
    swap_blocks,
    version,
    write_kv,
    write_kv_fp8,
    write_kv_layers,
)


from .step import DecodeStepper  # noqa: F401,E402


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from .native_build import build as _build

    return _build(force=force)
