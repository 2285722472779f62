"""Thin ctypes binding of the C ABI in ``include/pa.h``.

Argument marshalling only: every step of the path runs in the CUDA library
(``_build/libpagedkv.so``).  PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpagedkv.so")

PA_OK = 0
STATUS_NAMES = {
    0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA", 4: "PA_ERR_POOL_EXHAUSTED",
    5: "PA_ERR_BAD_TABLE", 6: "PA_ERR_BAD_SLOT", 7: "PA_ERR_BAD_CONTEXT", 8: "PA_ERR_TIMEOUT", 9: "PA_ERR_NOT_FOUND",
}
PA_F32, PA_F16, PA_BF16 = 0, 1, 2
KERNELS = {"auto": 0, "mma": 1, "simt": 2}
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024  # PA_STATIC_SCRATCH_BYTES
PA_E4M3 = 3  # one-byte FP8 codes (byte movers)
_TORCH_DTYPES = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class PAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class PoolExhausted(PAError, MemoryError):
    pass


STEP_DECODE, STEP_APPEND, STEP_FP8, STEP_FP8_WRITE, STEP_FP8_APPEND = 0, 1, 2, 3, 4


class StepCall(ctypes.Structure):
    """``pa_step_call``: the decode call of one step-runner slot."""
    _fields_ = [("kind", ctypes.c_int), ("out", ctypes.c_void_p), ("query", ctypes.c_void_p),
                ("new_key", ctypes.c_void_p), ("new_value", ctypes.c_void_p), ("slots", ctypes.c_void_p),
                ("key_cache", ctypes.c_void_p), ("value_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
                ("deltas", ctypes.c_void_p), ("num_seqs", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("num_blocks", ctypes.c_int), ("scale", ctypes.c_float),
                ("dtype", ctypes.c_int), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("max_context_len", ctypes.c_int), ("partition_pages", ctypes.c_int), ("kernel", ctypes.c_int)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("schedule", ctypes.c_int), ("partition_pages", ctypes.c_int),
                ("max_parts", ctypes.c_int),
                ("heads_per_cta", ctypes.c_int), ("grid_ctas", ctypes.c_int), ("threads_per_cta", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


# (name, restype, argtypes) of every exported function.
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_SIGNATURES = [
    ("pa_last_error_string", ctypes.c_char_p, []),
    ("pa_version", ctypes.c_char_p, []),
    ("pa_check_error", _I, [_P]),
    ("pa_write_kv", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    ("pa_copy_blocks", _I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    ("pa_swap_blocks", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    ("pa_write_kv_fp8", _I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    ("pa_decode_fp8", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    ("pa_decode_fp8_append", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P,
                                  _SZ, _P]),
    ("pa_decode_fp8_workspace_size", _SZ, [_I, _I, _I, _I, _I, _I, _I]),
    ("pa_write_kv_layers", _I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P]),
    ("pa_apply_table_deltas", _I, [_P, _I, _I, _P, _I, _P]),
    ("pa_decode", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    ("pa_decode_ex", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _I, _I, _I, _P]),
    ("pa_decode_append", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _I, _I, _I,
                              _P]),
    ("pa_decode_multi", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _I, _I, _I, _P]),
    ("pa_decode_multi_workspace_size", _SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    ("pa_decode_multi_make_plan", _I, [_I, _I, _I, _I, _I, _I, _I, _I, _SZ, _I, _I, _I, ctypes.POINTER(DecodePlan)]),
    ("pa_decode_make_plan", _I, [_I, _I, _I, _I, _I, _I, _I, _SZ, _I, _I, _I, ctypes.POINTER(DecodePlan)]),
    ("pa_decode_workspace_size", _SZ, [_I, _I, _I, _I, _I, _I, _I]),
    ("pa_decode_static_scratch", _I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    ("pa_diag_force_restart", None, [_I]),
    ("pa_diag_merge_timeout", _I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _SZ, ctypes.c_ulonglong, _P]),
    ("pa_stepper_create", _I, [_I, _P, _P, _P, ctypes.POINTER(_P)]),
    ("pa_stepper_destroy", None, [_P]),
    ("pa_stepper_set_slot", _I, [_P, _I, _P, _P, _SZ, _P, _P, _SZ]),
    ("pa_stepper_set_call", _I, [_P, _I, _P]),
    ("pa_stepper_launch", _I, [_P, _I, _SZ, _I]),
    ("pa_stepper_wait", _I, [_P, _I]),
    ("pa_pool_create", _I, [_I, _I, _P, ctypes.POINTER(_P)]),
    ("pa_pool_destroy", None, [_P]),
    ("pa_seq_create", _I, [_P, ctypes.POINTER(_I64)]),
    ("pa_seq_append", _I, [_P, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    ("pa_seq_append_batch", _I, [_P, _P, _I, _P, _P, ctypes.POINTER(_I)]),
    ("pa_seq_fork", _I, [_P, _I64, ctypes.POINTER(_I64)]),
    ("pa_seq_release", _I, [_P, _I64]),
    ("pa_seq_length", _I, [_P, _I64, ctypes.POINTER(_I64)]),
    ("pa_pool_blocks_needed", _I, [_P, _P, _P, _I, ctypes.POINTER(_I64)]),
    ("pa_seq_swap", _I, [_P, _P, _I64, ctypes.POINTER(_I64), _P, _I, ctypes.POINTER(_I)]),
    ("pa_pool_block_tables", _I, [_P, _P, _I, _P, _I, _P]),
    ("pa_pool_table_deltas", _I, [_P, _P, _I, _P, _I, ctypes.POINTER(_I), _P]),
    ("pa_pool_num_free", _I, [_P]),
    ("pa_pool_num_blocks", _I, [_P]),
    ("pa_pool_block_size", _I, [_P]),
    ("pa_pool_refcount", _I, [_P, ctypes.c_int32]),
    ("pa_pool_check_invariants", _I, [_P]),
    ("pa_pool_free_list", _I, [_P, _P, _I]),
    ("pa_pool_state_size", _SZ, [_P]),
    ("pa_pool_save", _I, [_P, _P, _SZ, ctypes.POINTER(_SZ)]),
    ("pa_pool_load", _I, [_P, _SZ, ctypes.POINTER(_P)]),
]


def library() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing (run __graft_entry__.build())")
            lib = ctypes.CDLL(LIB_PATH)
            for name, res, args in _SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def _check(status: int) -> None:
    if status != PA_OK:
        msg = library().pa_last_error_string()
        msg = msg.decode() if msg else ""
        if status == 4:
            raise PoolExhausted(status, msg)
        raise PAError(status, msg)


def _stream_ptr(stream, device: torch.device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _TORCH_DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _need(cond: bool, what: str) -> None:
    if not cond:
        raise ValueError(what)


def _cuda(t: torch.Tensor, name: str) -> None:
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.is_contiguous(), f"{name} must be contiguous")


def diag_merge_timeout(out: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int, block_size: int,
                       max_blocks_per_seq: int, workspace: torch.Tensor, wait_limit_ns: int, stream=None) -> None:
    """``pa_diag_merge_timeout``: the lean merge alone, waiting for records no decode publishes, so that
    its bounded wait runs out after ``wait_limit_ns`` (the device error word then reports a timeout)."""
    for name, t in (("out", out), ("context_lens", context_lens), ("workspace", workspace)):
        _cuda(t, name)
    _need(out.dim() == 3, "out must be [B, H_q, d]")
    b, hq, d = out.shape
    _check(library().pa_diag_merge_timeout(out.data_ptr(), context_lens.data_ptr(), b, hq, num_kv_heads, d, block_size,
                                           max_blocks_per_seq, _dtype_code(out), workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(), int(wait_limit_ns),
                                           _stream_ptr(stream, out.device)))


def diag_force_restart(on: bool) -> None:
    """``pa_diag_force_restart``: make every later lean decode redo its early set-up (tests only)."""
    library().pa_diag_force_restart(1 if on else 0)


def version() -> str:
    return library().pa_version().decode()


def check_error(stream=None, device=None) -> None:
    """Synchronise the stream and raise if a kernel flagged bad data since the last check."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(library().pa_check_error(_stream_ptr(stream, dev)))


def write_kv(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
             slot_mapping: torch.Tensor, stream=None) -> None:
    """``pa_write_kv``: scatter key/value ``[T, H_kv, d]`` into the caches at ``slot_mapping`` (int64)."""
    for name, t in (("key", key), ("value", value), ("key_cache", key_cache), ("value_cache", value_cache),
                    ("slot_mapping", slot_mapping)):
        _cuda(t, name)
    _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape, "caches must be [N, H_kv, bs, d]")
    num_blocks, hkv, bs, d = key_cache.shape
    _need(key.shape == value.shape and key.dim() == 3 and key.shape[1:] == (hkv, d), "key/value must be [T, H_kv, d]")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == key.shape[0], "slot_mapping: int64 [T]")
    _need(key.dtype == value.dtype == key_cache.dtype == value_cache.dtype, "dtypes must match")
    _check(library().pa_write_kv(key.data_ptr(), value.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(),
                                 slot_mapping.data_ptr(), key.shape[0], hkv, d, bs, num_blocks,
                                 _dtype_code(key_cache), _stream_ptr(stream, key_cache.device)))


def _block_geometry(key_cache: torch.Tensor, value_cache: Optional[torch.Tensor]):
    """(num_blocks, H_kv, bs, d, element code) of a cache pair, or of one interleaved FP8 cache
    ``[N, H_kv, 2, bs, d]`` when ``value_cache`` is None."""
    if value_cache is None:
        _need(key_cache.dim() == 5 and key_cache.shape[2] == 2, "one cache: interleaved FP8 [N, H_kv, 2, bs, d]")
        n, h, _, bs, d = key_cache.shape
    else:
        _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape and value_cache.dtype == key_cache.dtype,
              "caches must be [N, H_kv, bs, d] of one dtype")
        n, h, bs, d = key_cache.shape
    code = PA_E4M3 if key_cache.dtype in (torch.uint8, torch.float8_e4m3fn) else _dtype_code(key_cache)
    return n, h, bs, d, code


def copy_blocks(key_cache: torch.Tensor, value_cache: Optional[torch.Tensor], src_dst_pairs: torch.Tensor,
                stream=None) -> None:
    """``pa_copy_blocks``: for each (src, dst) row of ``src_dst_pairs`` (int64 [n, 2]) copy block src -> dst
    (``value_cache`` None: one interleaved FP8 cache, whole records)."""
    for name, t in (("key_cache", key_cache), ("src_dst_pairs", src_dst_pairs)) + (
            (("value_cache", value_cache),) if value_cache is not None else ()):
        _cuda(t, name)
    _need(src_dst_pairs.dtype == torch.int64 and (src_dst_pairs.numel() % 2 == 0), "pairs: int64 [n, 2]")
    num_blocks, hkv, bs, d, code = _block_geometry(key_cache, value_cache)
    _check(library().pa_copy_blocks(key_cache.data_ptr(), value_cache.data_ptr() if value_cache is not None else None,
                                    src_dst_pairs.data_ptr(), src_dst_pairs.numel() // 2, hkv, d, bs, num_blocks,
                                    code, _stream_ptr(stream, key_cache.device)))


def write_kv_layers(keys, values, key_caches, value_caches, slot_mapping: torch.Tensor, stream=None) -> None:
    """``pa_write_kv_layers``: ``pa_write_kv`` for every layer in one launch.  ``keys`` / ``values`` are
    sequences of per-layer ``[T, H_kv, d]`` tensors, ``key_caches`` / ``value_caches`` of per-layer
    ``[N, H_kv, bs, d]`` caches; ``slot_mapping`` (int64 [T]) is shared by all layers."""
    n = len(keys)
    _need(n >= 1 and len(values) == n and len(key_caches) == n and len(value_caches) == n,
          "one key, value, key cache and value cache per layer")
    _cuda(slot_mapping, "slot_mapping")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.dim() == 1, "slot_mapping: int64 [T]")
    kc0 = key_caches[0]
    _need(kc0.dim() == 4, "caches must be [N, H_kv, bs, d]")
    num_blocks, hkv, bs, d = kc0.shape
    for l in range(n):
        for name, t in (("key", keys[l]), ("value", values[l]), ("key_cache", key_caches[l]),
                        ("value_cache", value_caches[l])):
            _cuda(t, f"{name}[{l}]")
            _need(t.dtype == kc0.dtype, "dtypes must match")
        _need(key_caches[l].shape == kc0.shape and value_caches[l].shape == kc0.shape, "caches differ in shape")
        _need(keys[l].shape == values[l].shape == (slot_mapping.numel(), hkv, d), "key/value must be [T, H_kv, d]")
    arr = ctypes.c_void_p * n
    _check(library().pa_write_kv_layers(arr(*[t.data_ptr() for t in keys]), arr(*[t.data_ptr() for t in values]),
                                        arr(*[t.data_ptr() for t in key_caches]),
                                        arr(*[t.data_ptr() for t in value_caches]), n, slot_mapping.data_ptr(),
                                        slot_mapping.numel(), hkv, d, bs, num_blocks, _dtype_code(kc0),
                                        _stream_ptr(stream, kc0.device)))


def apply_table_deltas(block_tables: torch.Tensor, deltas: torch.Tensor, num_deltas: Optional[int] = None,
                       stream=None) -> None:
    """``pa_apply_table_deltas``: ``block_tables[row, j] = block`` for the first ``num_deltas`` (default all)
    (row, j, block) rows of ``deltas`` (int32 [n, 3], a CUDA tensor or pinned host memory)."""
    _cuda(block_tables, "block_tables")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2, "block_tables: int32 [rows, max_blocks]")
    _need(deltas.dtype == torch.int32 and deltas.is_contiguous() and deltas.numel() % 3 == 0, "deltas: int32 [n, 3]")
    _need(deltas.is_cuda or deltas.is_pinned(), "deltas must be a CUDA tensor or pinned host memory")
    n = deltas.numel() // 3 if num_deltas is None else int(num_deltas)
    _need(0 <= n <= deltas.numel() // 3, "num_deltas out of range")
    with torch.cuda.device(block_tables.device):
        _check(library().pa_apply_table_deltas(block_tables.data_ptr(), block_tables.shape[0], block_tables.shape[1],
                                               deltas.data_ptr(), n, _stream_ptr(stream, block_tables.device)))


def swap_blocks(dst_key_cache: torch.Tensor, dst_value_cache: Optional[torch.Tensor], src_key_cache: torch.Tensor,
                src_value_cache: Optional[torch.Tensor], block_pairs: torch.Tensor, stream=None) -> None:
    """``pa_swap_blocks``: block dst of the dst caches <- block src of the src caches for every (src, dst)
    row of ``block_pairs`` (int64 [n, 2]).  Each tensor is a CUDA tensor or a pinned CPU tensor
    (``pin_memory()``); the copy runs on the current CUDA device's stream."""
    _need((dst_value_cache is None) == (src_value_cache is None), "value caches: both or neither")
    tensors = tuple((n, t) for n, t in (("dst_key_cache", dst_key_cache), ("dst_value_cache", dst_value_cache),
                                        ("src_key_cache", src_key_cache), ("src_value_cache", src_value_cache),
                                        ("block_pairs", block_pairs)) if t is not None)
    for name, t in tensors:
        _need(t.is_contiguous(), f"{name} must be contiguous")
        _need(t.is_cuda or t.is_pinned(), f"{name} must be a CUDA tensor or pinned host memory")
    src_n, hkv, bs, d, code = _block_geometry(src_key_cache, src_value_cache)
    dst_n, *dst_geo = _block_geometry(dst_key_cache, dst_value_cache)
    _need(tuple(dst_geo) == (hkv, bs, d, code), "caches differ in block geometry or element type")
    _need(block_pairs.dtype == torch.int64 and block_pairs.numel() % 2 == 0, "block_pairs: int64 [n, 2]")
    cuda = [t.device for _, t in tensors if t.is_cuda]
    device = cuda[0] if cuda else torch.device("cuda", torch.cuda.current_device())

    def ptr(t):
        return t.data_ptr() if t is not None else None

    with torch.cuda.device(device):
        _check(library().pa_swap_blocks(ptr(dst_key_cache), ptr(dst_value_cache), ptr(src_key_cache),
                                        ptr(src_value_cache), block_pairs.data_ptr(), block_pairs.numel() // 2, hkv,
                                        d, bs, src_n, dst_n, code, _stream_ptr(stream, device)))


def decode_plan(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                max_blocks_per_seq: int, dtype: torch.dtype, workspace_bytes: int = 1 << 62,
                max_context_len: int = 0, partition_pages: int = 0, kernel: str = "auto",
                q_len: int = 1) -> DecodePlan:
    """The partition plan ``pa_decode_ex`` (``pa_decode_multi`` for q_len > 1) would use on the current device."""
    plan = DecodePlan()
    if q_len == 1:
        _check(library().pa_decode_make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                             max_blocks_per_seq, _TORCH_DTYPES[dtype], workspace_bytes,
                                             max_context_len, partition_pages, KERNELS[kernel], ctypes.byref(plan)))
    else:
        _check(library().pa_decode_multi_make_plan(num_seqs, q_len, num_heads, num_kv_heads, head_dim, block_size,
                                                   max_blocks_per_seq, _TORCH_DTYPES[dtype], workspace_bytes,
                                                   max_context_len, partition_pages, KERNELS[kernel],
                                                   ctypes.byref(plan)))
    return plan


def decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                          max_blocks_per_seq: int, dtype: torch.dtype) -> int:
    return int(library().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                  max_blocks_per_seq, _TORCH_DTYPES[dtype]))


def decode(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor, block_tables: torch.Tensor,
           context_lens: torch.Tensor, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None, max_context_len: int = 0, partition_pages: int = 0,
           kernel: str = "auto", stream=None) -> torch.Tensor:
    """``pa_decode_ex``: paged decode attention; returns ``out`` ``[B, H_q, d]``.

    ``workspace`` (any dtype, contiguous, on the same device) enables the
    split-KV partitions; ``None`` runs one partition per context.
    """
    for name, t in (("query", query), ("key_cache", key_cache), ("value_cache", value_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda(t, name)
    _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape, "caches must be [N, H_kv, bs, d]")
    num_blocks, hkv, bs, d = key_cache.shape
    _need(query.dim() == 3 and query.shape[2] == d, "query must be [B, H_q, d]")
    b, hq, _ = query.shape
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == b,
          "block_tables: int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == b, "context_lens: int32 [B]")
    _need(query.dtype == key_cache.dtype == value_cache.dtype, "query and caches must share a dtype")
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    _need(out.shape == query.shape and out.dtype == query.dtype, "out must match query")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        _cuda(workspace, "workspace")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(library().pa_decode_ex(out.data_ptr(), query.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(),
                                  block_tables.data_ptr(), context_lens.data_ptr(), b, hq, hkv, d, bs,
                                  block_tables.shape[1], num_blocks, float(scale), _dtype_code(query), ws_ptr or None,
                                  ws_bytes, max_context_len, partition_pages, KERNELS[kernel],
                                  _stream_ptr(stream, query.device)))
    return out


def _fp8_cache(key_cache: torch.Tensor, value_cache: Optional[torch.Tensor], k_scale: torch.Tensor,
               v_scale: torch.Tensor):
    """Checks FP8 caches; value_cache None means the interleaved layout [N, H_kv, 2, bs, d] in key_cache.
    Returns (num_blocks, H_kv, bs, d)."""
    for name, t in (("key_cache", key_cache), ("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda(t, name)
    _need(key_cache.dtype in (torch.uint8, torch.float8_e4m3fn), "FP8 caches hold E4M3 codes (uint8 or float8_e4m3fn)")
    if value_cache is None:
        _need(key_cache.dim() == 5 and key_cache.shape[2] == 2, "interleaved FP8 cache: [N, H_kv, 2, bs, d]")
        shape = (key_cache.shape[0], key_cache.shape[1], key_cache.shape[3], key_cache.shape[4])
    else:
        _cuda(value_cache, "value_cache")
        _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape, "caches must be [N, H_kv, bs, d]")
        _need(value_cache.dtype == key_cache.dtype, "caches must share a dtype")
        shape = tuple(key_cache.shape)
    _need(k_scale.dtype == v_scale.dtype == torch.float32 and k_scale.shape == v_scale.shape == shape[:2],
          "k_scale / v_scale: float32 [N, H_kv]")
    return shape


def write_kv_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: Optional[torch.Tensor],
                 k_scale: torch.Tensor, v_scale: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """``pa_write_kv_fp8``: quantise key/value ``[T, H_kv, d]`` (f32/f16/bf16) into the E4M3 caches at
    ``slot_mapping`` with the (block, kv head) scales (``value_cache`` None: the interleaved layout)."""
    num_blocks, hkv, bs, d = _fp8_cache(key_cache, value_cache, k_scale, v_scale)
    for name, t in (("key", key), ("value", value), ("slot_mapping", slot_mapping)):
        _cuda(t, name)
    _need(key.shape == value.shape and key.dim() == 3 and key.shape[1:] == (hkv, d), "key/value must be [T, H_kv, d]")
    _need(key.dtype == value.dtype, "key and value must share a dtype")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == key.shape[0], "slot_mapping: int64 [T]")
    vptr = value_cache.data_ptr() if value_cache is not None else None
    _check(library().pa_write_kv_fp8(key.data_ptr(), value.data_ptr(), key_cache.data_ptr(), vptr,
                                     k_scale.data_ptr(), v_scale.data_ptr(), slot_mapping.data_ptr(), key.shape[0],
                                     hkv, d, bs, num_blocks, _dtype_code(key), _stream_ptr(stream, key.device)))


def decode_fp8_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                              max_blocks_per_seq: int, dtype: torch.dtype) -> int:
    return int(library().pa_decode_fp8_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                      max_blocks_per_seq, _TORCH_DTYPES[dtype]))


def decode_fp8(query: torch.Tensor, key_cache: torch.Tensor, value_cache: Optional[torch.Tensor], k_scale: torch.Tensor,
               v_scale: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
               scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None, new_key: Optional[torch.Tensor] = None,
               new_value: Optional[torch.Tensor] = None) -> torch.Tensor:
    """``pa_decode_fp8``: paged decode attention over E4M3 caches with (block, kv head) scales; ``query``
    f16/bf16 ``[B, H_q, d]``.  ``workspace`` defaults to a fresh one of the plan's size.

    With ``new_key`` / ``new_value`` (``[B, H_kv, d]``, the query's dtype) it is
    ``pa_decode_fp8_append``: each sequence's new token is quantised into the slot of position
    L - 1 inside the decode, the same codes ``write_kv_fp8`` would store there.
    """
    num_blocks, hkv, bs, d = _fp8_cache(key_cache, value_cache, k_scale, v_scale)
    if new_key is not None or new_value is not None:
        _need(new_key is not None and new_value is not None, "new_key and new_value go together")
        _cuda(new_key, "new_key")
        _cuda(new_value, "new_value")
        _need(new_key.shape == (query.shape[0], hkv, d) and new_value.shape == new_key.shape,
              "new_key/new_value must be [B, H_kv, d]")
        _need(new_key.dtype == new_value.dtype == query.dtype, "new_key/new_value must have the query's dtype")
    for name, t in (("query", query), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda(t, name)
    _need(query.dim() == 3 and query.shape[2] == d, "query must be [B, H_q, d]")
    b, hq, _ = query.shape
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == b,
          "block_tables: int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == b, "context_lens: int32 [B]")
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    _need(out.shape == query.shape and out.dtype == query.dtype, "out must match query")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        n = decode_fp8_workspace_size(b, hq, hkv, d, bs, block_tables.shape[1], query.dtype)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=query.device)
    _cuda(workspace, "workspace")
    vptr = value_cache.data_ptr() if value_cache is not None else None
    tail = (block_tables.data_ptr(), context_lens.data_ptr(), b, hq, hkv, d, bs, block_tables.shape[1], num_blocks,
            float(scale), _dtype_code(query), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_ptr(stream, query.device))
    if new_key is None:
        _check(library().pa_decode_fp8(out.data_ptr(), query.data_ptr(), key_cache.data_ptr(), vptr,
                                       k_scale.data_ptr(), v_scale.data_ptr(), *tail))
    else:
        _check(library().pa_decode_fp8_append(out.data_ptr(), query.data_ptr(), new_key.data_ptr(),
                                              new_value.data_ptr(), key_cache.data_ptr(), vptr, k_scale.data_ptr(),
                                              v_scale.data_ptr(), *tail))
    return out


def decode_fp8_append(query: torch.Tensor, new_key: torch.Tensor, new_value: torch.Tensor, key_cache: torch.Tensor,
                      value_cache: Optional[torch.Tensor], k_scale: torch.Tensor, v_scale: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: Optional[float] = None,
                      out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """``pa_decode_fp8_append``: ``write_kv_fp8`` of each sequence's new token at position L - 1
    followed by ``decode_fp8``, in one kernel."""
    return decode_fp8(query, key_cache, value_cache, k_scale, v_scale, block_tables, context_lens, scale=scale,
                      out=out, workspace=workspace, stream=stream, new_key=new_key, new_value=new_value)


def decode_multi_workspace_size(num_seqs: int, q_len: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                block_size: int, max_blocks_per_seq: int, dtype: torch.dtype) -> int:
    return int(library().pa_decode_multi_workspace_size(num_seqs, q_len, num_heads, num_kv_heads, head_dim,
                                                        block_size, max_blocks_per_seq, _TORCH_DTYPES[dtype]))


def decode_multi(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor, block_tables: torch.Tensor,
                 context_lens: torch.Tensor, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, max_context_len: int = 0, partition_pages: int = 0,
                 kernel: str = "auto", stream=None) -> torch.Tensor:
    """``pa_decode_multi``: ``query`` ``[B, q_len, H_q, d]``; query token t of sequence b sits at position
    L_b - q_len + t and attends positions up to its own (causal).  Returns ``out`` of the query's shape."""
    for name, t in (("query", query), ("key_cache", key_cache), ("value_cache", value_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda(t, name)
    _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape, "caches must be [N, H_kv, bs, d]")
    num_blocks, hkv, bs, d = key_cache.shape
    _need(query.dim() == 4 and query.shape[3] == d, "query must be [B, q_len, H_q, d]")
    b, q_len, hq, _ = query.shape
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == b,
          "block_tables: int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == b, "context_lens: int32 [B]")
    _need(query.dtype == key_cache.dtype == value_cache.dtype, "query and caches must share a dtype")
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    _need(out.shape == query.shape and out.dtype == query.dtype, "out must match query")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        _cuda(workspace, "workspace")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(library().pa_decode_multi(out.data_ptr(), query.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(),
                                     block_tables.data_ptr(), context_lens.data_ptr(), b, q_len, hq, hkv, d, bs,
                                     block_tables.shape[1], num_blocks, float(scale), _dtype_code(query),
                                     ws_ptr or None, ws_bytes, max_context_len, partition_pages, KERNELS[kernel],
                                     _stream_ptr(stream, query.device)))
    return out


def decode_append(query: torch.Tensor, new_key: torch.Tensor, new_value: torch.Tensor, key_cache: torch.Tensor,
                  value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                  scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, max_context_len: int = 0, partition_pages: int = 0,
                  kernel: str = "auto", stream=None) -> torch.Tensor:
    """``pa_decode_append``: write the new token of every sequence at position L - 1, then decode.

    ``new_key`` / ``new_value``: ``[B, H_kv, d]``.  Same result as ``write_kv`` with the
    slots of positions L - 1 followed by ``decode``, in one kernel.
    """
    for name, t in (("query", query), ("new_key", new_key), ("new_value", new_value), ("key_cache", key_cache),
                    ("value_cache", value_cache), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda(t, name)
    _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape, "caches must be [N, H_kv, bs, d]")
    num_blocks, hkv, bs, d = key_cache.shape
    _need(query.dim() == 3 and query.shape[2] == d, "query must be [B, H_q, d]")
    b, hq, _ = query.shape
    _need(new_key.shape == (b, hkv, d) and new_value.shape == new_key.shape, "new_key/new_value must be [B, H_kv, d]")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == b,
          "block_tables: int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == b, "context_lens: int32 [B]")
    _need(query.dtype == key_cache.dtype == value_cache.dtype == new_key.dtype == new_value.dtype,
          "query, new key/value and caches must share a dtype")
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    _need(out.shape == query.shape and out.dtype == query.dtype, "out must match query")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        _cuda(workspace, "workspace")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(library().pa_decode_append(out.data_ptr(), query.data_ptr(), new_key.data_ptr(), new_value.data_ptr(),
                                      key_cache.data_ptr(), value_cache.data_ptr(), block_tables.data_ptr(),
                                      context_lens.data_ptr(), b, hq, hkv, d, bs, block_tables.shape[1], num_blocks,
                                      float(scale), _dtype_code(query), ws_ptr or None, ws_bytes, max_context_len,
                                      partition_pages, KERNELS[kernel], _stream_ptr(stream, query.device)))
    return out


def decode_static_scratch(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor, out: torch.Tensor,
                          scale: Optional[float] = None, stream=None) -> torch.Tensor:
    """``pa_decode_static_scratch``: ``decode`` with the library's built-in scratch.

    For callers that may not allocate device memory on the step path: nothing
    is allocated here either, so ``out`` is required.  Calls that overlap on
    the GPU (different streams) race on the one scratch; make the first call
    before any stream capture.  Sizes needing more than
    ``STATIC_SCRATCH_BYTES`` of scratch raise ``PAError`` (PA_ERR_UNSUPPORTED).
    """
    for name, t in (("query", query), ("key_cache", key_cache), ("value_cache", value_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens), ("out", out)):
        _cuda(t, name)
    _need(key_cache.dim() == 4 and value_cache.shape == key_cache.shape, "caches must be [N, H_kv, bs, d]")
    num_blocks, hkv, bs, d = key_cache.shape
    _need(query.dim() == 3 and query.shape[2] == d, "query must be [B, H_q, d]")
    b, hq, _ = query.shape
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == b,
          "block_tables: int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == b, "context_lens: int32 [B]")
    _need(query.dtype == key_cache.dtype == value_cache.dtype, "query and caches must share a dtype")
    _need(out.shape == query.shape and out.dtype == query.dtype, "out must match query")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(library().pa_decode_static_scratch(out.data_ptr(), query.data_ptr(), key_cache.data_ptr(),
                                              value_cache.data_ptr(), block_tables.data_ptr(),
                                              context_lens.data_ptr(), b, hq, hkv, d, bs, block_tables.shape[1],
                                              num_blocks, float(scale), _dtype_code(query),
                                              _stream_ptr(stream, query.device)))
    return out

class BlockPool:
    """Host block pool (``pa_pool``): free list, refcounts, fork, copy-on-write append."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        lib = library()
        handle = _P()
        order = None
        if free_order is not None:
            order = (ctypes.c_int32 * num_blocks)(*[int(x) for x in free_order])
        _check(lib.pa_pool_create(num_blocks, block_size, ctypes.cast(order, _P) if order is not None else None,
                                  ctypes.byref(handle)))
        self._h = handle
        self._lib = lib
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pa_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def create(self) -> int:
        sid = _I64()
        _check(self._lib.pa_seq_create(self._h, ctypes.byref(sid)))
        return sid.value

    def append(self, seq_id: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Append one token; returns (slot, (cow_src, cow_dst) or None)."""
        slot, src, dst = _I64(), _I64(), _I64()
        _check(self._lib.pa_seq_append(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)))
        return slot.value, ((src.value, dst.value) if src.value >= 0 else None)

    def append_batch(self, seq_ids):
        """Append one token to each sequence; returns (slots int64 [n], cow pairs int64 [k, 2]) as numpy."""
        import numpy as np

        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.size
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        k = _I()
        _check(self._lib.pa_seq_append_batch(self._h, ids.ctypes.data, n, slots.ctypes.data, pairs.ctypes.data,
                                             ctypes.byref(k)))
        return slots, pairs[:k.value].copy()

    def fork(self, seq_id: int) -> int:
        child = _I64()
        _check(self._lib.pa_seq_fork(self._h, seq_id, ctypes.byref(child)))
        return child.value

    def release(self, seq_id: int) -> None:
        _check(self._lib.pa_seq_release(self._h, seq_id))

    def blocks_needed(self, seq_ids, counts) -> int:
        """Free blocks that appending counts[i] tokens to seq_ids[i] (in order) would take
        (``pa_pool_blocks_needed``; nothing changes)."""
        import numpy as np

        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        assert ids.shape == cnt.shape
        out = _I64()
        _check(self._lib.pa_pool_blocks_needed(self._h, ids.ctypes.data, cnt.ctypes.data, ids.size,
                                               ctypes.byref(out)))
        return out.value

    def swap_to(self, dst: "BlockPool", seq_id: int):
        """Move a sequence into pool ``dst``: returns (its id there, int64 [n, 2] numpy (src block, dst block)
        pairs for ``swap_blocks``)."""
        import numpy as np

        n = self.length(seq_id)
        pairs = np.empty((max((n + self.block_size - 1) // self.block_size, 1), 2), dtype=np.int64)
        new_id, k = _I64(), _I()
        _check(self._lib.pa_seq_swap(self._h, dst._h, seq_id, ctypes.byref(new_id), pairs.ctypes.data,
                                     pairs.shape[0], ctypes.byref(k)))
        return new_id.value, pairs[:k.value].copy()

    def length(self, seq_id: int) -> int:
        n = _I64()
        _check(self._lib.pa_seq_length(self._h, seq_id, ctypes.byref(n)))
        return n.value

    def block_tables(self, seq_ids, max_blocks: int):
        """Host int32 tables [n, max_blocks] (-1 padded) and int32 lengths [n] (numpy)."""
        import numpy as np

        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tables = np.empty((ids.size, max_blocks), dtype=np.int32)
        lens = np.empty(ids.size, dtype=np.int32)
        _check(self._lib.pa_pool_block_tables(self._h, ids.ctypes.data, ids.size, tables.ctypes.data, max_blocks,
                                              lens.ctypes.data))
        return tables, lens

    def table_deltas(self, seq_ids, out=None, lens_out=None):
        """Delta export (``pa_pool_table_deltas``) for rows holding ``seq_ids``: returns (deltas int32 [k, 3],
        lens int32 [n]) as numpy views of ``out`` / ``lens_out`` when given (e.g. pinned staging), else new
        arrays."""
        import numpy as np

        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        if out is None:
            cap = sum((self.length(int(s)) + self.block_size - 1) // self.block_size for s in ids)
            out = np.empty((max(cap, 1), 3), dtype=np.int32)
        if lens_out is None:
            lens_out = np.empty(ids.size, dtype=np.int32)
        assert out.dtype == np.int32 and out.flags["C_CONTIGUOUS"] and lens_out.dtype == np.int32
        k = _I()
        _check(self._lib.pa_pool_table_deltas(self._h, ids.ctypes.data, ids.size, out.ctypes.data, out.size // 3,
                                              ctypes.byref(k), lens_out.ctypes.data))
        return out.reshape(-1, 3)[:k.value], lens_out[:ids.size]

    def num_free(self) -> int:
        return self._lib.pa_pool_num_free(self._h)

    def refcount(self, block: int) -> int:
        return self._lib.pa_pool_refcount(self._h, block)

    def free_list(self):
        import numpy as np

        out = np.empty(self.num_blocks, dtype=np.int32)
        n = self._lib.pa_pool_free_list(self._h, out.ctypes.data, self.num_blocks)
        return out[:n].tolist()

    def check_invariants(self) -> None:
        _check(self._lib.pa_pool_check_invariants(self._h))

    def save(self) -> bytes:
        """Checkpoint: the pool's whole state as bytes (``pa_pool_save``)."""
        n = self._lib.pa_pool_state_size(self._h)
        buf = ctypes.create_string_buffer(max(n, 1))
        written = _SZ()
        _check(self._lib.pa_pool_save(self._h, buf, n, ctypes.byref(written)))
        return buf.raw[:written.value]

    @classmethod
    def load(cls, state: bytes) -> "BlockPool":
        """Resume: a new pool from a ``save()`` image (``pa_pool_load``)."""
        lib = library()
        handle = _P()
        _check(lib.pa_pool_load(state, len(state), ctypes.byref(handle)))
        pool = cls.__new__(cls)
        pool._h, pool._lib = handle, lib
        pool.num_blocks = lib.pa_pool_num_blocks(handle)
        pool.block_size = lib.pa_pool_block_size(handle)
        return pool
