"""CPU oracle for paged decode attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA library: the
arithmetic lives in ``pa_oracle.c`` (fp64, plain loops) and in
``block_pool.py`` (the allocator model); this module only compiles the C file
with gcc and marshals numpy arrays into it.

Pins (tests under ``tests/`` marked ``not gpu``): dense softmax attention from
numpy/scipy on the gathered K/V, invariance under a permutation of the physical
blocks, NaN garbage in masked tail slots, hand-worked cases (L = 1, identical
keys, q = 0, a dominant key, a two-token fixture), the per-block-softmax
counter-example, element decoding against library casts, and the allocator
assertions of the vLLM/PagedAttention page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}

OK, BAD_ARG, BAD_TABLE, BAD_SLOT, NO_MEMORY = 0, -1, -2, -3, -4


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``_build/liboracle.so`` (gcc, plain C99)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_decode_rows.restype = i32
            lib.oracle_decode_rows.argtypes = [p, p, p, i32, p, p, p, i32, p, p, i32, i32, i32, i32,
                                               i32, i32, i32, dbl]
            lib.oracle_decode_multi_rows.restype = i32
            lib.oracle_decode_multi_rows.argtypes = [p, p, p, p, i32, p, p, p, i32, p, p, i32, i32, i32, i32,
                                                     i32, i32, i32, i32, dbl]
            lib.oracle_write_kv.restype = i32
            lib.oracle_write_kv.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32]
            lib.oracle_copy_blocks.restype = i32
            lib.oracle_copy_blocks.argtypes = [p, p, p, i32, i64, i32]
            lib.oracle_swap_blocks.restype = i32
            lib.oracle_swap_blocks.argtypes = [p, p, p, p, p, i32, i64, i32, i32]
            lib.oracle_decode_fp8_rows.restype = i32
            lib.oracle_decode_fp8_rows.argtypes = [p, p, p, i32, p, i32, p, p, p, p, p, p, i32, i32, i32, i32,
                                                   i32, i32, i32, dbl]
            lib.oracle_write_kv_fp8.restype = i32
            lib.oracle_write_kv_fp8.argtypes = [p, p, i32, p, p, p, p, p, i32, i32, i32, i32, i32]
            lib.oracle_e4m3_encode.restype = i32
            lib.oracle_e4m3_encode.argtypes = [p, i64, p]
            lib.oracle_element_to_double.restype = dbl
            lib.oracle_element_to_double.argtypes = [p, i32, i64]
            _lib = lib
        return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def element_to_double(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Decode every element of a storage array to float64 with the oracle's own decoder."""
    lib = _load()
    flat = np.ascontiguousarray(arr).reshape(-1)
    return np.array([lib.oracle_element_to_double(_ptr(flat), DTYPE_CODES[dtype], i) for i in range(flat.size)])


def decode(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray, block_tables: np.ndarray,
           context_lens: np.ndarray, dtype: str, scale: float, num_kv_heads: Optional[int] = None,
           rows: Optional[Sequence[tuple]] = None) -> np.ndarray:
    """fp64 decode attention over a paged cache.

    Returns ``[B, H_q, d]`` float64, or ``[len(rows), d]`` when ``rows`` (a list
    of ``(b, qh)``) selects output rows.
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    key_cache = np.ascontiguousarray(key_cache)
    value_cache = np.ascontiguousarray(value_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, num_heads, head_dim = q.shape
    num_blocks, hkv, block_size, d2 = key_cache.shape
    assert d2 == head_dim and value_cache.shape == key_cache.shape
    if num_kv_heads is not None:
        assert num_kv_heads == hkv
    if rows is None:
        rb, rh = np.meshgrid(np.arange(num_seqs), np.arange(num_heads), indexing="ij")
        rb, rh = rb.reshape(-1), rh.reshape(-1)
    else:
        rb = np.array([r[0] for r in rows]) if len(rows) else np.zeros(0)
        rh = np.array([r[1] for r in rows]) if len(rows) else np.zeros(0)
    rb = np.ascontiguousarray(rb, dtype=np.int32)
    rh = np.ascontiguousarray(rh, dtype=np.int32)
    out = np.zeros((rb.size, head_dim), dtype=np.float64)
    status = lib.oracle_decode_rows(_ptr(out), _ptr(rb), _ptr(rh), int(rb.size), _ptr(q), _ptr(key_cache),
                                    _ptr(value_cache), DTYPE_CODES[dtype], _ptr(bt), _ptr(lens), num_seqs,
                                    num_heads, hkv, head_dim, block_size, bt.shape[1], num_blocks, float(scale))
    if status != OK:
        raise ValueError(f"oracle decode failed with status {status}")
    return out.reshape(num_seqs, num_heads, head_dim) if rows is None else out


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """float32 values -> E4M3 codes (uint8): nearest, ties to even, saturating at 448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode(_ptr(x), int(x.size), _ptr(out))
    return out


def write_kv_fp8(key: np.ndarray, value: np.ndarray, dtype: str, key_cache: np.ndarray, value_cache: np.ndarray,
                 k_scale: np.ndarray, v_scale: np.ndarray, slot_mapping: np.ndarray) -> int:
    """In-place paged write into an E4M3 cache (uint8 [N, H_kv, bs, d]) with per-(block, kv head) float32
    scales [N, H_kv]: code = e4m3(float32(x) / scale).  Returns the oracle status."""
    lib = _load()
    num_blocks, hkv, block_size, head_dim = key_cache.shape
    key, value = np.ascontiguousarray(key), np.ascontiguousarray(value)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    assert key.shape == (slots.size, hkv, head_dim) and value.shape == key.shape
    assert key_cache.dtype == np.uint8 and value_cache.shape == key_cache.shape and value_cache.dtype == np.uint8
    assert key_cache.flags["C_CONTIGUOUS"] and value_cache.flags["C_CONTIGUOUS"]
    assert ks.shape == (num_blocks, hkv) and vs.shape == ks.shape
    return lib.oracle_write_kv_fp8(_ptr(key), _ptr(value), DTYPE_CODES[dtype], _ptr(key_cache), _ptr(value_cache),
                                   _ptr(ks), _ptr(vs), _ptr(slots), int(slots.size), hkv, head_dim, block_size,
                                   num_blocks)


def decode_fp8(q: np.ndarray, dtype: str, key_cache: np.ndarray, value_cache: np.ndarray, k_scale: np.ndarray,
               v_scale: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
               rows: Optional[Sequence[tuple]] = None) -> np.ndarray:
    """fp64 decode attention over an E4M3 cache with per-(block, kv head) scales; ``q`` in ``dtype``
    storage form.  Returns ``[B, H_q, d]`` float64, or ``[len(rows), d]`` for rows ``(b, qh)``."""
    lib = _load()
    q = np.ascontiguousarray(q)
    kc, vc = np.ascontiguousarray(key_cache), np.ascontiguousarray(value_cache)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, num_heads, head_dim = q.shape
    num_blocks, hkv, block_size, d2 = kc.shape
    assert d2 == head_dim and vc.shape == kc.shape and kc.dtype == np.uint8 and ks.shape == (num_blocks, hkv)
    if rows is None:
        rb, rh = np.meshgrid(np.arange(num_seqs), np.arange(num_heads), indexing="ij")
        rb, rh = rb.reshape(-1), rh.reshape(-1)
    else:
        rb = np.array([r[0] for r in rows]) if len(rows) else np.zeros(0)
        rh = np.array([r[1] for r in rows]) if len(rows) else np.zeros(0)
    rb = np.ascontiguousarray(rb, dtype=np.int32)
    rh = np.ascontiguousarray(rh, dtype=np.int32)
    out = np.zeros((rb.size, head_dim), dtype=np.float64)
    status = lib.oracle_decode_fp8_rows(_ptr(out), _ptr(rb), _ptr(rh), int(rb.size), _ptr(q), DTYPE_CODES[dtype],
                                        _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(lens), num_seqs,
                                        num_heads, hkv, head_dim, block_size, bt.shape[1], num_blocks, float(scale))
    if status != OK:
        raise ValueError(f"oracle fp8 decode failed with status {status}")
    return out.reshape(num_seqs, num_heads, head_dim) if rows is None else out


def decode_multi(q: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray, block_tables: np.ndarray,
                 context_lens: np.ndarray, dtype: str, scale: float, rows: Optional[Sequence[tuple]] = None
                 ) -> np.ndarray:
    """fp64 multi-query decode: ``q`` is ``[B, q_len, H_q, d]``; token t of sequence b sits at position
    L_b - q_len + t and attends positions 0 .. L_b - q_len + t (causal).

    Returns ``[B, q_len, H_q, d]`` float64, or ``[len(rows), d]`` for rows ``(b, t, qh)``.
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    key_cache = np.ascontiguousarray(key_cache)
    value_cache = np.ascontiguousarray(value_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, q_len, num_heads, head_dim = q.shape
    num_blocks, hkv, block_size, d2 = key_cache.shape
    assert d2 == head_dim and value_cache.shape == key_cache.shape
    if rows is None:
        rb, rt, rh = (x.reshape(-1) for x in np.meshgrid(np.arange(num_seqs), np.arange(q_len), np.arange(num_heads),
                                                           indexing="ij"))
    else:
        rb, rt, rh = (np.array([r[k] for r in rows]) for k in range(3))
    rb, rt, rh = (np.ascontiguousarray(x, dtype=np.int32) for x in (rb, rt, rh))
    out = np.zeros((rb.size, head_dim), dtype=np.float64)
    status = lib.oracle_decode_multi_rows(_ptr(out), _ptr(rb), _ptr(rt), _ptr(rh), int(rb.size), _ptr(q),
                                          _ptr(key_cache), _ptr(value_cache), DTYPE_CODES[dtype], _ptr(bt), _ptr(lens),
                                          num_seqs, q_len, num_heads, hkv, head_dim, block_size, bt.shape[1],
                                          num_blocks, float(scale))
    if status != OK:
        raise ValueError(f"oracle multi-query decode failed with status {status}")
    return out.reshape(num_seqs, q_len, num_heads, head_dim) if rows is None else out


def decode_inputs(inp, rows=None) -> np.ndarray:
    """``decode`` on a ``workloads.DecodeInputs`` (its caches as they stand)."""
    return decode(inp.q, inp.key_cache, inp.value_cache, inp.block_tables, inp.context_lens, inp.dtype,
                  inp.scale, inp.num_kv_heads, rows)


def write_kv(key: np.ndarray, value: np.ndarray, key_cache: np.ndarray, value_cache: np.ndarray,
             slot_mapping: np.ndarray) -> int:
    """In-place byte-exact paged write; returns the oracle status (0, or BAD_SLOT)."""
    lib = _load()
    num_blocks, hkv, block_size, head_dim = key_cache.shape
    key = np.ascontiguousarray(key)
    value = np.ascontiguousarray(value)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert key.shape == (slots.size, hkv, head_dim) and value.shape == key.shape
    assert key.dtype == value.dtype == key_cache.dtype == value_cache.dtype, "element types differ"
    assert key_cache.flags["C_CONTIGUOUS"] and value_cache.flags["C_CONTIGUOUS"]
    return lib.oracle_write_kv(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), _ptr(slots),
                               int(slots.size), hkv, head_dim, block_size, num_blocks, key_cache.itemsize)


def copy_blocks(key_cache: np.ndarray, value_cache: np.ndarray, pairs: np.ndarray) -> int:
    """In-place block copy dst <- src for every pair; returns the oracle status."""
    lib = _load()
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    num_blocks = key_cache.shape[0]
    block_bytes = key_cache.nbytes // num_blocks
    return lib.oracle_copy_blocks(_ptr(key_cache), _ptr(value_cache), _ptr(pairs), int(pairs.shape[0]),
                                  block_bytes, num_blocks)


def write_kv_layers(keys, values, key_caches, value_caches, slot_mapping: np.ndarray) -> int:
    """The paged write for every layer of a model: layer l's rows ``keys[l]`` / ``values[l]`` go into
    ``key_caches[l]`` / ``value_caches[l]`` at the shared ``slot_mapping`` (a sequence's blocks are the
    same physical ids in every layer's cache).  Returns the first non-OK oracle status, else OK."""
    status = OK
    for k, v, kc, vc in zip(keys, values, key_caches, value_caches):
        st = write_kv(k, v, kc, vc, slot_mapping)
        status = st if status == OK else status
    return status


def apply_table_deltas(block_tables: np.ndarray, deltas: np.ndarray) -> int:
    """Apply block-table deltas in place: every (row, logical block, physical block) row of ``deltas``
    sets ``block_tables[row, logical block]``; a row or column outside the table is skipped and
    reported (BAD_TABLE)."""
    status = OK
    rows, width = block_tables.shape
    for row, j, block in np.asarray(deltas, dtype=np.int64).reshape(-1, 3).tolist():
        if 0 <= row < rows and 0 <= j < width:
            block_tables[row, j] = block
        else:
            status = BAD_TABLE
    return status


def swap_blocks(dst_key: np.ndarray, dst_value: np.ndarray, src_key: np.ndarray, src_value: np.ndarray,
                pairs: np.ndarray) -> int:
    """Block copy between two pools (swap out / swap in): dst block <- src block for every
    (src, dst) pair, both caches, as bytes; returns the oracle status."""
    lib = _load()
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    assert dst_key.shape[1:] == src_key.shape[1:] and dst_key.dtype == src_key.dtype
    for a in (dst_key, dst_value, src_key, src_value):
        assert a.flags["C_CONTIGUOUS"]
    block_bytes = src_key[0].nbytes if src_key.shape[0] else dst_key[0].nbytes
    return lib.oracle_swap_blocks(_ptr(dst_key), _ptr(dst_value), _ptr(src_key), _ptr(src_value), _ptr(pairs),
                                  int(pairs.shape[0]), block_bytes, src_key.shape[0], dst_key.shape[0])


def slots_for_positions(block_tables: np.ndarray, seq_ids: Sequence[int], positions: Sequence[int],
                        block_size: int) -> np.ndarray:
    """Linear slot of logical position ``pos`` of sequence ``b``: table[b][pos // bs] * bs + pos % bs.

    (MiniPaged-Qwen, section 8.1: the slot handed back by append_token.)
    """
    out = np.empty(len(positions), dtype=np.int64)
    for i, (b, pos) in enumerate(zip(seq_ids, positions)):
        out[i] = int(block_tables[b][pos // block_size]) * block_size + pos % block_size
    return out
