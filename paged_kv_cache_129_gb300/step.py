"""Decode steps fed from host memory: packed uploads, double-buffered.

A serving loop hands the decode, every step, its queries, the new token's K/V,
the block tables and the context lengths from the host, and reads the outputs
back.  Copying each of those separately costs a copy launch and its latency
each, serialised with the kernel.  ``DecodeStepper`` keeps them in one pinned
host staging area per slot, laid out like the device staging area, so a step is
one host-to-device copy, one ``pa_decode_append`` (or ``pa_decode_ex``) call and
one device-to-host copy.  With two slots the upload of step i + 1 runs on a copy
stream while step i decodes.

Every byte moved or computed is moved by the CUDA runtime or computed by the
library's kernels, and the per-step sequence of copies, waits and calls runs in
the library's native step runner (pa_stepper_*); this module only lays out the
staging buffers and fills the call.
"""
from __future__ import annotations

import ctypes
import math
from types import SimpleNamespace
from typing import List, Optional, Tuple

import torch

from . import binding

_ALIGN = 256


def _layout(fields: List[Tuple[str, Tuple[int, ...], torch.dtype]]):
    offsets, off = {}, 0
    for name, shape, dtype in fields:
        off = (off + _ALIGN - 1) // _ALIGN * _ALIGN
        nbytes = math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
        offsets[name] = (off, shape, dtype, nbytes)
        off += nbytes
    return offsets, (off + _ALIGN - 1) // _ALIGN * _ALIGN


def _views(buf: torch.Tensor, offsets) -> SimpleNamespace:
    return SimpleNamespace(**{name: buf[off:off + nbytes].view(dtype).view(shape)
                              for name, (off, shape, dtype, nbytes) in offsets.items()})


class DecodeStepper:
    """Runs decode steps of a fixed batch shape from pinned host staging.

    Fill ``inputs(i)`` (host views: ``query``, ``block_tables``, ``context_lens``
    and, in append mode, ``new_key`` / ``new_value``), call ``launch(i)``, and
    ``result(i)`` returns the host view of step i's output once it has arrived.
    Step i uses slot ``i % slots``: refill that slot only after ``result(i)``.

    With ``tables="deltas"`` the block tables live on the device
    (``device_block_tables``, all -1 at first) and a step uploads only their
    changes: fill ``inputs(i).deltas`` with the pool's delta export
    (``BlockPool.table_deltas(seq_ids, out=inputs(i).deltas.numpy(),
    lens_out=inputs(i).context_lens.numpy())``) and pass its count to
    ``launch(i, num_deltas=k)``.  The deltas are applied on the decode's
    stream just before the decode, so stream order keeps them after the
    previous step's decode has read the table.

    FP8 caches (``k_scale`` / ``v_scale`` given, E4M3 codes in the caches,
    ``query_dtype`` f16 or bf16): with ``append`` a step is
    ``pa_decode_fp8_append`` (the new tokens quantised into position L - 1
    inside the decode), or with ``fp8_write="separate"`` ``pa_write_kv_fp8``
    of the new tokens at ``inputs(i).slots`` (int64) then ``pa_decode_fp8``;
    without ``append`` it is ``pa_decode_fp8``.
    """

    def __init__(self, key_cache: torch.Tensor, value_cache: torch.Tensor, num_seqs: int, num_heads: int,
                 max_blocks_per_seq: int, scale: Optional[float] = None, append: bool = True, slots: int = 2,
                 max_context_len: int = 0, partition_pages: int = 0, kernel: str = "auto", tables: str = "full",
                 k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                 query_dtype: Optional[torch.dtype] = None, fp8_write: str = "fused"):
        assert tables in ("full", "deltas") and fp8_write in ("fused", "separate")
        self.fp8 = k_scale is not None
        if self.fp8 and value_cache is None:  # interleaved FP8 layout [N, H_kv, 2, bs, d]
            assert key_cache.is_cuda and key_cache.dim() == 5 and key_cache.shape[2] == 2
            num_blocks, hkv, _, bs, d = key_cache.shape
        else:
            assert key_cache.is_cuda and key_cache.shape == value_cache.shape and key_cache.dim() == 4
            num_blocks, hkv, bs, d = key_cache.shape
        self.device = key_cache.device
        self.key_cache, self.value_cache = key_cache, value_cache
        if self.fp8:
            assert v_scale is not None and query_dtype in (torch.float16, torch.bfloat16)
            self.k_scale, self.v_scale = k_scale, v_scale
        dt = query_dtype if self.fp8 else key_cache.dtype
        self.shape = (num_seqs, num_heads, hkv, d, bs, max_blocks_per_seq, num_blocks)
        self.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        self.append, self.slots = append, slots
        self.fp8_slots = self.fp8 and append and fp8_write == "separate"
        self.max_context_len, self.partition_pages, self.kernel = max_context_len, partition_pages, kernel
        fields = [("query", (num_seqs, num_heads, d), dt)]
        if append:
            fields += [("new_key", (num_seqs, hkv, d), dt), ("new_value", (num_seqs, hkv, d), dt)]
            if self.fp8_slots:
                fields += [("slots", (num_seqs,), torch.int64)]
        self.deltas_mode = tables == "deltas"
        if self.deltas_mode:
            # the deltas go last, so that a step uploads only the prefix it uses
            fields += [("context_lens", (num_seqs,), torch.int32),
                       ("deltas", (num_seqs * max_blocks_per_seq, 3), torch.int32)]
            self.device_block_tables = torch.full((num_seqs, max_blocks_per_seq), -1, dtype=torch.int32,
                                                  device=self.device)
        else:
            fields += [("block_tables", (num_seqs, max_blocks_per_seq), torch.int32),
                       ("context_lens", (num_seqs,), torch.int32)]
        self._in, self._in_bytes = _layout(fields)
        self._last_h2d = self._in_bytes
        self._out, self._out_bytes = _layout([("out", (num_seqs, num_heads, d), dt)])
        self._h_in = [torch.empty(self._in_bytes, dtype=torch.uint8).pin_memory() for _ in range(slots)]
        self._d_in = [torch.empty(self._in_bytes, dtype=torch.uint8, device=self.device) for _ in range(slots)]
        self._h_out = [torch.empty(self._out_bytes, dtype=torch.uint8).pin_memory() for _ in range(slots)]
        self._d_out = [torch.empty(self._out_bytes, dtype=torch.uint8, device=self.device) for _ in range(slots)]
        self._hv_in = [_views(b, self._in) for b in self._h_in]
        self._dv_in = [_views(b, self._in) for b in self._d_in]
        self._hv_out = [_views(b, self._out).out for b in self._h_out]
        self._dv_out = [_views(b, self._out).out for b in self._d_out]
        ws_bytes = (binding.decode_fp8_workspace_size(num_seqs, num_heads, hkv, d, bs, max_blocks_per_seq, dt)
                    if self.fp8 else
                    binding.decode_workspace_size(num_seqs, num_heads, hkv, d, bs, max_blocks_per_seq, dt))
        # one workspace per slot: consecutive steps may overlap on the GPU
        self._ws = [torch.empty(max(ws_bytes, _ALIGN), dtype=torch.uint8, device=self.device) if ws_bytes else None
                    for _ in range(slots)]
        self.upload = torch.cuda.Stream(self.device)
        self.download = torch.cuda.Stream(self.device)
        self.compute = torch.cuda.current_stream(self.device)
        self._lib = binding.library()
        handle = ctypes.c_void_p()
        binding._check(self._lib.pa_stepper_create(slots, int(self.upload.cuda_stream),
                                                   int(self.compute.cuda_stream), int(self.download.cuda_stream),
                                                   ctypes.byref(handle)))
        self._st = handle
        for sl in range(slots):
            binding._check(self._lib.pa_stepper_set_slot(
                self._st, sl, self._h_in[sl].data_ptr(), self._d_in[sl].data_ptr(), self._in_bytes,
                self._h_out[sl].data_ptr(), self._d_out[sl].data_ptr(), self._out_bytes))
        self._slot_call = [None] * slots  # (key cache, value cache) each slot's call was set for

    def _set_call(self, s: int, kc: torch.Tensor, vc: torch.Tensor) -> None:
        """Give slot s its decode call (once per slot and pair of caches)."""
        key = (kc.data_ptr(), vc.data_ptr() if vc is not None else None)
        if self._slot_call[s] == key:
            return
        num_seqs, num_heads, hkv, d, bs, max_blocks, num_blocks = self.shape
        assert kc.shape == self.key_cache.shape and kc.dtype == self.key_cache.dtype
        assert (vc is None) == (self.value_cache is None) and (vc is None or vc.shape == kc.shape)
        dv, out, ws = self._dv_in[s], self._dv_out[s], self._ws[s]
        tables = self.device_block_tables if self.deltas_mode else dv.block_tables
        c = binding.StepCall()
        if self.fp8:
            c.kind = (binding.STEP_FP8_WRITE if self.fp8_slots else
                      binding.STEP_FP8_APPEND if self.append else binding.STEP_FP8)
        else:
            c.kind = binding.STEP_APPEND if self.append else binding.STEP_DECODE
        c.out, c.query = out.data_ptr(), dv.query.data_ptr()
        if self.append:
            c.new_key, c.new_value = dv.new_key.data_ptr(), dv.new_value.data_ptr()
            if self.fp8_slots:
                c.slots = dv.slots.data_ptr()
        c.key_cache, c.value_cache = kc.data_ptr(), (vc.data_ptr() if vc is not None else None)
        if self.fp8:
            c.k_scale, c.v_scale = self.k_scale.data_ptr(), self.v_scale.data_ptr()
        c.block_tables, c.context_lens = tables.data_ptr(), dv.context_lens.data_ptr()
        c.deltas = dv.deltas.data_ptr() if self.deltas_mode else None
        (c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim, c.block_size, c.max_blocks_per_seq,
         c.num_blocks) = num_seqs, num_heads, hkv, d, bs, max_blocks, num_blocks
        c.scale = self.scale
        c.dtype = binding._dtype_code(dv.query)
        if ws is not None:
            c.workspace, c.workspace_bytes = ws.data_ptr(), ws.numel()
        c.max_context_len, c.partition_pages = self.max_context_len, self.partition_pages
        c.kernel = binding.KERNELS[self.kernel]
        binding._check(self._lib.pa_stepper_set_call(self._st, s, ctypes.byref(c)))
        self._slot_call[s] = key

    @property
    def h2d_bytes(self) -> int:
        """Bytes the last launch uploaded (the whole staging area unless deltas are used)."""
        return self._last_h2d

    @property
    def d2h_bytes(self) -> int:
        return self._out_bytes

    def inputs(self, i: int) -> SimpleNamespace:
        """Pinned host views of step i's inputs (its slot's staging area)."""
        return self._hv_in[i % self.slots]

    def launch(self, i: int, key_cache: Optional[torch.Tensor] = None,
               value_cache: Optional[torch.Tensor] = None, num_deltas: int = 0) -> None:
        """Upload slot i % slots, decode it on the current stream, download its output.

        The sequence runs in native code (pa_stepper_launch) on three streams: the upload of a
        slot waits until the slot's previous decode has read its inputs; the decode waits for its
        upload (and for the previous download of the slot's output buffer); the download waits for
        the decode.  The decode stream thus holds only decodes and waits, and consecutive decodes
        keep overlapping.
        """
        s = i % self.slots
        kc = self.key_cache if key_cache is None else key_cache
        vc = self.value_cache if value_cache is None else value_cache
        nbytes = self._in_bytes
        if self.deltas_mode:
            off, shape, _, _ = self._in["deltas"]
            assert 0 <= num_deltas <= shape[0], "num_deltas out of range"
            nbytes = off + 12 * num_deltas
        else:
            num_deltas = 0
        self._set_call(s, kc, vc)
        binding._check(self._lib.pa_stepper_launch(self._st, i, nbytes, num_deltas))
        self._last_h2d = nbytes

    def close(self) -> None:
        if getattr(self, "_st", None):
            torch.cuda.synchronize(self.device)
            self._lib.pa_stepper_destroy(self._st)
            self._st = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def result(self, i: int) -> torch.Tensor:
        """Host view of step i's output, once its download has finished."""
        binding._check(self._lib.pa_stepper_wait(self._st, i))
        return self._hv_out[i % self.slots]
