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
library's kernels; this module only orders them.
"""
from __future__ import annotations

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
    ``query_dtype`` f16 or bf16): a step is ``pa_write_kv_fp8`` of the new
    tokens at ``inputs(i).slots`` (int64) when ``append``, then
    ``pa_decode_fp8``.
    """

    def __init__(self, key_cache: torch.Tensor, value_cache: torch.Tensor, num_seqs: int, num_heads: int,
                 max_blocks_per_seq: int, scale: Optional[float] = None, append: bool = True, slots: int = 2,
                 max_context_len: int = 0, partition_pages: int = 0, kernel: str = "auto", tables: str = "full",
                 k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                 query_dtype: Optional[torch.dtype] = None):
        assert tables in ("full", "deltas")
        assert key_cache.is_cuda and key_cache.shape == value_cache.shape and key_cache.dim() == 4
        self.device = key_cache.device
        self.key_cache, self.value_cache = key_cache, value_cache
        num_blocks, hkv, bs, d = key_cache.shape
        self.fp8 = k_scale is not None
        if self.fp8:
            assert v_scale is not None and query_dtype in (torch.float16, torch.bfloat16)
            self.k_scale, self.v_scale = k_scale, v_scale
        dt = query_dtype if self.fp8 else key_cache.dtype
        self.shape = (num_seqs, num_heads, hkv, d, bs, max_blocks_per_seq, num_blocks)
        self.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
        self.append, self.slots = append, slots
        self.max_context_len, self.partition_pages, self.kernel = max_context_len, partition_pages, kernel
        fields = [("query", (num_seqs, num_heads, d), dt)]
        if append:
            fields += [("new_key", (num_seqs, hkv, d), dt), ("new_value", (num_seqs, hkv, d), dt)]
            if self.fp8:
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
        self._uploaded = [torch.cuda.Event() for _ in range(slots)]
        self._decoded = [torch.cuda.Event() for _ in range(slots)]
        self._downloaded = [torch.cuda.Event() for _ in range(slots)]
        self._used = [False] * slots
        self._lib = binding.library()
        self._args = {}  # (slot, key cache, value cache) -> the C-ABI argument list

    def _call_args(self, s: int, kc: torch.Tensor, vc: torch.Tensor) -> list:
        key = (s, kc.data_ptr(), vc.data_ptr())
        args = self._args.get(key)
        if args is None:
            # assembled once per (slot, caches); the library still checks them on every call
            num_seqs, num_heads, hkv, d, bs, max_blocks, num_blocks = self.shape
            assert kc.shape == self.key_cache.shape and vc.shape == kc.shape and kc.dtype == self.key_cache.dtype
            dv, out, ws = self._dv_in[s], self._dv_out[s], self._ws[s]
            ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel()) if ws is not None else (None, 0)
            stream = int(self.compute.cuda_stream)
            code = binding._dtype_code(dv.query)
            kern = binding.KERNELS[self.kernel]
            tables = self.device_block_tables if self.deltas_mode else dv.block_tables
            if self.fp8:
                ks, vs = self.k_scale.data_ptr(), self.v_scale.data_ptr()
                args = [out.data_ptr(), dv.query.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks, vs, tables.data_ptr(),
                        dv.context_lens.data_ptr(), num_seqs, num_heads, hkv, d, bs, max_blocks, num_blocks,
                        self.scale, code, ws_ptr, ws_bytes, stream]
                if self.append:
                    args = (args, [dv.new_key.data_ptr(), dv.new_value.data_ptr(), kc.data_ptr(), vc.data_ptr(), ks,
                                   vs, dv.slots.data_ptr(), num_seqs, hkv, d, bs, num_blocks, code, stream])
            elif self.append:
                args = [out.data_ptr(), dv.query.data_ptr(), dv.new_key.data_ptr(), dv.new_value.data_ptr(),
                        kc.data_ptr(), vc.data_ptr(), tables.data_ptr(), dv.context_lens.data_ptr(),
                        num_seqs, num_heads, hkv, d, bs, max_blocks, num_blocks, self.scale, code, ws_ptr,
                        ws_bytes, self.max_context_len, self.partition_pages, kern, stream]
            else:
                args = [out.data_ptr(), dv.query.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                        tables.data_ptr(), dv.context_lens.data_ptr(), num_seqs, num_heads, hkv, d, bs,
                        max_blocks, num_blocks, self.scale, code, ws_ptr, ws_bytes, self.max_context_len,
                        self.partition_pages, kern, stream]
            self._args[key] = args
        return args

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

        Three streams: the upload of a slot waits until the slot's previous decode has read
        its inputs; the decode waits for its upload (and for the previous download of the
        slot's output buffer); the download waits for the decode.  The decode stream thus
        holds only decodes and waits, and consecutive decodes keep overlapping.
        """
        s = i % self.slots
        kc = self.key_cache if key_cache is None else key_cache
        vc = self.value_cache if value_cache is None else value_cache
        up, comp, down = self.upload, self.compute, self.download
        if self._used[s]:
            up.wait_event(self._decoded[s])
        nbytes = self._in_bytes
        if self.deltas_mode:
            off, shape, _, _ = self._in["deltas"]
            assert 0 <= num_deltas <= shape[0], "num_deltas out of range"
            nbytes = off + 12 * num_deltas
        torch.cuda.set_stream(up)
        try:
            self._d_in[s][:nbytes].copy_(self._h_in[s][:nbytes], non_blocking=True)
        finally:
            torch.cuda.set_stream(comp)
        self._last_h2d = nbytes
        self._uploaded[s].record(up)
        comp.wait_event(self._uploaded[s])
        if self._used[s]:
            comp.wait_event(self._downloaded[s])
        if self.deltas_mode and num_deltas:
            t = self.device_block_tables
            binding._check(self._lib.pa_apply_table_deltas(t.data_ptr(), t.shape[0], t.shape[1],
                                                           self._dv_in[s].deltas.data_ptr(), num_deltas,
                                                           int(comp.cuda_stream)))
        args = self._call_args(s, kc, vc)
        if self.fp8:
            if self.append:  # the new tokens' codes first, then the decode over them
                binding._check(self._lib.pa_write_kv_fp8(*args[1]))
                args = args[0]
            status = self._lib.pa_decode_fp8(*args)
        else:
            status = (self._lib.pa_decode_append if self.append else self._lib.pa_decode_ex)(*args)
        binding._check(status)
        self._decoded[s].record(comp)
        down.wait_event(self._decoded[s])
        torch.cuda.set_stream(down)
        try:
            self._h_out[s].copy_(self._d_out[s], non_blocking=True)
        finally:
            torch.cuda.set_stream(comp)
        self._downloaded[s].record(down)
        self._used[s] = True

    def result(self, i: int) -> torch.Tensor:
        """Host view of step i's output, once its download has finished."""
        s = i % self.slots
        self._downloaded[s].synchronize()
        return self._hv_out[s]
