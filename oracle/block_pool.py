"""Allocator model for the paged KV cache (test infrastructure).

Semantics follow the BlockPool simulation on the "vLLM 与 PagedAttention" page
(section "最小分页与 COW 模拟"), restated here:

* free list: ids ``0..N-1`` (or a given order); an allocation takes the LAST
  id of the list (LIFO);
* every block carries the tokens written into it and a reference count;
* fork: a new table listing the same blocks, each block's count + 1;
* append: if the table is empty or its tail block is full, allocate a fresh
  block (no copy, even if the full tail is shared); else if the tail block is
  shared (count > 1), drop one reference to it and allocate a private copy of
  its tokens (copy-on-write); else write in place. The token goes to the tail.

Additions where that page is silent (each one a stated reading):

* release (the page names it but gives none; the MiniPaged-Qwen block manager
  and the ATB sketch free a request's blocks): every block of the table loses
  one reference; a block whose count reaches zero returns to the END of the
  free list, in table order;
* an exhausted pool raises ``MemoryError`` and leaves every structure as it
  was (the page lists OOM rollback among what a real allocator must handle);
* ``append`` also reports the slot of the new token (block * bs + offset,
  MiniPaged-Qwen section 8.1) and the (src, dst) pair of a copy-on-write;
* swap (the vLLM/PagedAttention page lists preemption as releasing or
  migrating a request's physical blocks while its logical tokens are kept; the
  LLM-inference page swaps a request's KV blocks to CPU memory and back): a
  sequence moves from one pool to another pool of the same block size.  Every
  block of its table, in table order, gets a fresh block of the destination
  pool (LIFO) holding the same tokens; then the sequence is released in the
  source pool (so a block it shared stays there for the other holders).  The
  moved blocks are private (sharing is not carried across a swap).  The
  destination names the sequence with its own next id.  Too few free blocks in
  the destination raise ``MemoryError`` with both pools unchanged;
* table deltas (the MiniPaged-Qwen page's closing notes ask for richer block
  metadata at lower host overhead): instead of every table entry, an export
  names only the entries a device-resident copy of the tables lacks (one copy,
  which receives every export in order).  The pool remembers, per sequence, the
  row it was last exported to and its table then, and per row the sequence last
  exported into it; exporting a sequence into the row that still holds it
  yields the entries that changed or were added since (a copy-on-write replaces
  the tail entry, an append past a full block adds one); exporting it into any
  other row, or for the first time, yields all of its entries.  Entries past a
  table's end are never read by the decode, so stale ones are left in place.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple


@dataclass
class AppendResult:
    table: List[int]
    slot: int
    cow: Optional[Tuple[int, int]]  # (source block, private copy) or None


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        if block_size <= 0 or num_blocks < 0:
            raise ValueError("bad pool geometry")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free: List[int] = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(self.free) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool")
        self.data: Dict[int, list] = {}
        self.refs: Dict[int, int] = {}

    # -- primitives ------------------------------------------------------------------------
    def _take(self, tokens: Sequence = ()) -> int:
        if not self.free:
            raise MemoryError("KV pool exhausted")
        block = self.free.pop()
        self.data[block] = list(tokens)
        self.refs[block] = 1
        return block

    def _drop(self, block: int) -> None:
        self.refs[block] -= 1
        if self.refs[block] == 0:
            del self.refs[block]
            del self.data[block]
            self.free.append(block)

    # -- the page's operations ---------------------------------------------------------------
    def fork(self, table: Sequence[int]) -> List[int]:
        for block in table:
            self.refs[block] += 1
        return list(table)

    def append(self, table: Sequence[int], token=None) -> AppendResult:
        table = list(table)
        cow = None
        tail_full = (not table) or len(self.data[table[-1]]) == self.block_size
        if tail_full:
            table.append(self._take())
        elif self.refs[table[-1]] > 1:
            shared = table[-1]
            private = self._take(self.data[shared])  # raises before any reference changes
            self.refs[shared] -= 1
            table[-1] = private
            cow = (shared, private)
        tail = table[-1]
        offset = len(self.data[tail])
        self.data[tail].append(token)
        return AppendResult(table=table, slot=tail * self.block_size + offset, cow=cow)

    def read(self, table: Sequence[int]) -> list:
        return [tok for block in table for tok in self.data[block]]

    def release(self, table: Sequence[int]) -> None:
        for block in table:
            self._drop(block)


class SequencePool:
    """Sequence-id layer over ``BlockPool`` (create / append / fork / release / tables)."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        self.pool = BlockPool(num_blocks, block_size, free_order)
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.synced: Dict[int, Tuple[int, List[int]]] = {}  # sequence -> (row, table) at its last delta export
        self.row_owner: Dict[int, int] = {}  # row -> sequence last exported into it
        self._next_id = 0

    @property
    def block_size(self) -> int:
        return self.pool.block_size

    def create(self) -> int:
        sid = self._next_id
        self._next_id += 1
        self.tables[sid] = []
        self.lens[sid] = 0
        return sid

    def append(self, sid: int, token=None) -> AppendResult:
        res = self.pool.append(self.tables[sid], token)
        self.tables[sid] = res.table
        self.lens[sid] += 1
        return res

    def fork(self, sid: int) -> int:
        child = self.create()
        self.tables[child] = self.pool.fork(self.tables[sid])
        self.lens[child] = self.lens[sid]
        return child

    def release(self, sid: int) -> None:
        self.pool.release(self.tables.pop(sid))
        del self.lens[sid]
        self.synced.pop(sid, None)

    def table_deltas(self, seq_ids: Sequence[int]):
        """Delta export for rows ``0..n-1`` holding ``seq_ids``: ([(row, logical block, physical block)],
        [length per row])."""
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence in two rows")
        deltas, lens = [], []
        for row, sid in enumerate(seq_ids):
            table = self.tables[sid]
            last_row, last = self.synced.get(sid, (-1, []))
            if last_row != row or self.row_owner.get(row) != sid:
                last = []  # the row holds someone else's entries: send every entry
            for j, block in enumerate(table):
                if j >= len(last) or last[j] != block:
                    deltas.append((row, j, block))
            self.synced[sid] = (row, list(table))
            self.row_owner[row] = sid
            lens.append(self.lens[sid])
        return deltas, lens

    def swap_to(self, dst: "SequencePool", sid: int):
        """Move sequence ``sid`` into pool ``dst``; returns (its id there, [(src block, dst block)])."""
        if dst.block_size != self.block_size:
            raise ValueError("pools differ in block size")
        table = self.tables[sid]
        if len(dst.pool.free) < len(table):
            raise MemoryError("destination pool exhausted")
        new_table = [dst.pool._take(self.pool.data[block]) for block in table]
        new_sid = dst.create()
        dst.tables[new_sid] = new_table
        dst.lens[new_sid] = self.lens[sid]
        self.release(sid)
        return new_sid, list(zip(table, new_table))

    def blocks_needed(self, seq_ids: Sequence[int], counts: Sequence[int]) -> int:
        """Reservation check (the vLLM/PagedAttention page's continuous batching: an iteration may admit
        only the growth the pool can hold): the free blocks that appending counts[i] tokens to seq_ids[i], in
        order, would take -- by doing it on a copy of the pool and counting."""
        import copy

        trial = copy.deepcopy(self)
        before = len(trial.pool.free)
        trial.pool.free = trial.pool.free + [-1 - i for i in range(sum(counts) + 1)]  # never runs out
        for sid, n in zip(seq_ids, counts):
            for _ in range(n):
                trial.append(sid)
        return before + sum(counts) + 1 - len(trial.pool.free)

    def num_free(self) -> int:
        return len(self.pool.free)

    def refcount(self, block: int) -> int:
        return self.pool.refs.get(block, 0)

    def block_tables(self, seq_ids: Sequence[int], width: int):
        import numpy as np

        tables = np.full((len(seq_ids), width), -1, dtype=np.int32)
        lens = np.zeros(len(seq_ids), dtype=np.int32)
        for i, sid in enumerate(seq_ids):
            t = self.tables[sid]
            if len(t) > width:
                raise ValueError("table wider than the output")
            tables[i, :len(t)] = t
            lens[i] = self.lens[sid]
        return tables, lens

    def invariants(self) -> List[str]:
        """Reading of MiniPaged-Qwen's ``invariants_ok``; returns the violations found."""
        bad = []
        bs = self.block_size
        counted: Dict[int, int] = {}
        for sid, table in self.tables.items():
            n = self.lens[sid]
            if len(table) != (n + bs - 1) // bs:
                bad.append(f"seq {sid}: {len(table)} blocks for {n} tokens")
            # internal waste bound of the vLLM page: 0 <= N*bs - T < bs
            if not (0 <= len(table) * bs - n < bs or (n == 0 and not table)):
                bad.append(f"seq {sid}: waste bound broken")
            for j, block in enumerate(table):
                counted[block] = counted.get(block, 0) + 1
                expect = bs if j < len(table) - 1 else n - (len(table) - 1) * bs
                if len(self.pool.data.get(block, ())) != expect:
                    bad.append(f"seq {sid}: block {block} holds {len(self.pool.data.get(block, ()))} tokens")
        if counted != self.pool.refs:
            bad.append("reference counts differ from table membership")
        free = set(self.pool.free)
        if len(free) != len(self.pool.free):
            bad.append("duplicate id in free list")
        if free & set(counted):
            bad.append("a block is both free and referenced")
        if free | set(counted) != set(range(self.pool.num_blocks)):
            bad.append("free and used blocks do not cover the pool")
        return bad
