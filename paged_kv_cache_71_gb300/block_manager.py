"""Host-side block manager for a paged KV pool: who owns which physical block.

Two layers:

* ``BlockPool`` -- the physical blocks of one pool.  Free ids sit on a stack
  (a fixed numpy array and a top index; the id handed out next is the one on
  top, and a released id goes back on top), and every block carries a
  reference count: the number of sequences whose block table names it.
* ``SequenceTables`` -- the logical view: per sequence its block table and
  its token count.  It maps logical position p to the slot
  ``table[p // S] * S + p % S`` ("3.3 批处理与内存管理", section
  "PagedAttention：块表"), grows a table one block at a time as tokens
  arrive, lets a child sequence share all of a parent's blocks (parallel
  sampling / beam forks), and applies copy-on-write ("共享与写时复制"): a
  token may only be written into a block that no other sequence reads, so a
  write that lands in a shared, partly filled block first moves the writer
  onto a fresh block and records the (source, destination) pair whose data
  the ``copy_blocks`` kernel must copy.  Full shared blocks are never
  written again and stay shared.

Running out of free blocks raises ``MemoryError``: the pages leave that case
to the scheduler (preempt by swapping or recomputation), not to the pool.
Nothing here touches KV data; the kernels do.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


class BlockPool:
    """Free-id stack plus one reference count per physical block."""

    def __init__(self, num_blocks: int, free_order=None):
        n = int(num_blocks)
        order = np.arange(n, dtype=np.int64) if free_order is None else np.asarray(free_order, dtype=np.int64)
        if order.shape != (n,) or not np.array_equal(np.sort(order), np.arange(n)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self._stack = order.copy()          # ids; the top of the stack is _stack[_top - 1]
        self._top = n
        self.refcount = np.zeros(n, dtype=np.int64)

    @property
    def num_blocks(self) -> int:
        return int(self.refcount.shape[0])

    @property
    def num_free(self) -> int:
        return self._top

    def acquire(self) -> int:
        """Pop a free block and give it reference count 1."""
        if self._top == 0:
            raise MemoryError("KV pool exhausted: the scheduler must preempt (swap out or recompute)")
        self._top -= 1
        b = int(self._stack[self._top])
        self.refcount[b] = 1
        return b

    def retain(self, b: int) -> None:
        """One more table names block b."""
        self.refcount[b] += 1

    def release(self, b: int) -> None:
        """One table fewer names block b; at zero it goes back on the stack."""
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self._stack[self._top] = b
            self._top += 1


@dataclass
class _Seq:
    blocks: list = field(default_factory=list)
    length: int = 0


class SequenceTables:
    """Block tables of the sequences that live in one pool, with copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.block_size = int(block_size)
        self.pool = BlockPool(num_blocks, free_order)
        self._seqs: dict = {}
        self._copies: list[tuple[int, int]] = []

    # ---- queries
    def table(self, sid) -> list:
        return self._seqs[sid].blocks

    def length(self, sid) -> int:
        return self._seqs[sid].length

    def slot(self, sid, pos: int) -> int:
        """Cache slot of logical position ``pos``: physical block * S + offset."""
        S = self.block_size
        return self._seqs[sid].blocks[pos // S] * S + pos % S

    def block_tables(self, sids, width: int | None = None) -> np.ndarray:
        """int32 [len(sids), width] tables, entries past a sequence's last block set to -1."""
        rows = [self._seqs[s].blocks for s in sids]
        width = width or max(len(r) for r in rows)
        out = np.full((len(rows), width), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            out[i, : len(r)] = r
        return out

    # ---- changes
    def prefill(self, sid, n_tokens: int) -> None:
        """A new sequence holding n_tokens tokens: ceil(n / S) fresh blocks."""
        n = int(n_tokens)
        seq = _Seq()
        for _ in range((n + self.block_size - 1) // self.block_size):
            seq.blocks.append(self.pool.acquire())
        seq.length = n
        self._seqs[sid] = seq

    def next_slot(self, sid) -> int:
        """Reserve the slot of the sequence's next token and return it (one decode append)."""
        seq = self._seqs[sid]
        if seq.length % self.block_size == 0:
            seq.blocks.append(self.pool.acquire())       # the last block is full (or there is none)
        else:
            self._own_tail(seq)                          # writing into the partly filled last block
        pos = seq.length
        seq.length += 1
        return seq.blocks[pos // self.block_size] * self.block_size + pos % self.block_size

    def _own_tail(self, seq: _Seq) -> None:
        tail = seq.blocks[-1]
        if self.pool.refcount[tail] == 1:
            return
        fresh = self.pool.acquire()                      # taken first: on MemoryError nothing has changed
        self.pool.release(tail)
        seq.blocks[-1] = fresh
        self._copies.append((tail, fresh))

    def fork(self, parent, child) -> None:
        """The child starts as the parent's exact state, sharing every block."""
        src = self._seqs[parent]
        for b in src.blocks:
            self.pool.retain(b)
        self._seqs[child] = _Seq(list(src.blocks), src.length)

    def drop(self, sid) -> None:
        """The sequence is finished or preempted: its blocks lose one reference each."""
        for b in self._seqs.pop(sid).blocks:
            self.pool.release(b)

    def drain_copies(self) -> list[tuple[int, int]]:
        """Copy-on-write (src, dst) pairs recorded since the last call, in order."""
        out, self._copies = self._copies, []
        return out
