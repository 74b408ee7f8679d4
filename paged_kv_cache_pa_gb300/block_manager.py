"""Host-side block manager: allocation, fork, reserve with copy-on-write, free.

This is the bookkeeping that sits above the kernels and produces their inputs:
block tables, the slot of every new token (slot_mapping) and the (src, dst)
pairs of copy-on-write block copies.  The kernels see only physical block ids
and lengths and know nothing of sharing or reference counts
[Efficient Memory Management for Large Language Model Serving with
PagedAttention, "KV Cache Manager: Block Table Mapping", logical-to-physical
separation].

Behaviour follows the pages:

* Allocation pops a free block id in O(1); release decrements a reference
  count and returns the block to the free list at zero
  [vLLM Internals ..., "PagedAttention: page tables, for KV", BlockAllocator].
  The free list hands out the lowest free id first (or a caller-given order);
  that is the order the worked examples of "Paged Attention: Managing the KV
  Cache Like Virtual Memory" print.
* fork copies the table and increments every block's reference count;
  reserve copies a shared, partially filled last block before writing into it
  (copy-on-write), then appends blocks until the new tokens fit; free releases
  every block [Efficient Memory Management ..., "The three primitive
  operations" and "Copy-on-write mechanism"; Paged Attention: Managing the KV
  Cache ..., "A paged KV cache, in code", Sequence.reserve / fork / free].
* The slot of token position t is table[t // B] * B + t % B
  [Paged Attention: Managing the KV Cache ..., slot mapping note after the
  interleaving test].

No data moves here: a copy-on-write records a (src, dst) pair, which the
caller hands to ``pa_copy_blocks``.
"""
from __future__ import annotations

import heapq
from typing import Iterable, List, Optional, Tuple

BLOCK_SIZE = 16


class OutOfBlocks(RuntimeError):
    pass


class BlockPool:
    """Physical block ids 0..num_blocks-1 with reference counts."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE,
                 free_order: Optional[Iterable[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.refs = [0] * num_blocks
        self.copies: List[Tuple[int, int]] = []   # copy-on-write pairs, in order
        # A caller-given order is handed out first, then the rest lowest first.
        self._queue: List[int] = list(free_order) if free_order is not None else []
        if len(set(self._queue)) != len(self._queue) or any(
                not 0 <= b < num_blocks for b in self._queue):
            raise ValueError("free_order must list distinct valid block ids")
        given = set(self._queue)
        self._heap = [b for b in range(num_blocks) if b not in given]
        heapq.heapify(self._heap)
        self._queue.reverse()                      # pop() from the end

    @property
    def num_free(self) -> int:
        return len(self._queue) + len(self._heap)

    def alloc(self) -> int:
        if self._queue:
            b = self._queue.pop()
        elif self._heap:
            b = heapq.heappop(self._heap)
        else:
            raise OutOfBlocks("no free KV block")
        self.refs[b] = 1
        return b

    def release(self, b: int) -> None:
        if self.refs[b] <= 0:
            raise ValueError(f"release of free block {b}")
        self.refs[b] -= 1
        if self.refs[b] == 0:
            heapq.heappush(self._heap, b)

    def take_copies(self) -> List[Tuple[int, int]]:
        """Return and clear the copy-on-write pairs recorded so far."""
        out, self.copies = self.copies, []
        return out


class Sequence:
    """One sequence's block table and stored-token count."""

    def __init__(self, pool: BlockPool):
        self.pool = pool
        self.table: List[int] = []
        self.n = 0                                  # tokens whose K/V are stored

    def reserve(self, new: int) -> List[int]:
        """Make room for ``new`` more tokens and return their slots.

        A shared, partially filled last block is first copied (the pair is
        recorded in ``pool.copies``); then blocks are appended until the new
        tokens fit.  ``n`` advances by ``new``.
        """
        p, B = self.pool, self.pool.block_size
        if new < 0:
            raise ValueError("new must be >= 0")
        if self.n % B and p.refs[self.table[-1]] > 1:
            old = self.table[-1]
            b = p.alloc()
            p.copies.append((old, b))
            p.release(old)
            self.table[-1] = b
        while len(self.table) * B < self.n + new:
            self.table.append(p.alloc())
        slots = [self.table[t // B] * B + t % B for t in range(self.n, self.n + new)]
        self.n += new
        return slots

    def fork(self) -> "Sequence":
        child = Sequence(self.pool)
        child.table, child.n = list(self.table), self.n
        for b in self.table:
            self.pool.refs[b] += 1
        return child

    def free(self) -> None:
        for b in self.table:
            self.pool.release(b)
        self.table = []
        self.n = 0

    def fills(self) -> List[Tuple[int, int]]:
        """(physical block, filled slots) per logical block."""
        B = self.pool.block_size
        return [(b, min(B, self.n - i * B)) for i, b in enumerate(self.table)]


def blocks_for(length: int, block_size: int = BLOCK_SIZE) -> int:
    """Number of blocks that hold ``length`` tokens."""
    return -(-length // block_size)
