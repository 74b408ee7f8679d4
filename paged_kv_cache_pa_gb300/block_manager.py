"""Host-side block ledger: the pure-Python model of the KV block manager.

It keeps, in one object, a pool of physical block ids with a reference count
each and the block table and stored-token count of every sequence that uses
the pool.  It produces the kernels' inputs: block tables, the slot of every
new token (slot_mapping) and the (src, dst) pairs of copy-on-write block
copies.  The kernels see only physical block ids and lengths and know
nothing of sharing or reference counts [Efficient Memory Management for Large
Language Model Serving with PagedAttention, "KV Cache Manager: Block Table
Mapping", logical-to-physical separation].

Its structure is that of the native manager in ``csrc/pa_block_manager.cpp``
(sequences named by integer ids, every call checked before it changes
anything), so the two can be compared operation by operation; it exists to
generate the synthetic beam-search workload without loading the product
library, and as the second implementation the native manager is tested
against.

Behaviour:

* A new block is the first id of a caller-given order, else the lowest free
  id; a block whose last reference is dropped returns to the free set
  [vLLM Internals ..., "PagedAttention: page tables, for KV"].  The printed
  worked examples of "Paged Attention: Managing the KV Cache Like Virtual
  Memory" assume lowest-first.
* ``fork`` shares every block of the parent (one more reference each).
* ``append`` first counts the blocks it needs: a private copy of the last
  block when that block is partially filled and shared (copy-on-write), plus
  the blocks the new tokens spill into.  If the pool has fewer free blocks it
  raises and changes nothing.  Otherwise the copy's block is taken first, then
  the spill blocks, in that order (the printed examples fix the ids this
  yields) [Efficient Memory Management ..., "The three primitive operations"
  and "Copy-on-write mechanism"].
* The slot of position t is table[t // B] * B + t % B [Paged Attention:
  Managing the KV Cache ..., slot mapping note after the interleaving test].

No data moves here: a copy-on-write records a (src, dst) pair, which the
caller hands to ``pa_copy_blocks``.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field
from typing import Dict, Iterable, List, Optional, Tuple

BLOCK_SIZE = 16


class OutOfBlocks(RuntimeError):
    """Not enough free blocks; the ledger is unchanged."""


def blocks_for(length: int, block_size: int = BLOCK_SIZE) -> int:
    """Number of blocks that hold ``length`` tokens."""
    return -(-length // block_size)


@dataclass
class _Record:
    table: List[int] = field(default_factory=list)
    length: int = 0                                  # tokens whose K/V are stored


class BlockLedger:
    """One pool of ``num_blocks`` block ids and the sequences that use it."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE,
                 free_order: Optional[Iterable[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self._refs = [0] * num_blocks
        given = list(free_order) if free_order is not None else []
        if len(set(given)) != len(given) or any(not 0 <= b < num_blocks for b in given):
            raise ValueError("free_order must list distinct valid block ids")
        self._given = given[::-1]                    # next id at the end
        taken = set(given)
        self._lowest = [b for b in range(num_blocks) if b not in taken]
        heapq.heapify(self._lowest)
        self._records: Dict[int, _Record] = {}
        self._next_id = 0
        self._copies: List[Tuple[int, int]] = []

    # ---- pool ----------------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._given) + len(self._lowest)

    def refcount(self, block: int) -> int:
        return self._refs[block]

    def refcounts(self) -> List[int]:
        return list(self._refs)

    def _take(self) -> int:
        b = self._given.pop() if self._given else heapq.heappop(self._lowest)
        self._refs[b] = 1
        return b

    def _unref(self, block: int) -> None:
        self._refs[block] -= 1
        if self._refs[block] == 0:
            heapq.heappush(self._lowest, block)

    # ---- sequences -----------------------------------------------------------
    def new_sequence(self) -> int:
        sid = self._next_id
        self._next_id += 1
        self._records[sid] = _Record()
        return sid

    def fork(self, parent: int) -> int:
        src = self._records[parent]
        sid = self.new_sequence()
        self._records[sid] = _Record(list(src.table), src.length)
        for b in src.table:
            self._refs[b] += 1
        return sid

    def blocks_needed(self, seq: int, num_tokens: int) -> int:
        rec = self._records[seq]
        B = self.block_size
        tail_shared = rec.length % B != 0 and self._refs[rec.table[-1]] > 1
        spill = max(0, blocks_for(rec.length + num_tokens, B) - len(rec.table))
        return int(tail_shared) + spill

    def append(self, seq: int, num_tokens: int) -> List[int]:
        """Slots of ``num_tokens`` new tokens of ``seq``; raises OutOfBlocks
        (changing nothing) when the pool cannot supply the blocks."""
        if num_tokens < 0:
            raise ValueError("num_tokens must be >= 0")
        rec = self._records[seq]
        B = self.block_size
        need = self.blocks_needed(seq, num_tokens)
        if need > self.num_free:
            raise OutOfBlocks(f"sequence {seq} needs {need} blocks, {self.num_free} free")
        if rec.length % B != 0 and self._refs[rec.table[-1]] > 1:
            shared, private = rec.table[-1], self._take()
            self._copies.append((shared, private))
            self._unref(shared)
            rec.table[-1] = private
        while len(rec.table) < blocks_for(rec.length + num_tokens, B):
            rec.table.append(self._take())
        first, rec.length = rec.length, rec.length + num_tokens
        return [rec.table[t // B] * B + t % B for t in range(first, rec.length)]

    def release(self, seq: int) -> None:
        for b in self._records.pop(seq).table:
            self._unref(b)

    def table(self, seq: int) -> List[int]:
        return list(self._records[seq].table)

    def length(self, seq: int) -> int:
        return self._records[seq].length

    def fills(self, seq: int) -> List[Tuple[int, int]]:
        """(physical block, filled slots) per logical block."""
        rec, B = self._records[seq], self.block_size
        return [(b, min(B, rec.length - i * B)) for i, b in enumerate(rec.table)]

    def take_copies(self) -> List[Tuple[int, int]]:
        """Return and clear the copy-on-write pairs recorded so far."""
        out, self._copies = self._copies, []
        return out
