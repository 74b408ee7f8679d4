"""Python binding of the native KV block manager (``include/pa_bm.h``).

Argument marshalling only: the bookkeeping (allocation, reference counts,
fork, append with copy-on-write, free, swap of sequence groups) runs in the
C++ code of ``libpa_gb300.so``.  The manager produces the kernels' inputs::

    bm = BlockManager(num_gpu_blocks, num_cpu_blocks, block_size=16)
    s = bm.new_sequence()
    slots = bm.append(s, prompt_len)          # -> pa_cache_write slot_mapping
    child = bm.fork(s)                        # parallel sampling / beams
    bm.append(child, 1)                       # copy-on-write of a shared block
    pairs = bm.take_copies()                  # -> pa_copy_blocks
    tables, lens = bm.build_batch([s, child], max_blocks)   # -> pa_decode_attention
    out_pairs = bm.swap_out([s, child])       # -> pa_swap_blocks (GPU -> CPU)
"""
from __future__ import annotations

import ctypes
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

from . import PaError, load_library

PA_ERR_NO_BLOCKS = 6

_P, _I, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
_SIGNATURES = {
    "pa_bm_create": (_I, [_I, _I, _I, ctypes.POINTER(_P)]),
    "pa_bm_destroy": (None, [_P]),
    "pa_bm_set_free_order": (_I, [_P, _P, _I]),
    "pa_bm_num_free_gpu": (_I, [_P]),
    "pa_bm_num_free_cpu": (_I, [_P]),
    "pa_bm_block_size": (_I, [_P]),
    "pa_bm_refcount": (_I, [_P, _I, _I]),
    "pa_bm_seq_create": (_I, [_P, ctypes.POINTER(_I64)]),
    "pa_bm_seq_fork": (_I, [_P, _I64, ctypes.POINTER(_I64)]),
    "pa_bm_seq_free": (_I, [_P, _I64]),
    "pa_bm_seq_append": (_I, [_P, _I64, _I, _P]),
    "pa_bm_blocks_needed": (_I, [_P, _I64, _I]),
    "pa_bm_seq_len": (_I, [_P, _I64]),
    "pa_bm_seq_on_cpu": (_I, [_P, _I64]),
    "pa_bm_seq_table": (_I, [_P, _I64, _P, _I]),
    "pa_bm_build_batch": (_I, [_P, _P, _I, _P, _I, _P]),
    "pa_bm_take_copies": (_I, [_P, _P, _I]),
    "pa_bm_num_copies": (_I, [_P]),
    "pa_bm_swap_out": (_I, [_P, _P, _I, _P, _I, ctypes.POINTER(_I)]),
    "pa_bm_swap_in": (_I, [_P, _P, _I, _P, _I, ctypes.POINTER(_I)]),
}
_bound = False


class NoFreeBlocks(PaError):
    """Not enough free blocks; the manager is unchanged."""


def _lib():
    global _bound
    lib = load_library()
    if not _bound:
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _bound = True
    return lib


def _check(status: int, op: str) -> None:
    if status == PA_ERR_NO_BLOCKS:
        raise NoFreeBlocks(status, op)
    if status != 0:
        raise PaError(status, op)


def _ids(seqs: Iterable[int]) -> np.ndarray:
    return np.ascontiguousarray(list(seqs), dtype=np.int64)


class BlockManager:
    """GPU block pool plus CPU swap space, with sequences named by int ids."""

    def __init__(self, num_gpu_blocks: int, num_cpu_blocks: int = 0, block_size: int = 16,
                 free_order: Optional[Sequence[int]] = None):
        self._lib = _lib()
        h = _P()
        _check(self._lib.pa_bm_create(num_gpu_blocks, num_cpu_blocks, block_size,
                                      ctypes.byref(h)), "pa_bm_create")
        self._h = h
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            _check(self._lib.pa_bm_set_free_order(self._h, order.ctypes.data, len(order)),
                   "pa_bm_set_free_order")

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    # ---- pools -------------------------------------------------------------
    @property
    def block_size(self) -> int:
        return self._lib.pa_bm_block_size(self._h)

    @property
    def num_free_gpu(self) -> int:
        return self._lib.pa_bm_num_free_gpu(self._h)

    @property
    def num_free_cpu(self) -> int:
        return self._lib.pa_bm_num_free_cpu(self._h)

    def refcount(self, block: int, on_cpu: bool = False) -> int:
        return self._lib.pa_bm_refcount(self._h, int(on_cpu), block)

    # ---- sequences ---------------------------------------------------------
    def new_sequence(self) -> int:
        out = _I64()
        _check(self._lib.pa_bm_seq_create(self._h, ctypes.byref(out)), "pa_bm_seq_create")
        return out.value

    def fork(self, parent: int) -> int:
        out = _I64()
        _check(self._lib.pa_bm_seq_fork(self._h, parent, ctypes.byref(out)), "pa_bm_seq_fork")
        return out.value

    def free(self, seq: int) -> None:
        _check(self._lib.pa_bm_seq_free(self._h, seq), "pa_bm_seq_free")

    def append(self, seq: int, num_tokens: int) -> np.ndarray:
        """Slots (int64) of num_tokens new tokens; raises NoFreeBlocks."""
        slots = np.empty(num_tokens, np.int64)
        _check(self._lib.pa_bm_seq_append(self._h, seq, num_tokens,
                                          slots.ctypes.data if num_tokens else None),
               "pa_bm_seq_append")
        return slots

    def blocks_needed(self, seq: int, num_tokens: int) -> int:
        return self._lib.pa_bm_blocks_needed(self._h, seq, num_tokens)

    def seq_len(self, seq: int) -> int:
        return self._lib.pa_bm_seq_len(self._h, seq)

    def on_cpu(self, seq: int) -> bool:
        r = self._lib.pa_bm_seq_on_cpu(self._h, seq)
        if r < 0:
            raise KeyError(seq)
        return bool(r)

    def table(self, seq: int) -> List[int]:
        n = self._lib.pa_bm_seq_table(self._h, seq, None, 0)
        if n < 0:
            raise KeyError(seq)
        out = np.empty(max(n, 1), np.int32)
        self._lib.pa_bm_seq_table(self._h, seq, out.ctypes.data, n)
        return out[:n].tolist()

    def fills(self, seq: int) -> List[Tuple[int, int]]:
        """(physical block, filled slots) per logical block."""
        B, n = self.block_size, self.seq_len(seq)
        return [(b, min(B, n - i * B)) for i, b in enumerate(self.table(seq))]

    # ---- kernel inputs -----------------------------------------------------
    def build_batch(self, seqs: Sequence[int], max_blocks_per_seq: int):
        """(block_tables int32 [n][max_blocks_per_seq], context_lens int32 [n])."""
        ids = _ids(seqs)
        tables = np.empty((len(ids), max_blocks_per_seq), np.int32)
        lens = np.empty(len(ids), np.int32)
        _check(self._lib.pa_bm_build_batch(self._h, ids.ctypes.data, len(ids), tables.ctypes.data,
                                           max_blocks_per_seq, lens.ctypes.data),
               "pa_bm_build_batch")
        return tables, lens

    def take_copies(self) -> np.ndarray:
        """Copy-on-write (src, dst) pairs queued so far, int64 [P][2]."""
        n = self._lib.pa_bm_num_copies(self._h)
        out = np.empty((max(n, 1), 2), np.int64)
        k = self._lib.pa_bm_take_copies(self._h, out.ctypes.data, n)
        return out[:k].copy()

    def _swap(self, fn, seqs, op) -> np.ndarray:
        ids = _ids(seqs)
        cap = sum(len(self.table(int(s))) for s in ids)
        out = np.empty((max(cap, 1), 2), np.int64)
        n = _I()
        _check(fn(self._h, ids.ctypes.data, len(ids), out.ctypes.data, cap, ctypes.byref(n)), op)
        return out[:n.value].copy()

    def swap_out(self, seqs: Sequence[int]) -> np.ndarray:
        """Move a sequence group to the CPU swap space; (gpu, cpu) pairs."""
        return self._swap(self._lib.pa_bm_swap_out, seqs, "pa_bm_swap_out")

    def swap_in(self, seqs: Sequence[int]) -> np.ndarray:
        """Bring a swapped-out group back to the GPU pool; (cpu, gpu) pairs."""
        return self._swap(self._lib.pa_bm_swap_in, seqs, "pa_bm_swap_in")
