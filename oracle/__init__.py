"""CPU oracle for the paged-KV-cache decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``paged_kv_cache_pa_gb300``) never imports, links or calls it, and the two
share no code: the arithmetic lives in ``pa_oracle.c`` (plain C, fp64), this
module only marshals numpy arrays into it.

What each function computes, and the passage it follows, is stated in the
header of ``pa_oracle.c``.  In short:

* ``half_to_double`` / ``double_to_half``: IEEE binary16 and bfloat16 from
  their bit layouts, round-to-nearest-even on encode.
* ``cache_write``: byte copy of every new token's K/V rows into the pool slot
  named by ``slot_mapping`` (block ``slot // B``, offset ``slot % B``, with B
  the pool's block size, its third dimension).
* ``copy_blocks``: byte copy of block ``src`` onto block ``dst`` in every
  layer's K and V pool.
* ``swap_blocks``: the same byte copy between two pools (GPU pool and CPU
  swap space, either way).
* ``decode_attention``: softmax(scale * q.K^T) V over the sequence's
  ``context_lens[s]`` tokens reached through ``block_tables[s]``, two-pass,
  accumulated in double.
* ``prefill_attention``: chunked-prefill attention, each new token over the
  sequence's positions up to its own (causal), read through the block table.
* ``decode_attention_blockwise``: the same through per-block partial states
  and a merge (the block-wise form of the attention equation).
* ``attention_weights``: the normalised weights a_t alongside the output.

Pins: every function above is checked in ``tests/test_oracle_pins.py``
against library routines, closed forms, invariants and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into libpa_oracle.so beside it (gcc, no fast-math,
    no FMA contraction, no host-specific flags)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.pa_oracle_half_to_double.restype = ctypes.c_double
            lib.pa_oracle_half_to_double.argtypes = [ctypes.c_uint16, I]
            lib.pa_oracle_double_to_half.restype = ctypes.c_uint16
            lib.pa_oracle_double_to_half.argtypes = [ctypes.c_double, I]
            lib.pa_oracle_decode_halves.argtypes = [P, P, ctypes.c_int64, I]
            lib.pa_oracle_encode_halves.argtypes = [P, P, ctypes.c_int64, I]
            lib.pa_oracle_cache_write.restype = I
            lib.pa_oracle_cache_write.argtypes = [P, P, P, P, P, I, I, I, I, I]
            lib.pa_oracle_copy_blocks.restype = I
            lib.pa_oracle_copy_blocks.argtypes = [P, P, I, P, I, I, I, I, I]
            lib.pa_oracle_prefill_attention.restype = I
            lib.pa_oracle_prefill_attention.argtypes = [P, P, P, P, P, I, P, P, I, I, I, I, I,
                                                        I, I, ctypes.c_double, I, I]
            lib.pa_oracle_swap_blocks.restype = I
            lib.pa_oracle_swap_blocks.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I]
            attn = [P, P, P, P, P, I, P, I, I, I, I, I, I, ctypes.c_double, I, I]
            lib.pa_oracle_decode_attention.restype = I
            lib.pa_oracle_decode_attention.argtypes = attn
            lib.pa_oracle_decode_attention_blockwise.restype = I
            lib.pa_oracle_decode_attention_blockwise.argtypes = attn
            lib.pa_oracle_attention_weights.restype = I
            lib.pa_oracle_attention_weights.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I,
                                                        I, ctypes.c_double, I]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


_RC = {1: "invalid argument", 2: "block id out of range", 3: "slot out of range",
       4: "out of memory"}


def _check(rc: int) -> None:
    if rc:
        raise OracleError(f"oracle returned {rc}: {_RC.get(rc, 'unknown')}")


def _u16(a: np.ndarray) -> np.ndarray:
    """View 16-bit float codes (float16 or uint16/int16 arrays) as uint16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16 or a.dtype == np.int16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit codes, got {a.dtype}")
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def half_to_double(codes: np.ndarray, dtype: str) -> np.ndarray:
    c = _u16(codes)
    out = np.empty(c.shape, np.float64)
    _load().pa_oracle_decode_halves(_ptr(c), _ptr(out), c.size, DTYPES[dtype])
    return out


def double_to_half(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().pa_oracle_encode_halves(_ptr(x), _ptr(out), x.size, DTYPES[dtype])
    return out


def cache_write(key, value, k_cache, v_cache, slot_mapping) -> None:
    """In place on k_cache / v_cache ([num_blocks][Hkv][B][D] 16-bit codes).
    key / value: [num_tokens][Hkv][D]."""
    key, value = _u16(key), _u16(value)
    kc, vc = _u16(k_cache), _u16(v_cache)
    if not (np.shares_memory(kc, k_cache) and np.shares_memory(vc, v_cache)):
        raise ValueError("pools must be contiguous 16-bit arrays (written in place)")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, hkv, bs, d = kc.shape
    assert key.shape[1:] == (hkv, d) and vc.shape == kc.shape
    _check(_load().pa_oracle_cache_write(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc),
                                         _ptr(slots), key.shape[0], nb, hkv, d, bs))


def copy_blocks(k_caches, v_caches, block_pairs) -> None:
    """In place: for every layer, pools[dst] = pools[src] for each (src, dst)."""
    pairs = np.ascontiguousarray(block_pairs, dtype=np.int64).reshape(-1, 2)
    ks = [_u16(k) for k in k_caches]
    vs = [_u16(v) for v in v_caches]
    for a, b in zip(ks + vs, list(k_caches) + list(v_caches)):
        if not np.shares_memory(a, b):
            raise ValueError("pools must be contiguous 16-bit arrays")
    nb, hkv, bs, d = ks[0].shape
    kp = (ctypes.c_void_p * len(ks))(*[_ptr(k) for k in ks])
    vp = (ctypes.c_void_p * len(vs))(*[_ptr(v) for v in vs])
    _check(_load().pa_oracle_copy_blocks(ctypes.cast(kp, ctypes.c_void_p),
                                         ctypes.cast(vp, ctypes.c_void_p), len(ks),
                                         _ptr(pairs), pairs.shape[0], nb, hkv, d, bs))


def swap_blocks(dst_k, dst_v, src_k, src_v, block_pairs) -> None:
    """In place on the destination pools: for every layer,
    dst[pair dst] = src[pair src] for each (src, dst) row of block_pairs.
    Source and destination pools may have different block counts."""
    pairs = np.ascontiguousarray(block_pairs, dtype=np.int64).reshape(-1, 2)
    dk, dv = [_u16(x) for x in dst_k], [_u16(x) for x in dst_v]
    sk, sv = [_u16(x) for x in src_k], [_u16(x) for x in src_v]
    for a, b in zip(dk + dv, list(dst_k) + list(dst_v)):
        if not np.shares_memory(a, b):
            raise ValueError("destination pools must be contiguous 16-bit arrays")
    nd, hkv, bs, d = dk[0].shape
    ns = sk[0].shape[0]
    assert sk[0].shape[1:] == (hkv, bs, d)
    arr = lambda xs: ctypes.cast((ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs]),
                                 ctypes.c_void_p)
    _check(_load().pa_oracle_swap_blocks(arr(dk), arr(dv), arr(sk), arr(sv), len(dk),
                                         _ptr(pairs), pairs.shape[0], nd, ns, hkv, d, bs))


def _attn_args(q, k_cache, v_cache, block_tables, context_lens):
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    s, h, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    assert d2 == d and vc.shape == kc.shape
    assert bt.ndim == 2 and bt.shape[0] == s and cl.shape == (s,)
    return q, kc, vc, bt, cl, s, h, d, nb, hkv, bs


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     dtype: str, nthreads: int | None = None) -> np.ndarray:
    """float64 [S][H][D] output of paged decode attention (token-wise, two-pass)."""
    q, kc, vc, bt, cl, s, h, d, nb, hkv, bs = _attn_args(q, k_cache, v_cache, block_tables,
                                                       context_lens)
    out = np.zeros((s, h, d), np.float64)
    _check(_load().pa_oracle_decode_attention(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), s, h, hkv,
        d, nb, bs, float(scale), DTYPES[dtype], nthreads or default_threads()))
    return out


def prefill_attention(q, k_cache, v_cache, block_tables, query_start_loc, context_lens,
                      scale: float, dtype: str, nthreads: int | None = None) -> np.ndarray:
    """float64 [T][H][D]: chunked-prefill attention.  q [T][H][D] holds the new
    tokens of every sequence (sequence s: rows query_start_loc[s] ..
    query_start_loc[s+1]-1), already written to the cache as the sequence's
    last positions; context_lens[s] counts the tokens after the chunk.  Row
    i of sequence s attends causally over positions 0 .. context_lens[s] - n_s + i."""
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    T, H, D = q.shape
    nb, hkv, bs, d2 = kc.shape
    S = len(cl)
    assert d2 == D and vc.shape == kc.shape and qsl.shape == (S + 1,) and bt.shape[0] == S
    out = np.zeros((T, H, D), np.float64)
    _check(_load().pa_oracle_prefill_attention(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(qsl), _ptr(cl), S, T,
        H, hkv, D, nb, bs, float(scale), DTYPES[dtype], nthreads or default_threads()))
    return out


def decode_attention_blockwise(q, k_cache, v_cache, block_tables, context_lens,
                               scale: float, dtype: str,
                               nthreads: int | None = None) -> np.ndarray:
    """float64 [S][H][D] output through per-block partial states and a merge."""
    q, kc, vc, bt, cl, s, h, d, nb, hkv, bs = _attn_args(q, k_cache, v_cache, block_tables,
                                                       context_lens)
    out = np.zeros((s, h, d), np.float64)
    _check(_load().pa_oracle_decode_attention_blockwise(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), s, h, hkv,
        d, nb, bs, float(scale), DTYPES[dtype], nthreads or default_threads()))
    return out


def attention_weights(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                      dtype: str):
    """(out [S][H][D], weights [S][H][max_ctx]) -- weights a_t = w_t / Z, zero past L."""
    q, kc, vc, bt, cl, s, h, d, nb, hkv, bs = _attn_args(q, k_cache, v_cache, block_tables,
                                                       context_lens)
    max_ctx = int(cl.max()) if s else 0
    out = np.zeros((s, h, d), np.float64)
    w = np.zeros((s, h, max(max_ctx, 1)), np.float64)
    _check(_load().pa_oracle_attention_weights(
        _ptr(out), _ptr(w), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), s,
        h, hkv, d, nb, bs, float(scale), DTYPES[dtype]))
    return out, w[:, :, :max_ctx]
