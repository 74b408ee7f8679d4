"""GB300-native paged KV cache decode path.

Python binding of ``libpa_gb300.so`` (the C ABI declared in ``include/pa.h``)
with the same operation names.  This module only marshals arguments (device
pointers of torch tensors, sizes, the current CUDA stream); every step of the
path runs in the library's CUDA kernels.  There is no CPU fallback: calling an
operation without the built library, or with tensors that are not on a CUDA
device, raises.

    cache_write(key, value, k_cache, v_cache, slot_mapping)
    decode_attention(query, k_cache, v_cache, block_tables, context_lens,
                     max_context_len, scale, out=None, ...)
    copy_blocks(k_caches, v_caches, block_pairs)
    swap_blocks(dst_k_caches, dst_v_caches, src_k_caches, src_v_caches, block_pairs)
    prefill_attention(query, k_cache, v_cache, block_tables, query_start_loc,
                      context_lens, max_query_len, max_context_len, scale, ...)

Pools are [num_blocks][num_kv_heads][block_size][head_dim]; the block size
is read from their third dimension: 16 goes to the plain entry points, other
supported sizes (powers of two from 8 to 256) to the ``*_ex`` ones.

Build the library with ``python -m paged_kv_cache_pa_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

__all__ = ["cache_write", "decode_attention", "decode_attention_contiguous",
           "decode_workspace_size", "decode_partition_tokens", "decode_kernel_launches",
           "copy_blocks",
           "status_string", "PaError", "library_path", "load_library", "BLOCK_SIZE",
           "ERRBIT_BLOCK_OOB", "ERRBIT_SLOT_OOB", "ERRBIT_CONTEXT_LEN", "ERRBIT_TIMEOUT",
           "ERRBIT_INTERNAL",
           "MAX_LAYERS", "BLOCK_SIZES", "swap_blocks", "prefill_attention"]

BLOCK_SIZE = 16
BLOCK_SIZES = (8, 16, 32, 64, 128, 256)
MAX_LAYERS = 128
PA_F16, PA_BF16, PA_F32 = 0, 1, 2
ERRBIT_BLOCK_OOB, ERRBIT_SLOT_OOB, ERRBIT_CONTEXT_LEN, ERRBIT_TIMEOUT = 1, 2, 4, 8
ERRBIT_INTERNAL = 16  # PA_DEBUG builds only

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libpa_gb300.so")
_lib = None
_lock = threading.Lock()

# entry point -> (restype, argtypes)
_P, _I, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
_SIGNATURES = {
    "pa_cache_write": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "pa_cache_write_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pa_decode_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "pa_decode_partition_tokens": (_I, [_I, _I, _I]),
    "pa_decode_kernel_launches": (_I, [_I, _I, _I, _I, _I]),
    "pa_decode_attention": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                                 ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P]),
    "pa_decode_attention_ex": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I,
                                    _I, ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P]),
    "pa_decode_attention_contiguous": (_I, [_P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                            ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P]),
    "pa_copy_blocks": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _P]),
    "pa_copy_blocks_ex": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pa_prefill_attention": (_I, [_P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I,
                                  _I, _I, _I, ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P]),
    "pa_prefill_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "pa_swap_blocks": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pa_status_string": (ctypes.c_char_p, [_I]),
}


class PaError(RuntimeError):
    def __init__(self, status: int, op: str):
        self.status = status
        super().__init__(f"{op}: {status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libpa_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -m paged_kv_cache_pa_gb300.build` (there is no fallback path)")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().pa_status_string(int(status)).decode()


def _check(status: int, op: str) -> None:
    if status != 0:
        raise PaError(status, op)


def _dtype_code(dt) -> int:
    import torch
    if dt == torch.float16:
        return PA_F16
    if dt == torch.bfloat16:
        return PA_BF16
    if dt == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported dtype {dt}")


def _dev(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _opt_ptr(t, name):
    return None if t is None else _dev(t, name)


def cache_write(key, value, k_cache, v_cache, slot_mapping, error_word=None,
                stream=None) -> None:
    """Write key[t] / value[t] ([T][Hkv][D]) into pool slot slot_mapping[t]
    (int64; < 0 skips).  Pools: [num_blocks][Hkv][block_size][D]."""
    import torch
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    nb, hkv, bs, d = k_cache.shape
    if tuple(key.shape[1:]) != (hkv, d) or key.shape != value.shape:
        raise ValueError("shape mismatch between key/value and the pools")
    if v_cache.shape != k_cache.shape or k_cache.dtype != key.dtype or v_cache.dtype != key.dtype:
        raise ValueError("pools must match each other and the key dtype")
    args = (_dev(key, "key"), _dev(value, "value"), _dev(k_cache, "k_cache"),
            _dev(v_cache, "v_cache"), _dev(slot_mapping, "slot_mapping"), key.shape[0], nb)
    tail = (hkv, d, _dtype_code(key.dtype), _opt_ptr(error_word, "error_word"),
            _stream_ptr(stream, key.device))
    lib = load_library()
    if bs == BLOCK_SIZE:
        _check(lib.pa_cache_write(*args, *tail), "pa_cache_write")
    else:
        _check(lib.pa_cache_write_ex(*args, bs, *tail), "pa_cache_write_ex")


def decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                          max_context_len: int) -> int:
    return int(load_library().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads,
                                                       head_dim, max_context_len))


def decode_kernel_launches(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                           max_context_len: int) -> int:
    """Kernels one decode_attention call enqueues for these sizes."""
    return int(load_library().pa_decode_kernel_launches(num_seqs, num_heads, num_kv_heads,
                                                        head_dim, max_context_len))


def decode_partition_tokens(num_seqs: int, num_kv_heads: int, max_context_len: int) -> int:
    """Partition size pa_decode_attention uses; a merge kernel runs when
    max_context_len exceeds it."""
    return int(load_library().pa_decode_partition_tokens(num_seqs, num_kv_heads,
                                                         max_context_len))


def decode_attention(query, k_cache, v_cache, block_tables, context_lens,
                     max_context_len: int, scale: float, out=None, out_dtype=None,
                     workspace=None, error_word=None, stream=None):
    """Paged decode attention; returns ``out`` [S][H][D] (fp32 unless
    ``out_dtype`` / ``out`` says the input dtype).  ``workspace`` (uint8, >=
    decode_workspace_size bytes) is allocated here when not given.  Pools
    are [num_blocks][Hkv][block_size][D]."""
    import torch
    S, H, D = query.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S][max_blocks], context_lens [S]")
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype or torch.float32, device=query.device)
    if workspace is None:
        nbytes = decode_workspace_size(S, H, hkv, D, int(max_context_len))
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=query.device)
    head = (_dev(out, "out"), _dtype_code(out.dtype), _dev(query, "query"),
            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _dev(block_tables, "block_tables"), block_tables.shape[1],
            _dev(context_lens, "context_lens"), int(max_context_len), S, H, hkv, D, nb)
    tail = (float(scale), _dtype_code(query.dtype), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _opt_ptr(error_word, "error_word"),
            _stream_ptr(stream, query.device))
    lib = load_library()
    if bs == BLOCK_SIZE:
        _check(lib.pa_decode_attention(*head, *tail), "pa_decode_attention")
    else:
        _check(lib.pa_decode_attention_ex(*head, bs, *tail), "pa_decode_attention_ex")
    return out


def decode_attention_contiguous(query, k_cache, v_cache, context_lens, max_context_len: int,
                                scale: float, out=None, out_dtype=None, workspace=None,
                                error_word=None, stream=None):
    """Decode attention over a contiguous (unpaged) cache
    k_cache / v_cache [S][Hkv][max_rows][D] (max_rows a multiple of 16); the
    baseline that measures what the block table costs."""
    import torch
    S, H, D = query.shape
    s2, hkv, rows, d2 = k_cache.shape
    if s2 != S or d2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    if context_lens.dtype != torch.int32 or context_lens.shape != (S,):
        raise TypeError("context_lens must be int32 [S]")
    if out is None:
        out = torch.empty(S, H, D, dtype=out_dtype or torch.float32, device=query.device)
    if workspace is None:
        nbytes = decode_workspace_size(S, H, hkv, D, int(max_context_len))
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=query.device)
    st = load_library().pa_decode_attention_contiguous(
        _dev(out, "out"), _dtype_code(out.dtype), _dev(query, "query"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), rows, _dev(context_lens, "context_lens"), int(max_context_len),
        S, H, hkv, D, float(scale), _dtype_code(query.dtype), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt_ptr(error_word, "error_word"),
        _stream_ptr(stream, query.device))
    _check(st, "pa_decode_attention_contiguous")
    return out


def copy_blocks(k_caches: Sequence, v_caches: Sequence, block_pairs, error_word=None,
                stream=None) -> None:
    """For every layer: pools[dst] = pools[src] for each (src, dst) row of
    block_pairs (int64 [P][2], on the device)."""
    import torch
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("need the same, non-zero number of K and V pools")
    if block_pairs.dtype != torch.int64:
        raise TypeError("block_pairs must be int64")
    nb, hkv, bs, d = k_caches[0].shape
    for c in list(k_caches) + list(v_caches):
        if c.shape != k_caches[0].shape or c.dtype != k_caches[0].dtype:
            raise ValueError("all pools must have one shape and dtype")
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[_dev(c, "k_caches") for c in k_caches])
    vp = (ctypes.c_void_p * L)(*[_dev(c, "v_caches") for c in v_caches])
    npairs = block_pairs.shape[0] if block_pairs.numel() else 0
    head = (ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp, ctypes.c_void_p), L,
            _dev(block_pairs, "block_pairs") if npairs else None, npairs, nb)
    tail = (hkv, d, _dtype_code(k_caches[0].dtype), _opt_ptr(error_word, "error_word"),
            _stream_ptr(stream, k_caches[0].device))
    lib = load_library()
    if bs == BLOCK_SIZE:
        _check(lib.pa_copy_blocks(*head, *tail), "pa_copy_blocks")
    else:
        _check(lib.pa_copy_blocks_ex(*head, bs, *tail), "pa_copy_blocks_ex")


def _pool_ptr(t, name):
    """Pool pointer for pa_swap_blocks: a CUDA tensor or a pinned CPU tensor."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def swap_blocks(dst_k_caches: Sequence, dst_v_caches: Sequence, src_k_caches: Sequence,
                src_v_caches: Sequence, block_pairs, error_word=None, stream=None) -> None:
    """For every layer: dst[pair dst] = src[pair src] for each (src, dst) row
    of block_pairs (int64 [P][2], on the device).  Pools are
    [num_blocks][Hkv][block_size][D]; either side may be device memory or
    pinned host memory (the CPU swap space)."""
    import torch
    L = len(dst_k_caches)
    if not (L == len(dst_v_caches) == len(src_k_caches) == len(src_v_caches)) or not L:
        raise ValueError("need the same, non-zero number of pools on each side")
    if block_pairs.dtype != torch.int64:
        raise TypeError("block_pairs must be int64")
    nd, hkv, bs, d = dst_k_caches[0].shape
    ns = src_k_caches[0].shape[0]
    dt = dst_k_caches[0].dtype
    for c in list(dst_k_caches) + list(dst_v_caches):
        if tuple(c.shape) != (nd, hkv, bs, d) or c.dtype != dt:
            raise ValueError("destination pools must have one shape and dtype")
    for c in list(src_k_caches) + list(src_v_caches):
        if tuple(c.shape) != (ns, hkv, bs, d) or c.dtype != dt:
            raise ValueError("source pools must match the destination's block shape and dtype")
    arr = lambda xs, n: ctypes.cast((ctypes.c_void_p * L)(*[_pool_ptr(x, n) for x in xs]),
                                    ctypes.c_void_p)
    npairs = block_pairs.shape[0] if block_pairs.numel() else 0
    dev = next((c.device for c in [block_pairs] + list(dst_k_caches) + list(src_k_caches)
                if c.is_cuda), None)
    st = load_library().pa_swap_blocks(
        arr(dst_k_caches, "dst_k_caches"), arr(dst_v_caches, "dst_v_caches"),
        arr(src_k_caches, "src_k_caches"), arr(src_v_caches, "src_v_caches"), L,
        block_pairs.data_ptr() if npairs else None, npairs, nd, ns, bs, hkv, d, _dtype_code(dt),
        _opt_ptr(error_word, "error_word"), _stream_ptr(stream, dev))
    _check(st, "pa_swap_blocks")


def prefill_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                           max_query_len: int) -> int:
    return int(load_library().pa_prefill_workspace_size(num_seqs, num_heads, num_kv_heads,
                                                        head_dim, max_query_len))


def prefill_attention(query, k_cache, v_cache, block_tables, query_start_loc, context_lens,
                      max_query_len: int, max_context_len: int, scale: float, out=None,
                      out_dtype=None, workspace=None, error_word=None, stream=None):
    """Chunked-prefill attention: query [T][H][D] holds every sequence's new
    tokens (sequence s: rows query_start_loc[s] .. query_start_loc[s+1]-1),
    already written to the cache as its last positions; context_lens[s]
    counts the tokens after the chunk.  ``workspace`` (uint8, >=
    prefill_workspace_size bytes) is allocated here when not given.  Returns
    out [T][H][D]."""
    import torch
    T, H, D = query.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape mismatch")
    for t, n in ((block_tables, "block_tables"), (query_start_loc, "query_start_loc"),
                 (context_lens, "context_lens")):
        if t.dtype != torch.int32:
            raise TypeError(f"{n} must be int32")
    S = context_lens.shape[0]
    if query_start_loc.shape != (S + 1,) or block_tables.dim() != 2 or \
            block_tables.shape[0] != S:
        raise ValueError("query_start_loc must be [S+1], block_tables [S][max_blocks]")
    if out is None:
        out = torch.empty(T, H, D, dtype=out_dtype or torch.float32, device=query.device)
    if workspace is None:
        nbytes = prefill_workspace_size(S, H, hkv, D, int(max_query_len))
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=query.device)
    st = load_library().pa_prefill_attention(
        _dev(out, "out"), _dtype_code(out.dtype), _dev(query, "query"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(query_start_loc, "query_start_loc"), _dev(context_lens, "context_lens"),
        int(max_query_len), int(max_context_len), S, T, H, hkv, D, nb, bs, float(scale),
        _dtype_code(query.dtype), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt_ptr(error_word, "error_word"),
        _stream_ptr(stream, query.device))
    _check(st, "pa_prefill_attention")
    return out
