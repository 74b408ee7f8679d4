"""Shared helpers for the GPU parity tests: run one step of the decode path
through the library, and the same step through the CPU oracle on copies of
the same seeded inputs.

A step is: copy-on-write block copies (if the workload has any), the cache
write of each sequence's new token into slot_mapping, then decode attention
over context_lens tokens.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_pa_gb300 as pa
from paged_kv_cache_pa_gb300 import synthetic

ATOL = 2e-3          # attention, fp32 output: max |gpu - oracle|


def codes(t: torch.Tensor) -> np.ndarray:
    """16-bit float tensor -> host uint16 codes."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_step(wl, vals, out_dtype=torch.float32, error_word=None):
    """Run the step on the device, in place on vals' pools; returns out."""
    dev = vals["q"].device
    if len(wl.copy_pairs):
        pairs = torch.as_tensor(wl.copy_pairs, device=dev)
        pa.copy_blocks([vals["k_cache"]], [vals["v_cache"]], pairs, error_word=error_word)
    slots = torch.as_tensor(wl.slot_mapping, device=dev)
    pa.cache_write(vals["key"], vals["value"], vals["k_cache"], vals["v_cache"], slots,
                   error_word=error_word)
    tables = torch.as_tensor(wl.block_tables, device=dev)
    lens = torch.as_tensor(wl.context_lens, device=dev)
    return pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                               wl.max_context_len, wl.scale, out_dtype=out_dtype,
                               error_word=error_word)


def host_inputs(wl, vals, blocks=None):
    """Host copies for the oracle.  With ``blocks`` (sorted int64 ids), only
    those blocks are copied and the tables / slots / pairs are relabelled to
    positions in ``blocks``; otherwise whole pools are copied."""
    h = {k: codes(vals[k]) for k in ("q", "key", "value")}
    tables = wl.block_tables.astype(np.int64)
    slots = wl.slot_mapping.copy()
    pairs = wl.copy_pairs.copy()
    if blocks is None:
        h["k_cache"] = codes(vals["k_cache"])
        h["v_cache"] = codes(vals["v_cache"])
    else:
        idx = torch.as_tensor(blocks, device=vals["k_cache"].device)
        h["k_cache"] = codes(vals["k_cache"].index_select(0, idx))
        h["v_cache"] = codes(vals["v_cache"].index_select(0, idx))
        relabel = lambda b: np.searchsorted(blocks, b)
        B = wl.block_size
        tables = np.where(tables >= 0, relabel(np.maximum(tables, 0)), -1)
        slots = np.where(slots >= 0, relabel(np.maximum(slots, 0) // B) * B + slots % B, -1)
        if len(pairs):
            pairs = relabel(pairs)
    h["tables"] = tables.astype(np.int32)
    h["slots"] = slots.astype(np.int64)
    h["pairs"] = pairs.astype(np.int64).reshape(-1, 2)
    return h


def oracle_step(wl, h):
    """The same step on the host copies (pools updated in place); returns the
    float64 attention output."""
    if len(h["pairs"]):
        oracle.copy_blocks([h["k_cache"]], [h["v_cache"]], h["pairs"])
    oracle.cache_write(h["key"], h["value"], h["k_cache"], h["v_cache"], h["slots"])
    return oracle.decode_attention(h["q"], h["k_cache"], h["v_cache"], h["tables"],
                                   wl.context_lens, wl.scale, wl.dtype)


def step_blocks(wl):
    """Every block the step reads or writes (context blocks and copy targets)."""
    ids = wl.used_blocks if wl.used_blocks is not None else np.zeros(0, np.int64)
    if len(wl.copy_pairs):
        ids = np.union1d(ids, wl.copy_pairs.reshape(-1))
    return np.unique(ids).astype(np.int64)


def max_abs(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))


def custom_workload(lens, num_heads, num_kv_heads, head_dim, dtype, seed=7, extra_blocks=5,
                    scale=None, block_size=16):
    """A workload with the given lengths, blocks of ``block_size`` tokens
    scattered over a slightly larger pool (so some blocks belong to no
    sequence)."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    B = block_size
    wl = synthetic._from_lengths("custom", lens, num_heads, num_kv_heads, head_dim, dtype, seed,
                                 rng, pool_blocks=int(sum(-(-int(L) // B) for L in lens)) +
                                 extra_blocks, block_size=B)
    if scale is not None:
        wl.scale = scale
    return wl
