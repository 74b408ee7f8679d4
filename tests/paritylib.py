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


def prefill_problem(cases, H, Hkv, D, dtype, B, seed, extra_blocks=3, dev="cuda:0"):
    """(cached, new) per sequence -> device tensors and host copies.  Blocks
    are scattered; every slot no context covers holds NaN."""
    rng = np.random.default_rng(seed)
    S = len(cases)
    lens = np.array([c + n for c, n in cases], np.int32)
    qsl = np.concatenate([[0], np.cumsum([n for _, n in cases])]).astype(np.int32)
    nbs = [-(-int(L) // B) for L in lens]
    NB = sum(nbs) + extra_blocks
    perm = rng.permutation(NB)
    maxb = max(max(nbs), 1)
    tables = np.full((S, maxb), -1, np.int32)
    pos = 0
    for s, n in enumerate(nbs):
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    slots = np.concatenate([tables[s, np.arange(c, c + n) // B].astype(np.int64) * B +
                            np.arange(c, c + n) % B for s, (c, n) in enumerate(cases)])
    T = int(qsl[-1])
    g = torch.Generator(device=dev).manual_seed(seed)
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    kc = torch.randn(NB, Hkv, B, D, generator=g, device=dev).to(dt)
    vc = torch.randn(NB, Hkv, B, D, generator=g, device=dev).to(dt)
    cover = np.zeros((NB, B), bool)
    for s, L in enumerate(lens):
        for t in range(int(L)):
            cover[tables[s, t // B], t % B] = True
    cv = torch.as_tensor(cover, device=dev)[:, None, :, None]
    nan = torch.tensor(float("nan"), dtype=dt, device=dev)
    kc = torch.where(cv, kc, nan).contiguous()
    vc = torch.where(cv, vc, nan).contiguous()
    q = torch.randn(T, H, D, generator=g, device=dev).to(dt)
    key = torch.randn(T, Hkv, D, generator=g, device=dev).to(dt)
    val = torch.randn(T, Hkv, D, generator=g, device=dev).to(dt)
    d = dict(q=q, kc=kc, vc=vc, key=key, val=val, tables=tables, qsl=qsl, lens=lens,
             slots=slots, maxq=max(n for _, n in cases), maxc=int(lens.max()))
    d["host"] = {k: codes(d[k]) for k in ("q", "kc", "vc", "key", "val")}
    return d


def prefill_run(d, scale, out_dtype=torch.float32, err=None, workspace=None):
    """The chunk's cache write, then prefill attention, on the device."""
    dev = d["q"].device
    pa.cache_write(d["key"], d["val"], d["kc"], d["vc"], torch.as_tensor(d["slots"], device=dev),
                   error_word=err)
    return pa.prefill_attention(d["q"], d["kc"], d["vc"], torch.as_tensor(d["tables"], device=dev),
                                torch.as_tensor(d["qsl"], device=dev),
                                torch.as_tensor(d["lens"], device=dev), d["maxq"], d["maxc"],
                                scale, out_dtype=out_dtype, workspace=workspace, error_word=err)


def prefill_oracle(d, scale, dtype):
    """The same two steps on the host copies (float64 output)."""
    h = d["host"]
    oracle.cache_write(h["key"], h["val"], h["kc"], h["vc"], d["slots"])
    return oracle.prefill_attention(h["q"], h["kc"], h["vc"], d["tables"], d["qsl"], d["lens"],
                                    scale, dtype)


def shared_workload(lens, share, H, Hkv, D, dtype="f16", B=16, seed=5, reuse_later=False,
                    extra_blocks=7):
    """lens[s] tokens per sequence; share[s] leading blocks copied from
    sequence s - 1's table (0 for the first).  reuse_later: a sequence also
    copies s - 1's ids a few blocks after its first fresh block (sharing that
    re-forms mid-table; only the leading run may be read once)."""
    rng = np.random.default_rng(seed)
    S = len(lens)
    nb = [-(-int(L) // B) for L in lens]
    need = sum(nb) + extra_blocks
    ids = iter(rng.permutation(need).tolist())
    maxb = max(nb)
    tables = np.full((S, maxb), -1, np.int32)
    for s in range(S):
        c = min(share[s], nb[s], nb[s - 1]) if s else 0
        row = list(tables[s - 1, :c]) if c else []
        while len(row) < nb[s]:
            j = len(row)
            if reuse_later and s and c and j >= c + 2 and j < nb[s - 1] and j < c + 5:
                row.append(int(tables[s - 1, j]))      # equal ids again after a break
            else:
                row.append(next(ids))
        tables[s, :nb[s]] = row
    lens = np.asarray(lens, np.int32)
    used = np.unique(tables[tables >= 0]).astype(np.int64)
    pos = np.maximum(lens.astype(np.int64) - 1, 0)
    slots = np.where(lens > 0, tables[np.arange(S), pos // B].astype(np.int64) * B + pos % B, -1)
    return synthetic.Workload(name="shared", num_seqs=S, num_heads=H, num_kv_heads=Hkv,
                              head_dim=D, dtype=dtype, num_blocks=need, context_lens=lens,
                              block_tables=tables, slot_mapping=slots, seed=seed,
                              used_blocks=used, block_size=B)
