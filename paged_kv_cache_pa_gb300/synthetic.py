"""Seeded synthetic workloads for the paged decode path.

This module only builds inputs: sequence lengths, block placement, block
tables, the slot of each step's new token, copy-on-write pairs, and N(0, 1)
values.  It holds none of the kernels' arithmetic (no attention, no copy, no
cache write), so the tests and the bench can feed the same inputs to the CUDA
library and to the CPU oracle.

Shapes follow the pages' workloads:

* ``tiny``: 4 sequences, 8 heads = 8 KV heads, head_dim 64, fp16, lengths
  uniform in [1, 128], a 64-block pool dealt from one seeded permutation.
* ``opt13b``: OPT-13B attention (40 heads = 40 KV heads, head_dim 128, fp16;
  [Efficient Memory Management ..., section 2: 5120 hidden, 40 layers]),
  batch 256, length = prompt + output with prompt ~ lognormal(mean 220) and
  output ~ lognormal(mean 204), each clipped to [1, 1024], total clipped to
  2048 (ShareGPT means as measured on [Paged Attention: Managing the KV Cache
  Like Virtual Memory, "Where the memory goes"]; 2048 is OPT's maximum
  length).  The pool holds exactly the blocks in use, randomly permuted.
* ``gqa``: Qwen2.5-1.5B attention (12 query heads, 2 KV heads, head_dim 128,
  bf16; [Paged Attention: Managing the KV Cache ..., "Attention over
  scattered blocks"]), batch 64, lengths uniform in [512, 4096].
* ``beams``: 32 prompts x 6 beams, OPT-13B head shape, fp16, a 512-token
  prompt shared by the 6 beams of a group, 1..256 suffix tokens per group
  grown by a seeded beam search through the host block ledger
  (:class:`block_manager.BlockLedger`); each step copies shared partial last
  blocks (copy-on-write) before writing.
* ``long``: 8 sequences of 16384..32768 tokens, OPT-13B head shape, fp16,
  blocks drawn without replacement from a 196,608-block (60 GiB K+V) pool.

Lognormal reading: sigma = 1, mu = ln(mean) - sigma^2 / 2, rounded to the
nearest integer, then clipped.  Seeds are 1001 + config index unless given.

A step of the decode path is: copy-on-write copies (``beams`` only), the
cache write of one new token per sequence into the slot of position L - 1,
then attention over the L tokens.

Blocks hold 16 tokens unless a workload is re-laid with :func:`relayout`,
which keeps the lengths and deals blocks of another size.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

from .block_manager import BLOCK_SIZE, BlockLedger, blocks_for

CONFIGS = ("tiny", "opt13b", "gqa", "beams", "long")
SEEDS = {name: 1001 + i for i, name in enumerate(CONFIGS)}


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f16" or "bf16"
    num_blocks: int                 # pool size (blocks per layer pool)
    context_lens: np.ndarray        # int32 [S], includes the step's new token
    block_tables: np.ndarray        # int32 [S][max_blocks]; unused entries -1
    slot_mapping: np.ndarray        # int64 [S]: slot of position L-1
    copy_pairs: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))
    seed: int = 0
    scale: float = 0.0
    used_blocks: Optional[np.ndarray] = None   # int64 ids holding context tokens
    info: Dict[str, float] = field(default_factory=dict)
    block_size: int = BLOCK_SIZE    # tokens per pool block

    def __post_init__(self):
        if not self.scale:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def elt_bytes(self) -> int:
        return 2

    def kv_bytes(self) -> int:
        """K and V bytes the attention must read: sum_s L_s * Hkv * D * elt * 2."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * self.elt_bytes * 2


def _lognormal_int(rng: np.random.Generator, mean: float, n: int, lo: int, hi: int,
                   sigma: float = 1.0) -> np.ndarray:
    mu = math.log(mean) - sigma * sigma / 2.0
    x = np.rint(rng.lognormal(mu, sigma, n))
    return np.clip(x, lo, hi).astype(np.int64)


def _deal_tables(lens: np.ndarray, ids: np.ndarray, max_blocks: Optional[int] = None,
                 block_size: int = BLOCK_SIZE):
    """Give sequence s the next ceil(L_s/B) ids of ``ids``, in sequence order."""
    nb = [blocks_for(int(L), block_size) for L in lens]
    maxb = max_blocks or max(max(nb) if nb else 1, 1)
    tables = np.full((len(lens), maxb), -1, np.int32)
    pos = 0
    for s, n in enumerate(nb):
        tables[s, :n] = ids[pos:pos + n]
        pos += n
    return tables


def _slots_of_last(tables: np.ndarray, lens: np.ndarray,
                   block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Slot of position L-1 of each sequence (the token the step writes)."""
    B = block_size
    pos = np.maximum(lens.astype(np.int64) - 1, 0)
    blk = tables[np.arange(len(lens)), pos // B].astype(np.int64)
    return np.where(lens > 0, blk * B + pos % B, -1)   # empty: no token


def _from_lengths(name, lens, num_heads, num_kv_heads, head_dim, dtype, seed,
                  rng, pool_blocks=None, max_blocks=None, block_size=BLOCK_SIZE) -> Workload:
    lens = np.asarray(lens, np.int64)
    need = int(sum(blocks_for(int(L), block_size) for L in lens))
    if pool_blocks is None:
        pool_blocks = need
        ids = rng.permutation(pool_blocks)
    else:
        ids = rng.choice(pool_blocks, size=need, replace=False)
    tables = _deal_tables(lens, ids, max_blocks, block_size)
    return Workload(name=name, num_seqs=len(lens), num_heads=num_heads,
                    num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype,
                    num_blocks=pool_blocks, context_lens=lens.astype(np.int32),
                    block_tables=tables, slot_mapping=_slots_of_last(tables, lens, block_size),
                    seed=seed, used_blocks=np.sort(ids[:need]).astype(np.int64),
                    info={"mean_len": float(lens.mean()) if len(lens) else 0.0},
                    block_size=block_size)


def make_tiny(seed: Optional[int] = None, num_seqs: int = 4) -> Workload:
    seed = SEEDS["tiny"] if seed is None else seed
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 129, num_seqs)
    ids = rng.permutation(64)
    tables = _deal_tables(lens, ids, max_blocks=8)
    return Workload(name="tiny", num_seqs=num_seqs, num_heads=8, num_kv_heads=8,
                    head_dim=64, dtype="f16", num_blocks=64,
                    context_lens=lens.astype(np.int32), block_tables=tables,
                    slot_mapping=_slots_of_last(tables, lens), seed=seed,
                    used_blocks=np.sort(ids[:sum(blocks_for(int(L)) for L in lens)]),
                    info={"mean_len": float(lens.mean())})


def make_opt13b(seed: Optional[int] = None, num_seqs: int = 256) -> Workload:
    seed = SEEDS["opt13b"] if seed is None else seed
    rng = np.random.default_rng(seed)
    prompt = _lognormal_int(rng, 220.0, num_seqs, 1, 1024)
    out = _lognormal_int(rng, 204.0, num_seqs, 1, 1024)
    lens = np.minimum(prompt + out, 2048)
    return _from_lengths("opt13b", lens, 40, 40, 128, "f16", seed, rng, max_blocks=128)


def make_gqa(seed: Optional[int] = None, num_seqs: int = 64) -> Workload:
    seed = SEEDS["gqa"] if seed is None else seed
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 4097, num_seqs)
    return _from_lengths("gqa", lens, 12, 2, 128, "bf16", seed, rng, max_blocks=256)


def make_long(seed: Optional[int] = None, num_seqs: int = 8,
              pool_blocks: int = 196608) -> Workload:
    seed = SEEDS["long"] if seed is None else seed
    rng = np.random.default_rng(seed)
    lens = rng.integers(16384, 32769, num_seqs)
    return _from_lengths("long", lens, 40, 40, 128, "f16", seed, rng,
                         pool_blocks=pool_blocks, max_blocks=2048)


def make_beams(seed: Optional[int] = None, groups: int = 32, beams: int = 6,
               prompt: int = 512, max_suffix: int = 256, num_heads: int = 40,
               head_dim: int = 128, num_seqs: Optional[int] = None) -> Workload:
    """Beam groups sharing a prompt, grown by a seeded beam search.

    ``num_seqs`` (a smaller case for profiling) sets ``groups`` to
    num_seqs // beams, at least one.

    Every group prefills its prompt once and forks it ``beams - 1`` times.
    Its suffix length s_g ~ U{1..max_suffix}; for the s_g - 1 steps before the
    measured one, every beam stores one token (copying a shared partial last
    block first) and then every beam slot picks a parent uniformly among the
    group's beams (with replacement), forks it, and the old beams are freed.
    The measured step then stores one more token per beam: the copy-on-write
    pairs it needs become ``copy_pairs`` and its slots ``slot_mapping``.
    Blocks are handed out in a seeded random order over the pool.
    """
    if num_seqs:
        groups = max(1, num_seqs // beams)
    seed = SEEDS["beams"] if seed is None else seed
    rng = np.random.default_rng(seed)
    suffix = rng.integers(1, max_suffix + 1, groups)
    max_len = prompt + max_suffix
    # live blocks never exceed beams * blocks(max_len) per group, plus the
    # blocks a step allocates before it frees the old beams
    per_group = 2 * beams * blocks_for(max_len) + blocks_for(prompt)
    pool_blocks = groups * per_group
    ledger = BlockLedger(pool_blocks, free_order=rng.permutation(pool_blocks).tolist())
    all_beams = []
    for g in range(groups):
        root = ledger.new_sequence()
        ledger.append(root, prompt)
        group = [root] + [ledger.fork(root) for _ in range(beams - 1)]
        for _ in range(int(suffix[g]) - 1):
            for b in group:
                ledger.append(b, 1)
            parents = rng.integers(0, beams, beams)
            new = [ledger.fork(group[p]) for p in parents]
            for b in group:
                ledger.release(b)
            group = new
        all_beams.extend(group)
    ledger.take_copies()                     # history; not part of the step
    slots = np.array([ledger.append(b, 1)[0] for b in all_beams], np.int64)
    pairs = np.array(ledger.take_copies(), np.int64).reshape(-1, 2)
    lens = np.array([ledger.length(b) for b in all_beams], np.int32)
    maxb = blocks_for(max_len)
    tables = np.full((len(all_beams), maxb), -1, np.int32)
    for i, b in enumerate(all_beams):
        t = ledger.table(b)
        tables[i, :len(t)] = t
    used = np.unique(tables[tables >= 0]).astype(np.int64)
    logical = int(sum(blocks_for(int(L)) for L in lens))
    return Workload(name="beams", num_seqs=len(all_beams), num_heads=num_heads,
                    num_kv_heads=num_heads, head_dim=head_dim, dtype="f16",
                    num_blocks=pool_blocks, context_lens=lens, block_tables=tables,
                    slot_mapping=slots, copy_pairs=pairs, seed=seed, used_blocks=used,
                    info={"mean_len": float(lens.mean()), "unique_blocks": float(len(used)),
                          "logical_blocks": float(logical), "cow_pairs": float(len(pairs))})


def in_order(wl: Workload) -> Workload:
    """The same workload with every sequence's blocks laid out consecutively
    in the pool (sequence 0's blocks first), for comparing placements."""
    B = wl.block_size
    lens = wl.context_lens.astype(np.int64)
    need = int(sum(blocks_for(int(L), B) for L in lens))
    ids = np.arange(need, dtype=np.int64)
    tables = _deal_tables(lens, ids, wl.max_blocks_per_seq, B)
    return Workload(name=wl.name + "-inorder", num_seqs=wl.num_seqs, num_heads=wl.num_heads,
                    num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, dtype=wl.dtype,
                    num_blocks=max(need, 1), context_lens=wl.context_lens.copy(),
                    block_tables=tables, slot_mapping=_slots_of_last(tables, lens, B),
                    seed=wl.seed, scale=wl.scale, used_blocks=ids, info=dict(wl.info),
                    block_size=B)


def relayout(wl: Workload, block_size: int, seed: Optional[int] = None) -> Workload:
    """The same sequences (lengths, shapes, dtype, seed) stored in blocks of
    ``block_size`` tokens, scattered over a pool of the same byte size as
    ``wl``'s (or just large enough, if rounding each sequence up to whole
    blocks needs more).  Tables are dealt in sequence order from a seeded
    random choice of pool blocks, as the 16-token workloads are.  Copy-on-
    write pairs are not carried over (their blocks have no meaning here)."""
    if len(wl.copy_pairs):
        raise ValueError("relayout keeps no copy-on-write pairs")
    B = int(block_size)
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    lens = wl.context_lens.astype(np.int64)
    need = int(sum(blocks_for(int(L), B) for L in lens))
    same_bytes = -(-wl.num_blocks * wl.block_size // B)
    pool = max(need, same_bytes, 1)
    ids = rng.permutation(pool) if pool == need else rng.choice(pool, size=need, replace=False)
    maxb = max(-(-wl.max_blocks_per_seq * wl.block_size // B), 1)
    tables = _deal_tables(lens, ids, maxb, B)
    return Workload(name=f"{wl.name}-b{B}", num_seqs=wl.num_seqs, num_heads=wl.num_heads,
                    num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, dtype=wl.dtype,
                    num_blocks=pool, context_lens=wl.context_lens.copy(),
                    block_tables=tables, slot_mapping=_slots_of_last(tables, lens, B),
                    seed=wl.seed, scale=wl.scale,
                    used_blocks=np.sort(ids[:need]).astype(np.int64), info=dict(wl.info),
                    block_size=B)


MAKERS = {"tiny": make_tiny, "opt13b": make_opt13b, "gqa": make_gqa, "beams": make_beams,
          "long": make_long}


def make(name: str, **kw) -> Workload:
    return MAKERS[name](**kw)


# ---------------------------------------------------------------------------
# Values.  N(0, 1) in the workload's 16-bit dtype, drawn from a torch
# generator seeded with the workload seed, on the device the caller names.
# ---------------------------------------------------------------------------

def _torch_dtype(dtype: str):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def make_values(wl: Workload, device="cpu", seed: Optional[int] = None,
                fill_all_blocks: Optional[bool] = None, poison_unused: bool = False):
    """Tensors for one step: q [S][H][D], key/value [S][Hkv][D] (the new token),
    k_cache / v_cache [num_blocks][Hkv][block_size][D].

    Blocks listed in ``wl.used_blocks`` (and CoW destinations) always get
    N(0, 1) values.  Other blocks are filled too when ``fill_all_blocks``
    (default: pools under 4 GiB); otherwise they are left as allocated.
    ``poison_unused`` writes NaN into every slot no sequence's context covers
    (the tail of each last block and all unused blocks), so a kernel that reads
    past a sequence's length shows NaN in its output.
    """
    import torch
    seed = wl.seed if seed is None else seed
    dt = _torch_dtype(wl.dtype)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    S, H, Hkv, D, NB = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.num_blocks
    B = wl.block_size

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dt)

    q = randn(S, H, D)
    key = randn(S, Hkv, D)
    value = randn(S, Hkv, D)
    pool_bytes = NB * Hkv * B * D * 2
    if fill_all_blocks is None:
        fill_all_blocks = pool_bytes <= (4 << 30)
    k_cache = torch.empty(NB, Hkv, B, D, dtype=dt, device=device)
    v_cache = torch.empty(NB, Hkv, B, D, dtype=dt, device=device)
    if fill_all_blocks:
        chunk = max(1, (256 << 20) // (Hkv * B * D * 4))
        for c in (k_cache, v_cache):
            for b0 in range(0, NB, chunk):
                b1 = min(NB, b0 + chunk)
                c[b0:b1] = randn(b1 - b0, Hkv, B, D)
    else:
        ids = np.asarray(wl.used_blocks if wl.used_blocks is not None else [], np.int64)
        if len(wl.copy_pairs):
            ids = np.union1d(ids, wl.copy_pairs.reshape(-1))
        idx_all = torch.as_tensor(ids, device=device)
        chunk = max(1, (256 << 20) // (Hkv * B * D * 4))
        for c in (k_cache, v_cache):
            for i0 in range(0, len(ids), chunk):
                idx = idx_all[i0:i0 + chunk]
                c.index_copy_(0, idx, randn(len(idx), Hkv, B, D))
    if poison_unused:
        poison_pools(wl, k_cache, v_cache)
    return {"q": q, "key": key, "value": value, "k_cache": k_cache, "v_cache": v_cache}


def coverage_mask(wl: Workload) -> np.ndarray:
    """bool [num_blocks][block_size]: True where some sequence's context covers
    the slot (the new token's slot included)."""
    B = wl.block_size
    m = np.zeros((wl.num_blocks, B), bool)
    for s in range(wl.num_seqs):
        L = int(wl.context_lens[s])
        nb = blocks_for(L, B)
        for j in range(nb):
            b = int(wl.block_tables[s, j])
            n = min(B, L - j * B)
            m[b, :n] = True
    return m


def poison_pools(wl: Workload, k_cache, v_cache) -> None:
    """NaN into every uncovered slot of both pools (in place)."""
    import torch
    cover = torch.as_tensor(coverage_mask(wl), device=k_cache.device)
    nan = torch.tensor(float("nan"), dtype=k_cache.dtype, device=k_cache.device)
    for c in (k_cache, v_cache):
        c.copy_(torch.where(cover[:, None, :, None], c, nan))
