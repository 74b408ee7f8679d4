"""Host logic of bench.py on CPU: the cross-rank max over two gloo ranks,
the reference (CPU oracle) arm on rank 0 and on other ranks, and the
algorithmic-bytes count."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
from paged_kv_cache_pa_gb300 import synthetic  # noqa: E402


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.reduce_max(1.5 + 10 * rank, dist)))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.5), (1, 11.5)]


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.25) == 3.25


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_rank0_prints_one_line():
    r = _run_bench(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3"],
                   {"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_algorithmic_bytes_closed_form():
    wl = synthetic.make("tiny")
    attn, write, copy = bench.algorithmic_bytes(wl)
    L = wl.context_lens.astype(np.int64)
    S, H, Hkv, D = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim
    kv = int(L.sum()) * Hkv * D * 2 * 2
    assert attn == kv + S * H * D * 2 + S * H * D * 4 + int(((L + 15) // 16).sum()) * 4 + S * 4
    assert write == 2 * S * Hkv * D * 2 * 2 + S * 8
    assert copy == 0
    b = synthetic.make("beams")
    assert bench.algorithmic_bytes(b)[2] == 2 * len(b.copy_pairs) * 40 * 16 * 128 * 2 * 2


def test_shared_blocks_count_once():
    """Two sequences of 20 tokens share their first block: 16 + 4 + 4 tokens
    must come from memory, 40 are read logically."""
    wl = synthetic._from_lengths("pair", np.array([20, 20]), 4, 2, 64, "f16", 1,
                                 np.random.default_rng(1), pool_blocks=8)
    wl.block_tables = np.array([[5, 1], [5, 2]], np.int32)
    assert bench.kv_tokens(wl) == 24
    assert bench.kv_tokens(wl, shared_once=False) == 40
    b = synthetic.make("beams")
    assert bench.kv_tokens(b) < bench.kv_tokens(b, shared_once=False)
    for name in ("tiny", "gqa"):      # no sharing: the two counts agree
        w = synthetic.make(name)
        assert bench.kv_tokens(w) == bench.kv_tokens(w, shared_once=False)
