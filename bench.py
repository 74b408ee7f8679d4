"""Benchmark of the paged decode path on the OPT-13B-shaped decode step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config opt13b]

One step = one pass of the whole path over the batch: copy-on-write block
copies (when the workload has shared blocks; the OPT-13B-shaped batch has
none), the cache write of one new token per sequence, and paged decode
attention (plan, attention and merge kernels) over every sequence's context.
Inputs are synthetic and seeded (paged_kv_cache_pa_gb300.synthetic).

Metric: decode-attention achieved HBM GB/s = algorithmic bytes of the step /
step time, where the algorithmic bytes are what the method itself must move:
    attention: sum_s L_s * Hkv * D * 2 (K and V) * elt + q + out + table
               entries read (ceil(L_s/16) int32 each) + context_lens
    cache write: the new K/V rows read and written + slot_mapping
(last-block padding, workspace and L2 re-reads excluded).  Also reported:
sequences/s per layer, the roofline of the attention call, the CPU oracle as
a baseline, and an end-to-end number through the Python API with host
buffers.  Timed region: K steps between CUDA events on the launching stream,
bracketed by a barrier and device synchronisation; the K/V read per step
(~1.9 GB) is far larger than L2, so no flush is needed between steps.

With N > 1 (torchrun, one rank per GPU) every rank runs its own replica on
its own seeded batch (weak scaling; no collective on the data path); value =
all ranks' bytes / the slowest rank's time.

--impl reference times the CPU oracle (plain C, fp64, all host cores) on a
bounded sample of the same workload, same metric and unit.

Besides the named workload, a default run adds a ``per_config`` object with
the other decode workloads (grouped-query, long-context, shared-prefix beams,
tiny), each timed the same way with its own roofline fraction, spread and CPU
baseline; the chunked-prefill step with OPT-13B and grouped-query heads; and
the paged-versus-contiguous time ratio at 16-token blocks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention achieved HBM GB/s (% of GB300 peak) and sequences/sec per layer"
WORKLOADS = {
    "opt13b": "opt13b-shaped decode step: S=256, H=Hkv=40, D=128, fp16, block 16, lognormal "
              "prompt 220 + output 204, <=2048 tokens, scattered blocks, one layer",
    "gqa": "Qwen2.5-1.5B-shaped GQA decode step: S=64, H=12, Hkv=2, D=128, bf16, block 16, "
           "lengths U[512,4096], scattered blocks, one layer",
    "long": "long-context decode step: S=8, H=Hkv=40, D=128, fp16, block 16, lengths "
            "U[16384,32768], blocks drawn from a 60 GiB pool, one layer",
    "beams": "shared-prefix beam step: 32 prompts x 6 beams, H=Hkv=40, D=128, fp16, 512-token "
             "shared prompt, copy-on-write copies + cache write + attention, one layer",
    "tiny": "tiny decode step: S=4, H=Hkv=8, D=64, fp16, lengths U[1,128], 64-block pool",
}
UNIT = "GB/s"


def kv_tokens(wl, shared_once=True):
    """K/V tokens one step must read.  shared_once: each physical block's
    tokens count once however many tables hold it (the bytes that have to
    come from memory); otherwise every sequence's own L tokens (logical).
    The two agree unless sequences share blocks."""
    L = wl.context_lens.astype(np.int64)
    if not shared_once or len(L) == 0:
        return int(L.sum())
    B = wl.block_size
    nb = (L + B - 1) // B
    tables = np.asarray(wl.block_tables)
    j = np.arange(tables.shape[1])
    valid = j[None, :] < nb[:, None]
    toks = np.clip(L[:, None] - j[None, :] * B, 0, B)
    best = np.zeros(int(wl.num_blocks), np.int64)
    np.maximum.at(best, tables[valid].astype(np.int64), toks[valid])
    return int(best.sum())


def algorithmic_bytes(wl, out_elt=4, shared_once=True):
    """(attention bytes, cache-write bytes, copy bytes) of one step; blocks
    shared by several sequences count once unless shared_once is False."""
    S, H, Hkv, D, elt = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, 2
    L = wl.context_lens.astype(np.int64)
    B = wl.block_size
    nb = (L + B - 1) // B
    attn = kv_tokens(wl, shared_once) * Hkv * D * elt * 2 + S * H * D * elt + \
        S * H * D * out_elt + int(nb.sum()) * 4 + S * 4
    write = 2 * (S * Hkv * D * elt * 2) + S * 8
    copy = 2 * len(wl.copy_pairs) * Hkv * B * D * elt * 2
    return attn, write, copy


def reduce_max(value, dist=None, device=None):
    """Maximum of a per-rank float over all ranks (identity without a process
    group); works with NCCL (CUDA tensor) and gloo (CPU tensor)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_pa_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if (f.startswith("pa_decode") and f != "pa_decode_noalloc.cu") or f == "pa_ptx.cuh":
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config):
    """DRAM bytes per attention call from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec.get(config)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_call")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.5)

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts + frac, parts))
                except Exception:
                    continue
        os.unlink(self.path)
        inside = [p for ts, p in rows if t0 - 0.15 <= ts <= t1 + 0.15] or [p for _, p in rows]
        if not inside:
            return None
        sm = [float(p[2]) for p in inside if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for p in inside if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[6:10]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


def oracle_inputs(wl, seqs, seed=0, host_vals=None):
    """Inputs of the oracle for sequences ``seqs`` of ``wl`` (the blocks they
    use, renumbered): (q, kc, vc, tables, lens, algorithmic bytes)."""
    import torch
    seqs = np.asarray(seqs)
    tables = wl.block_tables[seqs]
    lens = wl.context_lens[seqs]
    used = np.unique(tables[tables >= 0])
    rel = np.where(tables >= 0, np.searchsorted(used, np.maximum(tables, 0)), -1).astype(np.int32)
    if host_vals is None:
        g = torch.Generator().manual_seed(seed)
        dt = torch.float16 if wl.dtype == "f16" else torch.bfloat16

        def r(*shape):
            return torch.randn(*shape, generator=g).to(dt).view(torch.int16).numpy().view(np.uint16)
        q = r(len(seqs), wl.num_heads, wl.head_dim)
        kc = r(len(used), wl.num_kv_heads, 16, wl.head_dim)
        vc = r(len(used), wl.num_kv_heads, 16, wl.head_dim)
    else:
        q, kc, vc = host_vals(seqs, used)
    sub = type(wl)(**{**wl.__dict__, "num_seqs": len(seqs), "context_lens": lens,
                      "block_tables": tables, "slot_mapping": wl.slot_mapping[seqs],
                      "copy_pairs": np.zeros((0, 2), np.int64)})
    return q, kc, vc, rel, lens, algorithmic_bytes(sub)[0]


def oracle_time(wl, inputs, threads):
    """Seconds of one oracle decode step on prepared inputs."""
    import oracle
    q, kc, vc, rel, lens, _ = inputs
    t = time.perf_counter()
    oracle.decode_attention(q, kc, vc, rel, lens, wl.scale, wl.dtype, nthreads=threads)
    return time.perf_counter() - t


def cpu_oracle_run(wl, seqs, threads=None, seed=0, host_vals=None):
    """Time the oracle on sequences ``seqs`` of ``wl``; returns (seconds,
    algorithmic bytes of those sequences, threads)."""
    import oracle
    threads = threads or oracle.default_threads()
    inputs = oracle_inputs(wl, seqs, seed, host_vals)
    return oracle_time(wl, inputs, threads), inputs[5], threads


def run_reference(args, wl, rank, world):
    """CPU oracle arm: rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    # size the per-step sample so the oracle's timed work stays within ~2
    # minutes; inputs are drawn for at most 8 distinct samples, which the
    # steps then cycle through (drawing them is slower than the oracle)
    t1, b1, _ = cpu_oracle_run(wl, [0], threads)
    rate = b1 / max(t1, 1e-6)
    per_seq = algorithmic_bytes(wl)[0] / wl.num_seqs
    budget_s = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.num_seqs, budget_s * rate / per_seq)))
    rng = np.random.default_rng(0)
    # distinct samples: at most 8, and at most ~0.5 GB of drawn inputs
    n_distinct = max(1, min(8, args.steps + args.warmup, int(0.5e9 // (n * per_seq))))
    prepared = [oracle_inputs(wl, rng.choice(wl.num_seqs, n, replace=False), seed=i)
                for i in range(n_distinct)]
    for i in range(args.warmup):
        oracle_time(wl, prepared[i % n_distinct], threads)
    tot_t = tot_b = 0.0
    for i in range(args.steps):
        inp = prepared[(args.warmup + i) % n_distinct]
        tot_t += oracle_time(wl, inp, threads)
        tot_b += inp[5]
    value = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS.get(args.config, args.config),
                   "parallelism": f"replicas x{world} (rank 0 runs the oracle)",
                   "sample_seqs_per_step": n, "distinct_samples": n_distinct},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": f"{n} random sequences of the workload per step, "
                                   f"{n_distinct} distinct samples cycled"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def layout_sweep(args, wl, dev):
    """Attention-call time on one workload in three layouts: the paged pool
    with scattered blocks, the paged pool with each sequence's blocks in
    order, and a contiguous cache [S][Hkv][rows][D] read without a table."""
    import torch
    import paged_kv_cache_pa_gb300 as pa
    from paged_kv_cache_pa_gb300 import synthetic
    S, H, Hkv, D = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim
    b_attn = algorithmic_bytes(wl)[0]
    out = torch.empty(S, H, D, dtype=torch.float32, device=dev)
    ws = torch.empty(pa.decode_workspace_size(S, H, Hkv, D, wl.max_context_len),
                     dtype=torch.uint8, device=dev)
    lens = torch.as_tensor(wl.context_lens, device=dev)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / args.steps

    res = {}
    for name, w in (("paged_scattered", wl), ("paged_in_order", synthetic.in_order(wl))):
        vals = synthetic.make_values(w, device=dev)
        tables = torch.as_tensor(w.block_tables, device=dev)
        ms = timed(lambda: pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables,
                                               lens, w.max_context_len, w.scale, out=out,
                                               workspace=ws))
        res[name] = {"ms_per_call": round(ms, 4), "GBps": round(b_attn / (ms * 1e-3) / 1e9, 1)}
        del vals
        torch.cuda.empty_cache()
    rows = int(-(-wl.max_context_len // 16) * 16)
    dt = synthetic._torch_dtype(wl.dtype)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    q = torch.randn(S, H, D, generator=g, device=dev).to(dt)
    kc = torch.randn(S, Hkv, rows, D, generator=g, device=dev).to(dt)
    vc = torch.randn(S, Hkv, rows, D, generator=g, device=dev).to(dt)
    ms = timed(lambda: pa.decode_attention_contiguous(q, kc, vc, lens, wl.max_context_len,
                                                      wl.scale, out=out, workspace=ws))
    res["contiguous"] = {"ms_per_call": round(ms, 4), "GBps": round(b_attn / (ms * 1e-3) / 1e9, 1)}
    base = res["contiguous"]["ms_per_call"]
    for v in res.values():
        v["time_vs_contiguous"] = round(v["ms_per_call"] / base, 4)
    del q, kc, vc
    torch.cuda.empty_cache()
    return {"layout_sweep": args.config, "workload": WORKLOADS.get(args.config),
            "steps": args.steps, "algorithmic_bytes": int(b_attn), "results": res}


def block_size_sweep(args, wl, dev):
    """Attention-call time on one workload's sequences stored in blocks of
    8 .. 256 tokens, each with the blocks scattered over the pool and in
    order; the contiguous cache is the common baseline."""
    import torch
    import paged_kv_cache_pa_gb300 as pa
    from paged_kv_cache_pa_gb300 import synthetic
    S, H, Hkv, D = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim
    out = torch.empty(S, H, D, dtype=torch.float32, device=dev)
    ws = torch.empty(pa.decode_workspace_size(S, H, Hkv, D, wl.max_context_len),
                     dtype=torch.uint8, device=dev)
    lens = torch.as_tensor(wl.context_lens, device=dev)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / args.steps

    rows = int(-(-wl.max_context_len // 16) * 16)
    dt = synthetic._torch_dtype(wl.dtype)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    q = torch.randn(S, H, D, generator=g, device=dev).to(dt)
    kc = torch.randn(S, Hkv, rows, D, generator=g, device=dev).to(dt)
    vc = torch.randn(S, Hkv, rows, D, generator=g, device=dev).to(dt)
    base = timed(lambda: pa.decode_attention_contiguous(q, kc, vc, lens, wl.max_context_len,
                                                        wl.scale, out=out, workspace=ws))
    del q, kc, vc
    torch.cuda.empty_cache()
    res = {"contiguous": {"ms_per_call": round(base, 4)}}
    for B in pa.BLOCK_SIZES:
        w0 = wl if B == wl.block_size else synthetic.relayout(wl, B)
        for order, w in (("scattered", w0), ("in_order", synthetic.in_order(w0))):
            vals = synthetic.make_values(w, device=dev)
            tables = torch.as_tensor(w.block_tables, device=dev)
            ms = timed(lambda: pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"],
                                                   tables, lens, w.max_context_len, w.scale,
                                                   out=out, workspace=ws))
            b_attn = algorithmic_bytes(w)[0]
            res[f"b{B}_{order}"] = {"ms_per_call": round(ms, 4),
                                    "GBps": round(b_attn / (ms * 1e-3) / 1e9, 1),
                                    "time_vs_contiguous": round(ms / base, 4)}
            del vals
            torch.cuda.empty_cache()
    print(json.dumps({"block_size_sweep": args.config, "workload": WORKLOADS.get(args.config),
                      "steps": args.steps, "results": res}), flush=True)


def swap_sweep(args, dev, tokens=2048, layers=40, num_kv_heads=40, head_dim=128):
    """Swap-out (device pool -> pinned host pool) and swap-in (back, into
    other block ids) of one request's KV cache over every layer, one
    pa_swap_blocks call per direction, at block sizes 8 .. 256.  The default
    request is a full-length OPT-13B-shaped one: 2048 tokens x 40 layers x
    40 KV heads x 128 x fp16, K and V = 1.68 GB each way.  Device pools hold
    twice the request's blocks; block ids on both sides are seeded random."""
    import torch
    import paged_kv_cache_pa_gb300 as pa
    row = num_kv_heads * head_dim                     # elements per token per pool
    dflat = [[torch.randn(2 * tokens * row, device=dev).half() for _ in range(2)]
             for _ in range(layers)]
    hflat = [[torch.empty(tokens * row, dtype=torch.float16).pin_memory() for _ in range(2)]
             for _ in range(layers)]
    nbytes = 2 * layers * tokens * row * 2
    res = {}
    rng = np.random.default_rng(2048)
    for B in pa.BLOCK_SIZES:
        nblk = tokens // B
        gk = [x[0].view(2 * nblk, num_kv_heads, B, head_dim) for x in dflat]
        gv = [x[1].view(2 * nblk, num_kv_heads, B, head_dim) for x in dflat]
        ck = [x[0].view(nblk, num_kv_heads, B, head_dim) for x in hflat]
        cv = [x[1].view(nblk, num_kv_heads, B, head_dim) for x in hflat]
        host_ids = rng.permutation(nblk)
        out_p = torch.as_tensor(np.stack([rng.choice(2 * nblk, nblk, replace=False), host_ids], 1),
                                device=dev)
        in_p = torch.as_tensor(np.stack([host_ids, rng.choice(2 * nblk, nblk, replace=False)], 1),
                               device=dev)

        def timed(fn):
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            n = max(5, min(args.steps, 50))
            a.record()
            for _ in range(n):
                fn()
            b.record()
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / n

        t_out = timed(lambda: pa.swap_blocks(ck, cv, gk, gv, out_p))
        t_in = timed(lambda: pa.swap_blocks(gk, gv, ck, cv, in_p))
        res[f"b{B}"] = {"blocks_per_layer": nblk, "out_ms": round(t_out, 4),
                        "in_ms": round(t_in, 4), "out_GBps": round(nbytes / t_out / 1e6, 1),
                        "in_GBps": round(nbytes / t_in / 1e6, 1),
                        "in_plus_out_ms": round(t_in + t_out, 4)}
    # reference: the same bytes as one contiguous copy-engine transfer each way
    del dflat, hflat
    torch.cuda.empty_cache()
    dbig = torch.empty(nbytes // 2, dtype=torch.float16, device=dev)
    hbig = torch.empty(nbytes // 2, dtype=torch.float16).pin_memory()

    def timed_copy(dst, src):
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(10):
            dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / 10

    t_d2h = timed_copy(hbig, dbig)
    t_h2d = timed_copy(dbig, hbig)
    ref = {"d2h_ms": round(t_d2h, 4), "h2d_ms": round(t_h2d, 4),
           "d2h_GBps": round(nbytes / t_d2h / 1e6, 1), "h2d_GBps": round(nbytes / t_h2d / 1e6, 1)}
    print(json.dumps({"swap_sweep": f"one {tokens}-token request, {layers} layers, "
                      f"{num_kv_heads} KV heads x {head_dim}, fp16, K and V",
                      "bytes_per_direction": nbytes, "host_memory": "pinned (cudaHostAlloc)",
                      "results": res,
                      "one_contiguous_copy_engine_transfer": ref}), flush=True)


PREFILL_SHAPES = {
    "opt13b": (40, 40, 128, "f16"),
    "gqa": (12, 2, 128, "bf16"),
}


def prefill_flops(cached, new, num_heads, head_dim):
    """Algorithmic FLOPs of causal chunked prefill: new token i of a
    sequence with c cached tokens sees c + i + 1 keys, each costing 2 D for
    q.k and 2 D for p.v, per query head."""
    keys = sum(n * c + n * (n + 1) // 2 for c, n in zip(cached, new))
    return 4 * head_dim * num_heads * keys


PREFILL_BATCHES = {
    # 8 chunks of 512 tokens on cached prefixes up to 1536 (a 4096-token budget)
    "chunks": ([0, 0, 512, 512, 1024, 1024, 1536, 1536], [512] * 8,
               "8 sequences x 512 new tokens on cached prefixes 0..1536 (4096-token budget)"),
    # one 512-token chunk on an 8192-token prefix among 40 fresh 256-token prompts
    "skewed": ([8192] + [0] * 40, [512] + [256] * 40,
               "one 512-token chunk on an 8192-token prefix with 40 fresh 256-token prompts"),
}


def prefill_bench(args, dev):
    """One chunked-prefill step (PREFILL_BATCHES[args.prefill_batch]), heads
    as the named workload; blocks scattered over the pool.  Times the cache
    write of the chunk plus the prefill attention, and the attention alone,
    over back-to-back steps."""
    import torch
    import paged_kv_cache_pa_gb300 as pa
    H, Hkv, D, dtype = PREFILL_SHAPES[args.config]
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    cached, new, batch_desc = PREFILL_BATCHES[args.prefill_batch]
    S = len(new)
    B = args.prefill_block_size
    lens = np.array([c + n for c, n in zip(cached, new)], np.int32)
    qsl = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    rng = np.random.default_rng(4096)
    nbs = [-(-int(L) // B) for L in lens]
    perm = rng.permutation(sum(nbs))
    maxb = max(nbs)
    tables = np.full((S, maxb), -1, np.int32)
    pos = 0
    for s_, n_ in enumerate(nbs):
        tables[s_, :n_] = perm[pos:pos + n_]
        pos += n_
    slots = np.concatenate([tables[s_, np.arange(c, c + n) // B].astype(np.int64) * B +
                            np.arange(c, c + n) % B for s_, (c, n) in enumerate(zip(cached, new))])
    T = int(qsl[-1])
    g = torch.Generator(device=dev).manual_seed(4096)
    kc = torch.randn(sum(nbs), Hkv, B, D, generator=g, device=dev).to(dt)
    vc = torch.randn(sum(nbs), Hkv, B, D, generator=g, device=dev).to(dt)
    q = torch.randn(T, H, D, generator=g, device=dev).to(dt)
    key = torch.randn(T, Hkv, D, generator=g, device=dev).to(dt)
    val = torch.randn(T, Hkv, D, generator=g, device=dev).to(dt)
    out = torch.empty(T, H, D, dtype=torch.float32, device=dev)
    t_d = torch.as_tensor(tables, device=dev)
    q_d = torch.as_tensor(qsl, device=dev)
    l_d = torch.as_tensor(lens, device=dev)
    s_d = torch.as_tensor(slots, device=dev)
    scale = 1.0 / np.sqrt(D)

    ws = torch.empty(max(256, pa.prefill_workspace_size(S, H, Hkv, D, max(new))),
                     dtype=torch.uint8, device=dev)

    def attn():
        pa.prefill_attention(q, kc, vc, t_d, q_d, l_d, max(new), int(lens.max()), scale, out=out,
                             workspace=ws)

    def step():
        pa.cache_write(key, val, kc, vc, s_d)
        attn()

    def timed(fn, n):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n

    n = max(10, min(args.steps, 200))
    ms_step = timed(step, n)
    ms_attn = timed(attn, n)
    flops = prefill_flops(cached, new, H, D)
    peak = None
    try:
        peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"]
    except (OSError, KeyError, ValueError):
        peak = 1900.0
    tf = flops / (ms_attn * 1e-3) / 1e12
    del kc, vc, q, key, val, out, ws
    torch.cuda.empty_cache()
    return {"prefill": args.config,
            "workload": f"chunked prefill: {batch_desc}, {H} query / {Hkv} KV "
                        f"heads, D={D}, {dtype}, block {B}, scattered blocks",
            "steps": n, "algorithmic_tflop": round(flops / 1e12, 4),
            "ms_attention": round(ms_attn, 4), "ms_step": round(ms_step, 4),
            "tflops": round(tf, 1), "peak_tflops": peak,
            "peak_kind": "measured dense bf16 matmul (burst)",
            "frac": round(tf / peak, 4)}


class DecodeStep:
    """Device buffers and the step function of one decode workload: the
    copy-on-write copies (if any), the cache write of each sequence's new
    token, and decode attention over every context."""

    def __init__(self, pa, synthetic, wl, dev, vals=None):
        import torch
        self.pa, self.wl, self.dev = pa, wl, dev
        self.vals = vals if vals is not None else synthetic.make_values(wl, device=dev)
        S, H, Hkv, D = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim
        self.tables = torch.as_tensor(wl.block_tables, device=dev)
        self.lens = torch.as_tensor(wl.context_lens, device=dev)
        self.slots = torch.as_tensor(wl.slot_mapping, device=dev)
        self.pairs = torch.as_tensor(wl.copy_pairs, device=dev) if len(wl.copy_pairs) else None
        self.out = torch.empty(S, H, D, dtype=torch.float32, device=dev)
        self.ws = torch.empty(pa.decode_workspace_size(S, H, Hkv, D, wl.max_context_len),
                              dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # our kernels per step: [copy] + cache write + the attention call's
        # (plan, one or two attention kernels, [merge])
        self.launches = (self.pairs is not None) + 1 + pa.decode_kernel_launches(
            S, H, Hkv, D, wl.max_context_len)

    def __call__(self, ev_a=None, ev_b=None):
        pa, v = self.pa, self.vals
        if self.pairs is not None:
            pa.copy_blocks([v["k_cache"]], [v["v_cache"]], self.pairs, error_word=self.err)
        pa.cache_write(v["key"], v["value"], v["k_cache"], v["v_cache"], self.slots,
                       error_word=self.err)
        if ev_a is not None:
            ev_a.record()
        pa.decode_attention(v["q"], v["k_cache"], v["v_cache"], self.tables, self.lens,
                            self.wl.max_context_len, self.wl.scale, out=self.out,
                            workspace=self.ws, error_word=self.err)
        if ev_b is not None:
            ev_b.record()


def _pct(xs):
    a = np.asarray(xs, np.float64)
    return {"p10": round(float(np.percentile(a, 10)), 4),
            "p50": round(float(np.percentile(a, 50)), 4),
            "p90": round(float(np.percentile(a, 90)), 4)}


def l2_size(dev):
    import torch
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (126 << 20)


def time_decode(step, K, warmup, dev, dist=None, no_graph=False, sampler=None, windows=10):
    """Time K steps of ``step`` (a DecodeStep).

    K/V far above L2: the K steps run back to back between two events (a
    CUDA graph of up to 50 steps or eager launches, whichever a short sample
    finds faster); ``windows`` more K-step windows give the spread.  K/V
    within four L2 sizes: every step is timed alone between its own events
    after an L2 flush (a read of twice the L2), and the spread is over those
    K steps; the same steps back to back are the hot-L2 figure.  Also the
    attention call alone, eager, an event pair around each call."""
    import torch
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(warmup):
        step()
    barrier()
    assert int(step.err.item()) == 0, f"device error word {int(step.err.item())}"

    g_steps = max(d for d in range(1, min(K, 50) + 1) if K % d == 0)
    timed_graph, timed_launch = None, "eager"
    if not no_graph:
        try:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                for _ in range(g_steps):
                    step()
            g_.replay()
            torch.cuda.synchronize(dev)
            timed_graph, timed_launch = g_, f"CUDA graph of {g_steps} steps"
        except Exception as exc:  # capture not possible here: eager launches
            timed_graph = None
            timed_launch = f"eager (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize(dev)
    if timed_graph is not None:
        # keep whichever launch method runs this step faster: graph replay
        # saves the host's launch overhead, eager launches keep every
        # programmatic overlap between the kernels
        def sample(fn, n):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            a_.record(stream)
            for _ in range(n):
                fn()
            b_.record(stream)
            barrier()
            return a_.elapsed_time(b_) / n
        reps = max(1, 200 // g_steps)
        t_graph = reduce_max(sample(timed_graph.replay, reps) / g_steps, dist, dev)
        t_eager = reduce_max(sample(step, reps * g_steps), dist, dev)
        if t_eager <= t_graph:
            timed_graph = None
            timed_launch = f"eager (faster than a CUDA graph of {g_steps} steps here)"
        else:
            timed_launch += " (faster than eager launches here)"

    # K steps back to back, events only at the two ends (an event between two
    # kernels would cut their programmatic overlap)
    def back_to_back():
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        barrier()
        t_start.record(stream)
        if timed_graph is not None:
            for _ in range(K // g_steps):
                timed_graph.replay()
        else:
            for _ in range(K):
                step()
        t_end.record(stream)
        barrier()
        return reduce_max(t_start.elapsed_time(t_end), dist, dev)

    l2_bytes = l2_size(dev)
    near_l2 = step.wl.kv_bytes() < 4 * l2_bytes
    if near_l2:
        flush_buf = torch.ones(l2_bytes, dtype=torch.float16, device=dev)  # 2 x L2 bytes
        one_step = None
        try:
            one_step = torch.cuda.CUDAGraph()
            with torch.cuda.graph(one_step):
                step()
            one_step.replay()
            torch.cuda.synchronize(dev)
        except Exception:  # capture not possible here: eager launches
            one_step = None
            torch.cuda.synchronize(dev)
        run_one = one_step.replay if one_step is not None else step
        for _ in range(3):
            flush_buf.sum()
            run_one()

    if sampler:
        sampler.start()
    barrier()
    wall0 = time.time()
    per_step = None
    if near_l2:
        ca = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        cb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            flush_buf.sum()
            ca[i].record(stream)
            run_one()
            cb[i].record(stream)
        barrier()
        per_step = [a.elapsed_time(b) for a, b in zip(ca, cb)]
        total_ms = reduce_max(sum(per_step), dist, dev)
        timed_launch = ("each step timed alone after an L2 flush, " +
                        ("a CUDA graph of one step" if one_step is not None else "eager launches"))
    else:
        total_ms = back_to_back()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1) if sampler else None
    if near_l2:
        spread = dict(_pct(per_step), over=f"the {K} timed steps (ms per step)")
        hot_ms = back_to_back()
        hot = {"ms_per_step": round(hot_ms / K, 4), "launch": "back to back, " + (
            f"CUDA graph of {g_steps} steps" if timed_graph is not None else "eager")}
        del flush_buf
    else:
        wins = [total_ms / K] + [back_to_back() / K for _ in range(windows)]
        spread = dict(_pct(wins), over=f"{len(wins)} windows of {K} steps back to back "
                                       f"(ms per step; the first is the timed region)")
        hot = None
    # the attention call timed alone: K more eager steps with an event pair
    # around every call (each call then also waits for the host to submit its
    # launches)
    evs_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    evs_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        step(evs_a[i], evs_b[i])
    barrier()
    attn_ms = sum(a.elapsed_time(b) for a, b in zip(evs_a, evs_b)) / K
    assert int(step.err.item()) == 0, f"device error word {int(step.err.item())}"
    return {"ms_per_step": total_ms / K, "launch": timed_launch, "near_l2": near_l2,
            "l2_bytes": l2_bytes, "hot": hot, "spread": spread, "attn_ms": attn_ms,
            "clocks": clocks, "graph": timed_graph, "g_steps": g_steps}


def cpu_baseline(wl, vals, dev, core_seconds=10.0, max_bytes=0.6e9, max_reps=50):
    """The oracle (plain C, fp64, all host cores) on the same device inputs:
    all of the batch's sequences if their K/V fit ``max_bytes``, else a
    seeded subset that does; passes repeat until ~``core_seconds`` of CPU
    work."""
    import torch
    import oracle
    oracle.build()
    S = wl.num_seqs
    per = wl.context_lens.astype(np.int64) * wl.num_kv_heads * wl.head_dim * 4
    order = np.random.default_rng(0).permutation(S)
    keep = order[np.cumsum(per[order]) <= max_bytes]
    seqs = np.sort(keep if len(keep) else order[:1])
    q_h = vals["q"].view(torch.int16).cpu().numpy().view(np.uint16)

    def host_vals(sq, used):
        idx = torch.as_tensor(np.asarray(used, np.int64), device=dev)
        kc, vc = (vals[n].index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
                  for n in ("k_cache", "v_cache"))
        return q_h[sq], kc, vc
    inputs = oracle_inputs(wl, seqs, host_vals=host_vals)
    threads = oracle.default_threads()
    t_cpu = b_cpu = 0.0
    reps = 0
    while reps < 1 or (t_cpu * threads < core_seconds and reps < max_reps):
        t_cpu += oracle_time(wl, inputs, threads)
        b_cpu += inputs[5]
        reps += 1
    what = (f"all {S} sequences of the batch" if len(seqs) == S else
            f"{len(seqs)} of the batch's {S} sequences (seeded choice)")
    return {"value": round(b_cpu / t_cpu / 1e9, 4), "unit": UNIT, "cores": threads,
            "kind": "oracle", "seconds": round(t_cpu, 2),
            "sample": f"{what}, attention only, {reps} pass(es)"}


def step_numbers(wl, t, peak, world=1):
    """Throughput figures of one timed workload."""
    b_attn, b_write, b_copy = algorithmic_bytes(wl)
    b_attn_logical = algorithmic_bytes(wl, shared_once=False)[0]
    b_step = b_attn + b_write + b_copy
    ms = t["ms_per_step"]
    value = world * b_step / (ms * 1e-3) / 1e9
    attn_gbs = b_attn / (ms * 1e-3) / 1e9
    d = {"b_attn": b_attn, "b_write": b_write, "b_copy": b_copy, "b_step": b_step,
         "value": value, "attn_gbs": attn_gbs, "frac": attn_gbs / peak,
         "attn_gbs_isolated": b_attn / (t["attn_ms"] * 1e-3) / 1e9,
         "logical": ({"attention_bytes": int(b_attn_logical),
                      "GBps": round(world * (b_attn_logical + b_write + b_copy) /
                                    (ms * 1e-3) / 1e9, 2)}
                     if b_attn_logical != b_attn else None)}
    return d


def l2_note(t):
    if not t["near_l2"]:
        return "inputs larger than L2 (K/V read per step >> 126 MB L2)"
    return (f"K/V per step within a few L2 sizes: an L2 flush (a read of "
            f"{2 * t['l2_bytes'] >> 20} MiB) before every timed step; hot_l2 = the same "
            f"steps back to back")


def cow_copy_timing(pa, wl, dev, layer_counts=(1, 40), reps=20):
    """The workload's copy-on-write pairs as one pa_copy_blocks launch over 1
    and over 40 layers.  Each layer gets its own pool holding just the
    blocks the pairs name (relabelled), so 40 layers fit in memory; every
    timed call follows an L2 flush."""
    import torch
    pairs = np.asarray(wl.copy_pairs, np.int64)
    if not len(pairs):
        return None
    ids = np.unique(pairs)
    rel = np.searchsorted(ids, pairs)
    Hkv, D, B = wl.num_kv_heads, wl.head_dim, wl.block_size
    dt = torch.float16 if wl.dtype == "f16" else torch.bfloat16
    L = max(layer_counts)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    kc = [torch.randn(len(ids), Hkv, B, D, generator=g, device=dev).to(dt) for _ in range(L)]
    vc = [torch.randn(len(ids), Hkv, B, D, generator=g, device=dev).to(dt) for _ in range(L)]
    p_d = torch.as_tensor(rel, device=dev)
    flush = torch.ones(l2_size(dev), dtype=torch.float16, device=dev)
    res = {"pairs": int(len(pairs))}
    for n in layer_counts:
        for _ in range(3):
            pa.copy_blocks(kc[:n], vc[:n], p_d)
        torch.cuda.synchronize(dev)
        a = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        b = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        for i in range(reps):
            flush.sum()
            a[i].record()
            pa.copy_blocks(kc[:n], vc[:n], p_d)
            b[i].record()
        torch.cuda.synchronize(dev)
        ms = sum(x.elapsed_time(y) for x, y in zip(a, b)) / reps
        nbytes = 2 * len(pairs) * n * Hkv * B * D * 2 * 2      # read + write, K and V
        res[f"layers_{n}"] = {"ms": round(ms, 4), "bytes": int(nbytes),
                              "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    del kc, vc, flush
    torch.cuda.empty_cache()
    return res


def measure_config(name, args, pa, synthetic, dev, peak, rank=0, cpu=True):
    """One workload's entry of the bench line's per_config object."""
    import torch
    wl = synthetic.make(name, seed=synthetic.SEEDS[name] + 100 * rank)
    step = DecodeStep(pa, synthetic, wl, dev)
    t = time_decode(step, args.steps, args.warmup, dev, no_graph=args.no_graph)
    n = step_numbers(wl, t, peak)
    entry = {
        "workload": WORKLOADS[name], "ms_per_step": round(t["ms_per_step"], 4),
        "value": round(n["value"], 2), "unit": UNIT,
        "seqs_per_s_per_layer": round(wl.num_seqs / (t["ms_per_step"] * 1e-3), 1),
        "launch": t["launch"], "l2": l2_note(t), "spread": t["spread"], "hot_l2": t["hot"],
        "roofline": {"bound": "hbm", "achieved": round(n["attn_gbs"], 2), "peak": peak,
                     "unit": "GB/s", "frac": round(n["frac"], 4),
                     "traffic": recorded_traffic(name),
                     "algorithmic_bytes": int(n["b_attn"]),
                     "isolated_call": {"ms_per_call": round(t["attn_ms"], 4),
                                       "achieved": round(n["attn_gbs_isolated"], 2)}},
        "logical": n["logical"],
        "pct_of_spec_8000": round(100 * n["attn_gbs"] / 8000.0, 2),
    }
    if t["hot"] is not None:
        entry["hot_l2"]["value"] = round(n["b_step"] / (t["hot"]["ms_per_step"] * 1e-3) / 1e9, 2)
        entry["hot_l2"]["frac"] = round(n["b_attn"] / (t["hot"]["ms_per_step"] * 1e-3) / 1e9
                                        / peak, 4)
    if name == "beams":
        entry["cow_copy"] = cow_copy_timing(pa, wl, dev)
    if name == "tiny":
        # the same chain of kernels on one sequence of one token: the floor
        # a launch-bound step is measured against
        rng = np.random.default_rng(7)
        fw = synthetic._from_lengths("floor", [1], 8, 8, 64, "f16", 7, rng)
        fstep = DecodeStep(pa, synthetic, fw, dev)
        ft = time_decode(fstep, args.steps, args.warmup, dev, no_graph=args.no_graph)
        entry["floor"] = {"ms_per_step": round(ft["ms_per_step"], 4),
                          "hot_ms_per_step": ft["hot"]["ms_per_step"] if ft["hot"] else None,
                          "what": "one sequence of one token (8 heads, D=64): the same "
                                  "kernel chain with almost no work, timed the same way"}
        del fstep
    if cpu:
        entry["cpu_baseline"] = cpu_baseline(wl, step.vals, dev, core_seconds=6.0)
    del step, t
    torch.cuda.empty_cache()
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="opt13b")
    ap.add_argument("--seqs", type=int, default=0,
                    help="batch size override (smaller cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the steps eagerly instead of replaying a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the named workload (no per_config object)")
    ap.add_argument("--layout-sweep", action="store_true",
                    help="time the attention call with blocks scattered, blocks in order, and "
                         "on a contiguous (unpaged) cache; prints its own JSON line")
    ap.add_argument("--prefill", action="store_true",
                    help="time a chunked-prefill step (8 x 512 new tokens) with the named "
                         "workload's heads; prints its own JSON line")
    ap.add_argument("--prefill-block-size", type=int, default=16,
                    help="tokens per block for --prefill (8 .. 256)")
    ap.add_argument("--prefill-batch", choices=sorted(PREFILL_BATCHES), default="chunks",
                    help="batch for --prefill: 'chunks' (8 x 512 on prefixes up to 1536) or "
                         "'skewed' (one 512-token chunk on an 8192-token prefix among 40 "
                         "fresh 256-token prompts)")
    ap.add_argument("--swap-sweep", action="store_true",
                    help="time swap-out and swap-in of one full-length request over all "
                         "layers at block sizes 8..256; prints its own JSON line")
    ap.add_argument("--block-size-sweep", action="store_true",
                    help="time the attention call with the workload's sequences in blocks of "
                         "8..256 tokens, scattered and in order, against a contiguous cache; "
                         "prints its own JSON line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from paged_kv_cache_pa_gb300 import synthetic
    kw = {"num_seqs": args.seqs} if args.seqs else {}
    wl = synthetic.make(args.config, seed=synthetic.SEEDS[args.config] + 100 * rank, **kw)

    if args.impl == "reference":
        run_reference(args, wl, rank, world)
        return

    import torch
    import paged_kv_cache_pa_gb300 as pa
    from paged_kv_cache_pa_gb300.build import build
    build()
    pa.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.layout_sweep:
        print(json.dumps(layout_sweep(args, wl, dev)), flush=True)
        return
    if args.block_size_sweep:
        block_size_sweep(args, wl, dev)
        return
    if args.swap_sweep:
        swap_sweep(args, dev)
        return
    if args.prefill:
        print(json.dumps(prefill_bench(args, dev)), flush=True)
        return

    peak, peak_kind = peaks()
    step = DecodeStep(pa, synthetic, wl, dev)
    vals = step.vals
    S, H, Hkv, D = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim
    K = args.steps
    sampler = ClockSampler(local_rank) if rank == 0 or world > 1 else None
    t = time_decode(step, K, args.warmup, dev, dist=dist, no_graph=args.no_graph,
                    sampler=sampler)
    ms_per_step = t["ms_per_step"]
    n = step_numbers(wl, t, peak, world)
    b_attn, b_write, b_copy, b_step = n["b_attn"], n["b_write"], n["b_copy"], n["b_step"]
    value = n["value"]
    hot = t["hot"]
    if hot is not None:
        hot["value"] = round(world * b_step / (hot["ms_per_step"] * 1e-3) / 1e9, 2)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # end to end through the Python API: every step's inputs go host -> device
    # in one copy from a pinned staging buffer and its output comes back to
    # pinned host memory, the copies of neighbouring steps overlapping the
    # compute as a serving loop would; the KV pools are the cache and stay
    # resident
    e2e = None
    if not args.no_e2e:
        pairs = step.pairs
        ws = step.ws
        host_parts = [vals["q"].cpu(), vals["key"].cpu(), vals["value"].cpu(),
                      torch.as_tensor(wl.slot_mapping), torch.as_tensor(wl.block_tables),
                      torch.as_tensor(wl.context_lens)]
        offs, total = [], 0
        for x in host_parts:
            offs.append(total)
            total += (x.numel() * x.element_size() + 255) // 256 * 256
        staging = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for x, o in zip(host_parts, offs):
            nb = x.numel() * x.element_size()
            staging[o:o + nb].copy_(x.contiguous().view(-1).view(torch.uint8))
        h2d = int(total)
        d2h = S * H * D * 4

        # Two sets of device inputs and outputs: step i+1's inputs go host ->
        # device and step i-1's output device -> host on a copy stream while
        # step i computes; events order the reuse of each buffer.
        copy_stream = torch.cuda.Stream(dev)
        hout = [torch.empty(S, H, D, dtype=torch.float32).pin_memory() for _ in range(2)]
        outs = [torch.empty(S, H, D, dtype=torch.float32, device=dev) for _ in range(2)]
        bufs, views = [], []
        for _ in range(2):
            b_ = torch.empty(total, dtype=torch.uint8, device=dev)
            bufs.append(b_)
            views.append([b_[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
                          for x, o in zip(host_parts, offs)])
        ev = lambda: torch.cuda.Event()
        h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def pipeline(n_steps):
            # step i's inputs and step i-1's output move on the copy stream
            # while step i computes on `stream`
            cs = torch.cuda.current_stream(dev)
            for i in range(n_steps + 1):
                b = i % 2
                if i < n_steps:
                    with torch.cuda.stream(copy_stream):
                        if i >= 2:
                            copy_stream.wait_event(comp_done[b])   # step i-2 read bufs[b]
                        bufs[b].copy_(staging, non_blocking=True)
                        h2d_done[b].record(copy_stream)
                    cs.wait_event(h2d_done[b])
                    if i >= 2:
                        cs.wait_event(d2h_done[b])                  # outs[b] read back
                    q_d, k_d, v_d, s_d, t_d, l_d = views[b]
                    if pairs is not None:
                        pa.copy_blocks([vals["k_cache"]], [vals["v_cache"]], pairs)
                    pa.cache_write(k_d, v_d, vals["k_cache"], vals["v_cache"], s_d)
                    pa.decode_attention(q_d, vals["k_cache"], vals["v_cache"], t_d, l_d,
                                        wl.max_context_len, wl.scale, out=outs[b], workspace=ws)
                    comp_done[b].record(cs)
                if i >= 1:  # the previous step's result back to the host
                    pb = (i - 1) % 2
                    with torch.cuda.stream(copy_stream):
                        copy_stream.wait_event(comp_done[pb])
                        hout[pb].copy_(outs[pb], non_blocking=True)
                        d2h_done[pb].record(copy_stream)

        def e2e_steps(n_steps, t_start=None, t_end=None):
            stream.synchronize()
            if t_start is not None:
                t_start.record(copy_stream)
            pipeline(n_steps)
            if t_end is not None:
                t_end.record(copy_stream)
            copy_stream.synchronize()
            stream.synchronize()

        # Short steps are bound by the host's launch overhead: capture 25
        # pipelined steps (the same public calls and copies) in a CUDA graph
        # and replay it; fall back to the eager loop if capture fails.
        kg = 25
        graph, launch = None, "eager"
        if not args.no_graph:
            try:
                e2e_steps(3)
                g_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_):
                    cap = torch.cuda.current_stream(dev)
                    copy_stream.wait_stream(cap)
                    pipeline(kg)
                    cap.wait_stream(copy_stream)
                g_.replay()
                torch.cuda.synchronize(dev)
                graph, launch = g_, f"CUDA graph of {kg} pipelined steps"
            except Exception as exc:  # capture not possible here: eager loop
                graph = None
                launch = f"eager (graph capture failed: {type(exc).__name__})"
                torch.cuda.synchronize(dev)
        # time the eager pipeline, and the graph replay if capture worked,
        # and keep the faster (both copy every step's inputs and output)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2e_steps(3)
        barrier()
        e2e_steps(args.e2e_steps, e0, e1)
        barrier()
        n_e2e = args.e2e_steps
        e_ms_eager = reduce_max(e0.elapsed_time(e1) / n_e2e, dist, dev)
        eager_label = launch if graph is None else "eager"
        best = (e_ms_eager, eager_label, n_e2e)
        if graph is not None:
            reps = max(1, args.e2e_steps // kg)
            for _ in range(3):
                graph.replay()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            barrier()
            g0.record(stream)
            for _ in range(reps):
                graph.replay()
            g1.record(stream)
            barrier()
            e_ms_graph = reduce_max(g0.elapsed_time(g1) / (reps * kg), dist, dev)
            if e_ms_graph < e_ms_eager:
                best = (e_ms_graph, launch + " (faster than eager launches here)", reps * kg)
            else:
                best = (e_ms_eager, f"eager (faster than a {launch} here)", n_e2e)
        e_ms, launch, n_e2e = best
        e2e = {"value": round(world * b_step / (e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e_ms, 4), "steps": n_e2e, "launch": launch}
        if t["near_l2"]:
            e2e["l2"] = "steps back to back, no L2 flush (hot)"
        del graph, bufs, views, outs

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, vals, dev, max_bytes=2.5e9)
    launches = int(K * step.launches)
    del step, vals
    t.pop("graph", None)
    torch.cuda.empty_cache()

    # every other workload, the prefill step and the paged/contiguous ratio,
    # measured the same way on this GPU (rank 0 only: one replica suffices)
    per_config = None
    if rank == 0 and not args.no_per_config and not args.seqs:
        per_config = {}
        for name in ("gqa", "long", "beams", "tiny"):
            if name != args.config:
                per_config[name] = measure_config(name, args, pa, synthetic, dev, peak,
                                                  cpu=not args.no_cpu_baseline)
        pf = {}
        for heads in ("opt13b", "gqa"):
            pargs = argparse.Namespace(**{**vars(args), "config": heads, "prefill_batch": "chunks",
                                          "prefill_block_size": 16})
            pf[heads] = prefill_bench(pargs, dev)
        per_config["prefill"] = pf
        largs = argparse.Namespace(**{**vars(args), "config": "opt13b"})
        lay = layout_sweep(largs, synthetic.make("opt13b"), dev)
        per_config["layout_b16_opt13b"] = {
            "time_vs_contiguous": {k: v["time_vs_contiguous"] for k, v in lay["results"].items()},
            "ms_per_call": {k: v["ms_per_call"] for k, v in lay["results"].items()},
            "what": "the attention call alone, back to back, paged with 16-token blocks "
                    "scattered or in order, against the same kernels on a contiguous cache"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic",
        "config": {"workload": WORKLOADS.get(args.config, args.config) +
                               (f" (cut to {S} sequences)" if args.seqs else ""),
                   "mean_context": round(float(wl.context_lens.mean()), 1),
                   "kv_bytes_per_step": int(wl.kv_bytes()),
                   "l2": l2_note(t),
                   "parallelism": f"replicas x{world}", "launch": t["launch"]},
        "seqs_per_s_per_layer": round(world * S / (ms_per_step * 1e-3), 1),
        # blocks shared by several sequences (copy-on-write prefixes) are
        # counted once above; here once per sequence that reads them
        "logical": n["logical"],
        "spread": t["spread"],
        "pct_of_peak": {"measured_copy": round(100 * value / world / peak, 2),
                        "spec_8000": round(100 * value / world / 8000.0, 2)},
        "roofline": {"bound": "hbm", "achieved": round(n["attn_gbs"], 2), "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy GB/s (reads + writes; a read-only "
                                  f"stream such as decode can exceed it, so frac is against a "
                                  f"lower bound of the read peak)",
                     "unit": "GB/s", "frac": round(n["frac"], 4),
                     "frac_of_spec_8000": round(n["attn_gbs"] / 8000.0, 4),
                     # the recorded figure is for the full-size batch
                     "traffic": None if args.seqs else recorded_traffic(args.config),
                     "kernel": "pa_decode_attention (plan, attention and merge kernels)",
                     "duration": "timed-region step time (cache write + attention call"
                                 + (" + copy-on-write copies" if b_copy else "") + ")",
                     "ms": round(ms_per_step, 4), "algorithmic_bytes": int(b_attn),
                     "isolated_call": {"ms_per_call": round(t["attn_ms"], 4),
                                       "achieved": round(n["attn_gbs_isolated"], 2),
                                       "how": "eager, an event pair around each call" +
                                              (", no L2 flush" if t["near_l2"] else "")}},
        "hot_l2": hot,
        "gpu_launches": launches,
        "clocks": t["clocks"],
        "e2e": e2e,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
