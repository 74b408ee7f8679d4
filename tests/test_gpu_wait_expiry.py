"""The give-up path of the kernels' bounded waits, run on the GPU.

Every wait inside the attention kernels (a ring stage, a hand-off buffer, a
tensor-core result) is bounded: when it runs out, the CTA raises its abort
flag, ORs PA_ERRBIT_TIMEOUT into the error word, lets its own copies and
tensor-core work in flight finish, and returns.  On a healthy GPU no wait
ever runs out, so a test copy of the library is built whose ordinary waits
give up after a few non-blocking polls (libpa_gb300_shortwait.so; the waits
for a CTA's own work in flight keep their full limits).

An ordinary call through that copy must return PA_OK and report the
timeout bit, and the GPU must keep answering: the child process that made
the call runs a torch computation afterwards, and the next call through the
product library, in this process, matches the oracle.  The test copy runs in
a child process of its own because each library links its own copy of the
CUDA runtime, and a process should load only one of them.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

from paritylib import (ATOL, custom_workload, host_inputs, max_abs, prefill_oracle,  # noqa: E402
                       prefill_problem, prefill_run, shared_workload)

pytestmark = pytest.mark.gpu

DECODE_CASES = ["cuda_cores", "tensor_cores", "tensor_cores_no_plan", "shared_prefix"]
PREFILL_CASES = {"prefill_f16": (8, 8, 128, "f16"), "prefill_bf16": (12, 2, 128, "bf16")}
PREFILL_CHUNKS = [(0, 200), (300, 130), (37, 64), (0, 1)]


def _decode_workload(case):
    from paged_kv_cache_pa_gb300 import synthetic
    if case == "cuda_cores":       # G = 1: the CUDA-core kernel
        return synthetic.make("tiny", num_seqs=16)
    if case == "tensor_cores":     # G = 6: the tensor-core kernel, several partitions
        return custom_workload([700, 1500, 33, 4000, 900, 2], 12, 2, 128, "bf16")
    if case == "tensor_cores_no_plan":  # G = 6, a batch small enough to skip the plan
        return custom_workload([40, 90, 7, 200, 0, 150], 12, 2, 128, "bf16")
    # G = 1 with shared prefixes: both attention kernels in one call
    return shared_workload([900, 950, 990, 400, 1300], [0, 50, 50, 0, 20], 4, 4, 128, "f16")


def _decode(pa, wl, vals, err):
    dev = vals["q"].device
    tables = torch.as_tensor(wl.block_tables, device=dev)
    lens = torch.as_tensor(wl.context_lens, device=dev)
    return pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                               wl.max_context_len, wl.scale, error_word=err)


def _child(case, lib_path):
    """In a fresh process: one call through the short-wait library, then a
    torch computation on the same GPU; prints the error word as JSON."""
    import paged_kv_cache_pa_gb300 as pa
    from paged_kv_cache_pa_gb300 import synthetic
    pa._LIB_PATH = lib_path                 # this process loads only the test copy
    dev = torch.device("cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if case in PREFILL_CASES:
        H, Hkv, D, dtype = PREFILL_CASES[case]
        d = prefill_problem(PREFILL_CHUNKS, H, Hkv, D, dtype, 16, seed=11)
        prefill_run(d, 1.0 / np.sqrt(D), err=err)
    else:
        wl = _decode_workload(case)
        _decode(pa, wl, synthetic.make_values(wl, device=dev), err)
    torch.cuda.synchronize()
    a = torch.randn(256, 256, device=dev)
    ok = bool(torch.allclose(a @ torch.eye(256, device=dev), a))
    print(json.dumps({"err": int(err.item()), "gpu_answers": ok}), flush=True)


def _run_child(case):
    from paged_kv_cache_pa_gb300.build import build
    lib = build(variant="shortwait")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), case, lib],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("case", DECODE_CASES)
def test_decode_waits_give_up_then_the_next_call_is_right(case):
    if not torch.cuda.is_available():  # pragma: no cover
        pytest.skip("needs a CUDA device")
    res = _run_child(case)
    assert res["err"] & 8, res          # PA_ERRBIT_TIMEOUT
    assert res["gpu_answers"]
    import oracle
    import paged_kv_cache_pa_gb300 as pa
    from paged_kv_cache_pa_gb300 import synthetic
    dev = torch.device("cuda:0")
    wl = _decode_workload(case)
    vals = synthetic.make_values(wl, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = _decode(pa, wl, vals, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    h = host_inputs(wl, vals)
    want = oracle.decode_attention(h["q"], h["k_cache"], h["v_cache"], h["tables"],
                                   wl.context_lens, wl.scale, wl.dtype)
    assert max_abs(out.cpu().numpy(), want) <= ATOL


@pytest.mark.parametrize("case", sorted(PREFILL_CASES))
def test_prefill_waits_give_up_then_the_next_call_is_right(case):
    if not torch.cuda.is_available():  # pragma: no cover
        pytest.skip("needs a CUDA device")
    res = _run_child(case)
    assert res["err"] & 8, res          # PA_ERRBIT_TIMEOUT
    assert res["gpu_answers"]
    H, Hkv, D, dtype = PREFILL_CASES[case]
    scale = 1.0 / np.sqrt(D)
    d = prefill_problem(PREFILL_CHUNKS, H, Hkv, D, dtype, 16, seed=11)
    err = torch.zeros(1, dtype=torch.int32, device=torch.device("cuda:0"))
    out = prefill_run(d, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max_abs(out.cpu().numpy(), prefill_oracle(d, scale, dtype)) <= ATOL


if __name__ == "__main__":
    _child(sys.argv[1], sys.argv[2])
