"""The PA_DEBUG build of the library, run on the GPU.

build(variant="debug") compiles the library with -DPA_DEBUG and -DPA_NVTX.
The decode kernels then check every work item the plan hands them: a real
sequence, a token range inside its context (inside every member's context
for a shared-prefix item), and a partition slot that exists.  The merge
kernel checks every partition count.  Whatever fails is reported as
PA_ERRBIT_INTERNAL and skipped.  Every C-ABI compute call is also an NVTX
range.

On correct plans nothing may fail.  Each case runs a whole decode step
through that library: the copy-on-write copies, the cache write and
attention.  The step must leave the error word 0 and match the oracle.  The
cases cover the CUDA-core and tensor-core kernels, with the plan and
without it (small batches), partitions, shared prefixes, 8-token blocks and
every head size.

The library runs in a child process of its own.  Each library links its own
copy of the CUDA runtime, so a process loads only one of them.
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

pytestmark = pytest.mark.gpu

CASES = ["gqa_partitions", "g1_cuda_cores", "gqa_no_plan", "shared_prefix", "beams", "block8",
         "d64", "d256"]


def _workload(case):
    from paged_kv_cache_pa_gb300 import synthetic
    from paritylib import custom_workload, shared_workload
    if case == "gqa_partitions":   # G = 6, tensor cores, several partitions
        return custom_workload([700, 1500, 33, 4000, 900, 2], 12, 2, 128, "bf16")
    if case == "g1_cuda_cores":    # G = 1, CUDA cores, no plan (a small batch)
        return synthetic.make("tiny", num_seqs=16)
    if case == "gqa_no_plan":      # G = 6 on the tensor cores, no plan, an empty sequence
        return custom_workload([40, 90, 7, 200, 0, 150], 12, 2, 128, "bf16")
    if case == "shared_prefix":    # G = 1 with shared prefixes: both kernels
        return shared_workload([900, 950, 990, 400, 1300], [0, 50, 50, 0, 20], 4, 4, 128, "f16")
    if case == "beams":            # copy-on-write copies and shared prompts
        return synthetic.make("beams", groups=3, beams=4, num_heads=8)
    if case == "block8":           # 8-token blocks on the tensor-core path
        return synthetic.relayout(custom_workload([300, 1000, 77], 8, 2, 128, "f16"), 8)
    if case == "d64":
        return custom_workload([600, 1200, 5], 16, 2, 64, "bf16")
    return custom_workload([900, 40, 1], 4, 4, 256, "f16")   # d256


def _child(lib_path):
    """In a fresh process: every case through the debug library; prints one
    JSON line per case with the error word and the max |gpu - oracle|."""
    import paged_kv_cache_pa_gb300 as pa
    from paged_kv_cache_pa_gb300 import synthetic
    from paritylib import gpu_step, host_inputs, max_abs, oracle_step, step_blocks
    pa._LIB_PATH = lib_path           # this process loads only the debug library
    dev = torch.device("cuda:0")
    for case in CASES:
        wl = _workload(case)
        vals = synthetic.make_values(wl, device=dev)
        h = host_inputs(wl, vals, step_blocks(wl))
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        out = gpu_step(wl, vals, error_word=err)
        torch.cuda.synchronize()
        want = oracle_step(wl, h)
        print(json.dumps({"case": case, "err": int(err.item()),
                          "max_abs": max_abs(out.cpu().numpy(), want)}), flush=True)


def _results():
    from paged_kv_cache_pa_gb300.build import build
    lib = build(variant="debug")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), lib],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    rows = [json.loads(x) for x in r.stdout.strip().splitlines() if x.startswith("{")]
    return {row["case"]: row for row in rows}


_CACHE = {}


@pytest.mark.parametrize("case", CASES)
def test_debug_build_checks_pass_and_match_the_oracle(case):
    if not torch.cuda.is_available():  # pragma: no cover
        pytest.skip("needs a CUDA device")
    if "rows" not in _CACHE:
        _CACHE["rows"] = _results()
    from paritylib import ATOL
    row = _CACHE["rows"][case]
    assert row["err"] == 0, row        # no check failed, no block or slot out of range
    assert row["max_abs"] <= ATOL, row


if __name__ == "__main__":
    _child(sys.argv[1])
