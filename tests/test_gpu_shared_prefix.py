"""GPU parity for shared prefixes: runs of consecutive sequences whose block
tables start with the same block ids (beam search, parallel sampling, a
common system prompt).  The plan reads such a prefix once for the whole run
(one item whose query rows are every member's queries) and each sequence's
own remainder separately; the result must still be each sequence's own
attention, so every case is compared with the CPU oracle, which knows
nothing of sharing.

Tables are built so that sharing forms, breaks and re-forms: a sequence
copies a chosen number of leading block ids from the sequence before it and
takes fresh blocks for the rest (which may again equal ids further on)."""
import numpy as np
import pytest
import torch

from paritylib import ATOL, gpu_step, host_inputs, max_abs, oracle_step, shared_workload

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped
    pytest.skip("needs a CUDA device", allow_module_level=True)

from paged_kv_cache_pa_gb300 import synthetic  # noqa: E402

DEV = torch.device("cuda:0")


def _check(wl, poison=True):
    vals = synthetic.make_values(wl, device=DEV, poison_unused=poison)
    h = host_inputs(wl, vals)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    # decode attention only: the new tokens' slots may sit in shared blocks
    # (this test is about reading, not copy-on-write), so no cache write
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    import paged_kv_cache_pa_gb300 as pa
    out = pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                              wl.max_context_len, wl.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    import oracle
    want = oracle.decode_attention(h["q"], h["k_cache"], h["v_cache"], h["tables"],
                                   wl.context_lens, wl.scale, wl.dtype)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert max_abs(got, want) <= ATOL
    return got, want


@pytest.mark.parametrize("H, Hkv, D, dtype", [
    (4, 4, 128, "f16"),      # G = 1: shared prefixes on the tensor-core kernel, the rest on CUDA cores
    (4, 4, 64, "bf16"),
    (8, 4, 128, "bf16"),     # G = 2: runs of up to 4
    (6, 2, 128, "f16"),      # G = 3: runs of up to 2 (6 query rows)
    (8, 2, 64, "f16"),       # G = 4: runs of up to 2
    (12, 2, 128, "bf16"),    # G = 6: no shared-prefix items (plain path)
])
def test_beam_like_runs(H, Hkv, D, dtype):
    rng = np.random.default_rng(H * 100 + D)
    lens, share = [], []
    for g in range(5):                                  # 5 prompts x 6 beams
        prompt = int(rng.integers(100, 700))
        for b in range(6):
            lens.append(prompt + int(rng.integers(1, 200)))
            share.append(0 if b == 0 else prompt // 16)
    _check(shared_workload(lens, share, H, Hkv, D, dtype))


@pytest.mark.parametrize("B", [8, 16, 64])
def test_sharing_forms_breaks_and_reforms(B):
    # runs of 11 (longer than one group), 1, 3; shares below the minimum; a
    # member whose whole context is the shared prefix; an empty sequence
    # between runs; ids equal again after the first differing block
    lens = [900, 901, 1200, 640, 700, 777, 1000, 1001, 1002, 1003, 999,
            300,
            0,
            513, 512, 800,
            60, 60,
            1500, 1490]
    share = [0, 56, 56, 40, 40, 43, 43, 62, 62, 62, 62,
             5,
             0,
             0, 32, 32,
             0, 3,
             0, 90]
    share = [c * 16 // B for c in share]                # the same tokens at any block size
    wl = shared_workload(lens, share, 4, 4, 128, "f16", B=B, reuse_later=True)
    _check(wl)


def test_long_shared_prefix_spans_several_partitions():
    # few sequences -> small partitions: the shared prefix is many pieces
    lens = [2000, 2100, 1990, 2500, 2048, 2049]
    share = [0, 100, 100, 124, 124, 128]
    wl = shared_workload(lens, share, 4, 4, 128, "bf16")
    _check(wl)


def test_every_sequence_shares_everything():
    # identical tables and lengths: each result is its own query's attention
    # over the same keys
    lens = [777] * 8
    share = [0] + [49] * 7
    wl = shared_workload(lens, share, 8, 8, 128, "f16")
    got, _ = _check(wl)


def test_shared_prefix_step_with_copy_on_write():
    """The beam workload's full step: copy-on-write copies, the cache write
    and attention, against the oracle's step on the same inputs."""
    wl = synthetic.make("beams", groups=6)
    vals = synthetic.make_values(wl, device=DEV)
    h = host_inputs(wl, vals)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gpu_step(wl, vals, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle_step(wl, h)
    assert max_abs(out.cpu().numpy(), want) <= ATOL


@pytest.mark.parametrize("H, Hkv, D, dtype", [(8, 8, 128, "f16"), (4, 2, 64, "bf16")])
def test_shared_and_unshared_calls_back_to_back_on_one_workspace(H, Hkv, D, dtype):
    """Calls enqueued back to back on one stream and one workspace,
    alternating a batch with shared prefixes and the same sequences cut
    below the sharing threshold (no shared-prefix items: different work
    lists in both of the plan's lists).  With one query head per KV head a
    call runs the tensor-core and the CUDA-core kernel, and the CUDA-core
    kernel reads its list as soon as it launches, without waiting for the
    tensor-core grid, so a stale or early list read would show here.
    Every output must equal the one the same batch gives alone, to the bit;
    the shared batch is also checked against the oracle."""
    import paged_kv_cache_pa_gb300 as pa
    rng = np.random.default_rng(41)
    S = 24
    lens = rng.integers(300, 1400, S)
    share = [0 if s % 6 == 0 else int(rng.integers(10, 18)) for s in range(S)]
    wl = shared_workload(lens, share, H, Hkv, D, dtype, seed=41)
    _check(wl, poison=False)                        # the shared batch against the oracle
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    mx = int(wl.max_context_len)
    la = torch.as_tensor(wl.context_lens, device=DEV)
    lb = torch.clamp(la, max=40)                    # shares at most 40 tokens: no runs form
    nbytes = pa.decode_workspace_size(S, H, Hkv, D, mx)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def call(lens_t, ws, out):
        pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens_t, mx,
                            wl.scale, out=out, workspace=ws, error_word=err)

    ref = {}
    for name, lens_t in (("a", la), ("b", lb)):
        ref[name] = torch.empty(S, H, D, dtype=torch.float32, device=DEV)
        call(lens_t, torch.empty(nbytes, dtype=torch.uint8, device=DEV), ref[name])
        torch.cuda.synchronize()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    outs = [torch.empty(S, H, D, dtype=torch.float32, device=DEV) for _ in range(40)]
    for i, out in enumerate(outs):
        call(la if i % 2 == 0 else lb, ws, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i, out in enumerate(outs):
        assert torch.equal(out, ref["a" if i % 2 == 0 else "b"]), i


@pytest.mark.parametrize("S,launches", [(4096, 4), (4097, 2)])
def test_shared_prefixes_at_the_batch_limit(S, launches):
    """4096 sequences, the most the plan looks for shared prefixes in (its
    1024 threads keep four sequences each), in runs of four that share 10 to
    15 leading blocks; and one sequence more, where detection is off and
    every sequence is read through its own table."""
    import paged_kv_cache_pa_gb300 as pa
    rng = np.random.default_rng(S)
    lens = rng.integers(256, 400, S)
    share = [0 if s % 4 == 0 else int(rng.integers(10, 16)) for s in range(S)]
    wl = shared_workload(lens, share, 2, 2, 64, "f16", seed=S)
    assert pa.decode_kernel_launches(S, 2, 2, 64, wl.max_context_len) == launches
    _check(wl, poison=False)
