"""GPU parity for chunked-prefill attention: the chunk's K/V go into the cache
through pa_cache_write, then pa_prefill_attention runs on the device and the
oracle runs the same two steps on host copies.  Bars as for decode: pools
bit-exact, attention max |gpu - oracle| <= 2e-3 on fp32 output."""
import numpy as np
import pytest
import torch

from paritylib import ATOL, codes, max_abs, prefill_oracle, prefill_problem, prefill_run

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import paged_kv_cache_pa_gb300 as pa  # noqa: E402

DEV = torch.device("cuda:0")
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


_problem = prefill_problem
_run = prefill_run
_oracle = prefill_oracle


CASES = [(0, 1), (0, 64), (0, 65), (0, 200), (37, 1), (100, 16), (500, 130), (63, 64), (1, 127),
         (64, 64), (15, 49)]


@pytest.mark.parametrize("H,Hkv,D,dtype,B", [
    (8, 8, 128, "f16", 16), (12, 2, 128, "bf16", 16), (8, 2, 64, "f16", 16),
    (4, 4, 64, "bf16", 8), (12, 2, 128, "bf16", 8), (8, 1, 128, "f16", 64),
    (6, 3, 64, "bf16", 256),
])
def test_prefill_parity(H, Hkv, D, dtype, B):
    d = _problem(CASES, H, Hkv, D, dtype, B, seed=H * 100 + D + B)
    scale = 1.0 / np.sqrt(D)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(d, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = _oracle(d, scale, dtype)
    assert np.array_equal(codes(d["kc"]), d["host"]["kc"])
    assert np.array_equal(codes(d["vc"]), d["host"]["vc"])
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    e = max_abs(got, want)
    print(f"prefill H={H} Hkv={Hkv} D={D} {dtype} B={B}: max|gpu-oracle| = {e:.3e}")
    assert e <= ATOL


def test_prefill_long_mixed_chunks():
    """A chunked-prefill batch like a scheduler's token budget: long cached
    prefixes with 512-token chunks, a whole 700-token prompt, decode rows."""
    cases = [(1536, 512), (0, 700), (3000, 1), (2047, 1), (511, 512), (4000, 96)]
    d = _problem(cases, 12, 2, 128, "bf16", 16, seed=77)
    scale = 1.0 / np.sqrt(128)
    out = _run(d, scale)
    torch.cuda.synchronize()
    want = _oracle(d, scale, "bf16")
    assert max_abs(out.cpu().numpy(), want) <= ATOL


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_half_output_is_rounded_fp32_output(dtype):
    cases = [(0, 90), (40, 33)]
    d = _problem(cases, 8, 2, 128, dtype, 16, seed=3)
    d2 = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in d.items()}
    scale = 0.09
    o32 = _run(d, scale)
    o16 = _run(d2, scale, out_dtype=TDT[dtype])
    torch.cuda.synchronize()
    assert torch.equal(o32.to(TDT[dtype]).view(torch.int16), o16.view(torch.int16))


def test_prefill_of_one_token_matches_decode():
    """Sequences with one new token: the prefill rows agree with decode
    attention over the same cache (both within the bar of the oracle)."""
    cases = [(10, 1), (300, 1), (1000, 1), (0, 1)]
    d = _problem(cases, 12, 2, 128, "bf16", 16, seed=5)
    scale = 1.0 / np.sqrt(128)
    out = _run(d, scale)
    dec = pa.decode_attention(d["q"], d["kc"], d["vc"], torch.as_tensor(d["tables"], device=DEV),
                              torch.as_tensor(d["lens"], device=DEV), d["maxc"], scale)
    torch.cuda.synchronize()
    assert max_abs(out.cpu().numpy(), dec.cpu().numpy()) <= ATOL


def test_prefill_errors_are_flagged():
    cases = [(20, 30), (0, 40), (5, 5)]
    d = _problem(cases, 4, 2, 64, "f16", 16, seed=9)
    lens = torch.as_tensor(d["lens"], device=DEV)
    lens[1] = 10                                   # fewer cached tokens than new ones
    tables = torch.as_tensor(d["tables"], device=DEV)
    tables[2, 0] = 10_000                          # a block id past the pool
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.prefill_attention(d["q"], d["kc"], d["vc"], tables,
                               torch.as_tensor(d["qsl"], device=DEV), lens, d["maxq"], d["maxc"],
                               0.1, error_word=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.ERRBIT_CONTEXT_LEN and e & pa.ERRBIT_BLOCK_OOB
    assert torch.all(out[30:70] == 0)              # the bad sequence's rows
    assert torch.all(torch.isfinite(out))
    with pytest.raises(pa.PaError) as ei:          # head_dim 256: not built for prefill
        q = torch.zeros(4, 2, 256, dtype=torch.float16, device=DEV)
        k = torch.zeros(4, 2, 16, 256, dtype=torch.float16, device=DEV)
        pa.prefill_attention(q, k, k, tables[:1], torch.tensor([0, 4], dtype=torch.int32,
                                                               device=DEV),
                             torch.tensor([4], dtype=torch.int32, device=DEV), 4, 4, 0.1)
    assert ei.value.status == 2


@pytest.mark.parametrize("H,Hkv,dtype", [(8, 2, "bf16"), (6, 6, "f16"), (9, 3, "bf16")])
def test_prefill_many_items_per_cta(H, Hkv, dtype):
    """Far more work items (query-tile pairs) than SMs, of very different
    lengths: the persistent CTAs take several items each, heaviest first, and
    every pipeline runs on across items.  The same workspace serves two
    calls (the plan resets the claim counter)."""
    rng = np.random.default_rng(H * 7 + Hkv)
    cases = [(int(rng.integers(0, 600)), int(rng.integers(1, 330))) for _ in range(48)]
    cases[5] = (0, 384)                      # exactly three query tiles
    cases[11] = (700, 1)                     # decode rows among the chunks
    d = _problem(cases, H, Hkv, 128, dtype, 16, seed=H + Hkv)
    maxq = d["maxq"]
    nbytes = pa.prefill_workspace_size(len(cases), H, Hkv, 128, maxq)
    mt = -(-maxq // 128)
    ix, iy = (mt, H // 2) if (H // Hkv) % 2 == 0 else (-(-mt // 2), H)
    assert nbytes >= 16 * len(cases) * ix * iy and nbytes % 256 == 0
    assert len(cases) * ix * iy > 2 * 152
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    scale = 1.0 / np.sqrt(128)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(d, scale, err=err, workspace=ws)
    out2 = pa.prefill_attention(d["q"], d["kc"], d["vc"], torch.as_tensor(d["tables"], device=DEV),
                                torch.as_tensor(d["qsl"], device=DEV),
                                torch.as_tensor(d["lens"], device=DEV), maxq, d["maxc"], scale,
                                workspace=ws, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = _oracle(d, scale, dtype)
    e = max_abs(out.cpu().numpy(), want)
    print(f"many items H={H} Hkv={Hkv} {dtype}: max|gpu-oracle| = {e:.3e}")
    assert e <= ATOL
    assert torch.equal(out, out2)           # same arithmetic whatever CTA took an item


def test_prefill_workspace_checks():
    cases = [(10, 20), (0, 5)]
    d = _problem(cases, 4, 2, 64, "f16", 16, seed=1)
    need = pa.prefill_workspace_size(2, 4, 2, 64, d["maxq"])
    assert need % 256 == 0 and need > 4 * 128 * 64 * 4    # room for split partials
    assert pa.prefill_workspace_size(2, 5, 2, 64, 10) == 0     # heads not a multiple of KV heads
    assert pa.prefill_workspace_size(2, 4, 2, 96, 10) == 0     # head_dim not built
    small = torch.empty(need, dtype=torch.uint8, device=DEV)[1:]    # misaligned
    with pytest.raises(pa.PaError) as ei:
        _run(d, 0.1, workspace=small)
    assert ei.value.status == 4
    short = torch.empty(need - 256, dtype=torch.uint8, device=DEV)  # too small
    with pytest.raises(pa.PaError) as ei:
        _run(d, 0.1, workspace=short)
    assert ei.value.status == 4
    assert pa.prefill_workspace_size(2, 4, 2, 64, 100_000) > need
    assert pa.prefill_workspace_size(2, 4, 2, 128, 20) > need


@pytest.mark.parametrize("scale", [0.0, -0.05])
def test_prefill_non_positive_scale(scale):
    """A scale of 0 (every visible key weighs the same) and a negative scale
    take the form that scales the scores before the maximum."""
    cases = [(30, 70), (0, 130), (200, 1)]
    d = _problem(cases, 8, 2, 128, "bf16", 16, seed=11)
    out = _run(d, scale)
    torch.cuda.synchronize()
    want = _oracle(d, scale, "bf16")
    assert max_abs(out.cpu().numpy(), want) <= ATOL


@pytest.mark.parametrize("H,Hkv,dtype,B", [(12, 2, "bf16", 16), (6, 6, "f16", 16),
                                          (9, 3, "bf16", 8), (4, 4, "f16", 64)])
def test_prefill_split_items(H, Hkv, dtype, B):
    """Items with more K/V tiles than an SM's even share are split over their
    keys; the two parts are merged exactly.  One long sequence among many short
    ones; a sequence whose second query tile is short, so that with tiles
    paired by tokens the second part has no keys for the first tile; decode
    rows; a sequence with a bad block id (its keys skipped) stays out."""
    rng = np.random.default_rng(H + Hkv + B)
    cases = [(3100, 256), (64, 256), (900, 129), (2000, 1)]
    cases += [(int(rng.integers(0, 40)), int(rng.integers(1, 64))) for _ in range(40)]
    d = _problem(cases, H, Hkv, 128, dtype, B, seed=H * 3 + B)
    scale = 1.0 / np.sqrt(128)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(d, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = _oracle(d, scale, dtype)
    e = max_abs(out.cpu().numpy(), want)
    print(f"split items H={H} Hkv={Hkv} {dtype} B={B}: max|gpu-oracle| = {e:.3e}")
    assert e <= ATOL
    # with the output in the input dtype, the merge rounds once, like the plain path
    d2 = _problem(cases, H, Hkv, 128, dtype, B, seed=H * 3 + B)
    o16 = _run(d2, scale, out_dtype=TDT[dtype])
    torch.cuda.synchronize()
    assert torch.equal(out.to(TDT[dtype]).view(torch.int16), o16.view(torch.int16))


def test_prefill_sequences_without_new_tokens():
    """Sequences with no new tokens in the batch (n = 0, with or without a
    cached context) contribute no rows and no work; a batch of only such
    sequences is a no-op."""
    cases = [(0, 0), (40, 0), (10, 30), (0, 0), (100, 70), (300, 0), (0, 1)]
    d = _problem(cases, 8, 2, 128, "bf16", 16, seed=21)
    scale = 1.0 / np.sqrt(128)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(d, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = _oracle(d, scale, "bf16")
    assert out.shape[0] == 101
    assert max_abs(out.cpu().numpy(), want) <= ATOL
    empty = _problem([(0, 0), (25, 0)], 8, 2, 128, "bf16", 16, seed=22)
    q = torch.zeros(0, 8, 128, dtype=torch.bfloat16, device=DEV)
    o = pa.prefill_attention(q, empty["kc"], empty["vc"],
                             torch.as_tensor(empty["tables"], device=DEV),
                             torch.as_tensor(empty["qsl"], device=DEV),
                             torch.as_tensor(empty["lens"], device=DEV), 0, 25, scale)
    torch.cuda.synchronize()
    assert o.shape == (0, 8, 128)


def _random_prefill(i):
    """Seeded random batch i: query groups 1..6, KV heads 1..4, head_dim 64 or
    128, fp16 / bf16, blocks of 8..256 tokens, 1..9 sequences each with a
    cached prefix of 0..2500 tokens and 0..600 new ones."""
    rng = np.random.default_rng(9100 + i)
    hkv = int(rng.integers(1, 5))
    H = hkv * int(rng.integers(1, 7))
    D = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["f16", "bf16"]))
    B = int(rng.choice([8, 16, 16, 32, 64, 256]))
    S = int(rng.integers(1, 10))
    cases = [(int(rng.integers(0, 2501)) * int(rng.integers(0, 2)), int(rng.integers(0, 601)))
             for _ in range(S)]
    if all(n == 0 for _, n in cases):
        cases[0] = (cases[0][0], 1)
    return cases, H, hkv, D, dtype, B


@pytest.mark.parametrize("i", range(12))
def test_prefill_random_batches(i):
    cases, H, Hkv, D, dtype, B = _random_prefill(i)
    d = _problem(cases, H, Hkv, D, dtype, B, seed=9100 + i)
    scale = 1.0 / np.sqrt(D)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(d, scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = _oracle(d, scale, dtype)
    assert np.array_equal(codes(d["kc"]), d["host"]["kc"])
    assert np.array_equal(codes(d["vc"]), d["host"]["vc"])
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert max_abs(got, want) <= ATOL, (cases, H, Hkv, D, dtype, B)
