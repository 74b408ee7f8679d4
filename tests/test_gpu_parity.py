"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars: cache write and block copy bit-exact over whole pools (so stray writes
show); attention max |gpu - oracle| <= 2e-3 on fp32 output; half-precision
output within 2e-3 plus half an ulp of the output type at the oracle value,
and bit-identical to rounding the fp32 output to nearest even.
"""
import numpy as np
import pytest
import torch

from paritylib import (ATOL, codes, custom_workload, gpu_step, host_inputs, max_abs,
                       oracle_step, step_blocks)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped
    pytest.skip("needs a CUDA device", allow_module_level=True)

import paged_kv_cache_pa_gb300 as pa  # noqa: E402
from paged_kv_cache_pa_gb300 import synthetic  # noqa: E402

DEV = torch.device("cuda:0")


def _err_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _run_and_check(wl, poison=False, out_dtype=torch.float32, whole_pool=True,
                   fill_all_blocks=None):
    vals = synthetic.make_values(wl, device=DEV, fill_all_blocks=fill_all_blocks,
                                 poison_unused=poison)
    blocks = None if whole_pool else step_blocks(wl)
    h = host_inputs(wl, vals, blocks)
    err = _err_word()
    out = gpu_step(wl, vals, out_dtype=out_dtype, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle_step(wl, h)
    # pools after copy + write: bit-exact
    if blocks is None:
        got_k, got_v = codes(vals["k_cache"]), codes(vals["v_cache"])
    else:
        idx = torch.as_tensor(blocks, device=DEV)
        got_k = codes(vals["k_cache"].index_select(0, idx))
        got_v = codes(vals["v_cache"].index_select(0, idx))
    assert np.array_equal(got_k, h["k_cache"])
    assert np.array_equal(got_v, h["v_cache"])
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    return got, want


# ---------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "opt13b", "gqa", "beams"])
def test_workload_step_parity(name):
    wl = synthetic.make(name)
    got, want = _run_and_check(wl)
    err = max_abs(got, want)
    print(f"{name}: max|gpu-oracle| = {err:.3e}")
    assert err <= ATOL


def test_long_context_partitions_parity():
    """8 sequences of 16K-32K tokens scattered over a 60 GiB pool; the oracle
    gets the blocks the step touches.  Untouched blocks stay as they were."""
    wl = synthetic.make("long")
    vals = synthetic.make_values(wl, device=DEV, fill_all_blocks=False)
    blocks = step_blocks(wl)
    rng = np.random.default_rng(0)
    bystanders = np.setdiff1d(rng.choice(wl.num_blocks, 256, replace=False), blocks)
    bidx = torch.as_tensor(bystanders, device=DEV)
    before = codes(vals["k_cache"].index_select(0, bidx)), codes(vals["v_cache"].index_select(0, bidx))
    h = host_inputs(wl, vals, blocks)
    err = _err_word()
    out = gpu_step(wl, vals, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle_step(wl, h)
    idx = torch.as_tensor(blocks, device=DEV)
    assert np.array_equal(codes(vals["k_cache"].index_select(0, idx)), h["k_cache"])
    assert np.array_equal(codes(vals["v_cache"].index_select(0, idx)), h["v_cache"])
    assert np.array_equal(codes(vals["k_cache"].index_select(0, bidx)), before[0])
    assert np.array_equal(codes(vals["v_cache"].index_select(0, bidx)), before[1])
    e = max_abs(out.cpu().numpy(), want)
    print(f"long: max|gpu-oracle| = {e:.3e}")
    assert e <= ATOL


# ---------------------------------------------------------------------------
# shapes, lengths and edge cases at sizes the oracle finishes in seconds
# ---------------------------------------------------------------------------

EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512,
             513, 1023, 1024, 1025, 1500]


@pytest.mark.parametrize("H,Hkv,D,dtype", [
    (8, 8, 64, "f16"), (4, 4, 128, "f16"), (4, 4, 128, "bf16"), (4, 4, 256, "bf16"),
    (8, 4, 128, "f16"), (12, 2, 128, "bf16"), (6, 2, 64, "f16"), (16, 2, 128, "f16"),
    (10, 2, 256, "f16"), (5, 1, 128, "bf16"), (7, 1, 64, "bf16"),
    (6, 2, 256, "bf16"), (14, 2, 256, "f16"), (16, 2, 256, "bf16"),  # D = 256, G = 3, 7, 8
])
def test_shapes_and_block_edges(H, Hkv, D, dtype):
    wl = custom_workload(EDGE_LENS, H, Hkv, D, dtype, seed=H * 1000 + D)
    got, want = _run_and_check(wl, poison=True)
    assert max_abs(got, want) <= ATOL


def test_partition_edges_at_512():
    """Enough (sequence, KV head) units that the plan uses 512-token
    partitions; lengths straddle the partition boundaries."""
    lens = ([511, 512, 513, 1023, 1024, 1025, 1536, 1537, 2047, 2048] * 7)[:64]
    wl = custom_workload(lens, 40, 40, 128, "f16", seed=3)
    got, want = _run_and_check(wl)
    assert max_abs(got, want) <= ATOL


def _merge_hpc(S, H):
    """Query heads a merge CTA takes for these sizes (the host's rule)."""
    hpc = 1
    while hpc < 8 and S * -(-H // hpc) > 3072:
        hpc *= 2
    return hpc


@pytest.mark.parametrize("S,H,Hkv,D,dtype,hpc", [
    (1600, 8, 8, 64, "f16", 8),     # CUDA-core kernel, one thread a column group
    (800, 16, 16, 128, "bf16", 8),  # two float4 columns a thread
    (400, 20, 20, 256, "f16", 4),   # head_dim 256: two columns a thread
    (100, 40, 40, 128, "f16", 2),   # two partition groups a head
    (128, 32, 8, 128, "bf16", 2),   # tensor-core kernel (4 query heads a KV head)
])
def test_merge_several_heads_a_cta(S, H, Hkv, D, dtype, hpc):
    """Batches large enough that one merge CTA takes several query heads:
    most sequences fit one partition (their CTAs leave at once), every
    eleventh needs a merge of two partitions."""
    assert _merge_hpc(S, H) == hpc
    rng = np.random.default_rng(S + H + D)
    lens = rng.integers(1, 33, S)
    lens[::11] = rng.integers(520, 1000, len(lens[::11]))
    wl = custom_workload(lens, H, Hkv, D, dtype, seed=S + D)
    assert pa.decode_partition_tokens(S, Hkv, wl.max_context_len) == 512
    got, want = _run_and_check(wl, whole_pool=False)
    assert max_abs(got, want) <= ATOL


def test_poisoned_padding_is_never_read():
    """NaN in every slot past each sequence's length and in every unused
    block: the output stays finite and equal to the oracle's."""
    wl = synthetic.make("tiny")
    got, want = _run_and_check(wl, poison=True)
    assert max_abs(got, want) <= ATOL


@pytest.mark.parametrize("lens", [[1, 5, 77, 300, 700], [1, 5, 77, 200, 255]])  # the second: no plan
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_half_output_is_rounded_fp32_output(dtype, lens):
    wl = custom_workload(lens, 8, 2, 128, dtype, seed=11)
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    vals = synthetic.make_values(wl, device=DEV)
    h = host_inputs(wl, vals)
    # run twice on identical inputs: fp32 output and half output
    vals2 = {k: v.clone() for k, v in vals.items()}
    out32 = gpu_step(wl, vals)
    out16 = gpu_step(wl, vals2, out_dtype=tdt)
    torch.cuda.synchronize()
    assert torch.equal(out32.to(tdt).view(torch.int16), out16.view(torch.int16))
    want = oracle_step(wl, h)
    # tolerance: 2e-3 plus half an ulp of the output type at |want|
    mant = 10 if dtype == "f16" else 7
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -14))) - mant)
    assert np.all(np.abs(out16.float().cpu().numpy() - want) <= ATOL + 0.5 * ulp)


def test_context_of_one_returns_v0():
    wl = custom_workload([1] * 9, 12, 2, 128, "bf16", seed=5)
    vals = synthetic.make_values(wl, device=DEV)
    out = gpu_step(wl, vals)
    torch.cuda.synchronize()
    # position 0 of every sequence is the token the step wrote: value[s]
    v = vals["value"].float().repeat_interleave(6, dim=1)
    assert torch.equal(out, v)


def test_empty_sequences_give_zero_rows():
    wl = custom_workload([0, 40, 0, 3], 4, 2, 64, "f16", seed=9)
    got, want = _run_and_check(wl)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert max_abs(got, want) <= ATOL


# ---------------------------------------------------------------------------
# small batches without the plan: at most 256 (sequence, KV head) pairs, each
# context within one partition, no shared-prefix items; each pair is one item
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,H,Hkv,D,dtype,B,max_len,direct", [
    (128, 2, 2, 64, "f16", 16, 255, True),      # G = 1, CUDA cores, 256 pairs
    (129, 2, 2, 64, "f16", 16, 255, False),     # two pairs more: the plan runs
    (32, 64, 8, 128, "bf16", 16, 0, True),      # G = 8, a whole partition
    (256, 4, 1, 128, "f16", 16, 200, True),     # G = 4, one KV head
    (42, 6, 6, 256, "f16", 16, 0, True),        # D = 256, a whole partition
    (60, 8, 4, 128, "f16", 8, 255, True),       # G = 2 on 8-token blocks
])
def test_small_batches_without_the_plan(S, H, Hkv, D, dtype, B, max_len, direct):
    if max_len == 0:                            # the longest context one partition holds
        max_len = pa.decode_partition_tokens(S, Hkv, 512)
    rng = np.random.default_rng(S * 31 + H)
    lens = rng.integers(1, max_len + 1, size=S)
    lens[0], lens[1], lens[2], lens[-1] = max_len, 0, 1, 0
    wl = custom_workload(lens, H, Hkv, D, dtype, seed=S + D, block_size=B)
    assert wl.max_context_len == max_len
    assert (pa.decode_kernel_launches(S, H, Hkv, D, max_len) == 1) == direct
    got, want = _run_and_check(wl)
    assert np.all(got[lens == 0] == 0)
    assert max_abs(got, want) <= ATOL


def test_small_batch_bad_length_on_tensor_cores_is_flagged():
    wl = custom_workload([40, 90, 7, 200, 150], 12, 2, 128, "bf16", seed=4)
    assert pa.decode_kernel_launches(5, 12, 2, 128, wl.max_context_len) == 1
    vals = synthetic.make_values(wl, device=DEV)
    h = host_inputs(wl, vals)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    lens[1] = -3                                       # negative
    lens[3] = 10_000                                   # above max_context_len
    err = _err_word()
    out = pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                              wl.max_context_len, wl.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.ERRBIT_CONTEXT_LEN
    assert torch.all(out[1] == 0) and torch.all(out[3] == 0)
    import oracle
    want = oracle.decode_attention(h["q"], h["k_cache"], h["v_cache"], h["tables"],
                                   wl.context_lens, wl.scale, wl.dtype)
    keep = [0, 2, 4]
    assert max_abs(out.cpu().numpy()[keep], want[keep]) <= ATOL


# ---------------------------------------------------------------------------
# query groups on the tensor-core kernel: extreme batch shapes for the plan,
# the item pipeline and the merge
# ---------------------------------------------------------------------------

def test_gqa_one_long_sequence():
    """One sequence of 20000 tokens: every item is a partition of its two
    KV heads, and the merge folds 40 partitions per head."""
    wl = custom_workload([20000], 12, 2, 128, "bf16", seed=21)
    got, want = _run_and_check(wl)
    assert max_abs(got, want) <= ATOL


def test_gqa_fewer_items_than_ctas():
    """Four short sequences: most CTAs get no item at all."""
    wl = custom_workload([1, 17, 40, 33], 8, 2, 64, "f16", seed=22)
    got, want = _run_and_check(wl, poison=True)
    assert max_abs(got, want) <= ATOL


def test_gqa_empty_sequences_between():
    """Empty sequences among long and short ones give zero rows and no
    items."""
    lens = [0, 300, 0, 0, 5000, 0, 1, 0, 2048, 17, 0]
    wl = custom_workload(lens, 8, 2, 128, "f16", seed=23)
    got, want = _run_and_check(wl, poison=True)
    for s, L in enumerate(lens):
        if L == 0:
            assert np.all(got[s] == 0)
    assert max_abs(got, want) <= ATOL


def test_gqa_many_sequences():
    """More sequences than the plan kernel's 1024 threads (it takes them in
    tiles) and many more items than CTAs."""
    rng = np.random.default_rng(24)
    lens = rng.integers(0, 90, 2500)
    wl = custom_workload(lens, 8, 2, 64, "bf16", seed=24)
    got, want = _run_and_check(wl)
    assert max_abs(got, want) <= ATOL


def test_output_is_bit_reproducible():
    wl = synthetic.make("gqa")
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    outs = [pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                                wl.max_context_len, wl.scale) for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("H,Hkv,D,dtype", [(8, 8, 128, "f16"), (12, 2, 128, "bf16")])
def test_back_to_back_calls_share_a_workspace(H, Hkv, D, dtype):
    """Calls enqueued back to back on one stream, alternating two batches of
    different lengths (different work lists) and sharing one workspace,
    each after a cache write as in a decode step: every output equals the
    one the same batch gives alone, to the bit.  The plan kernel of a call
    rewrites the work list while the kernel ahead of it may still run, so a
    race with the previous call's attention would show here."""
    rng = np.random.default_rng(31)
    lens_a = rng.integers(1, 3000, 48)
    lens_b = rng.integers(1, 600, 48)
    lens_b[::7] = 2999                          # a few long ones: several partitions
    wl = custom_workload(np.maximum(lens_a, lens_b), H, Hkv, D, dtype, seed=31)
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    mx = int(wl.max_context_len)
    la = torch.as_tensor(lens_a.astype(np.int32), device=DEV)
    lb = torch.as_tensor(lens_b.astype(np.int32), device=DEV)
    slots = torch.full((wl.num_seqs,), -1, dtype=torch.int64, device=DEV)  # a write of nothing
    S = wl.num_seqs
    nbytes = pa.decode_workspace_size(S, H, Hkv, D, mx)
    err = _err_word()

    def call(lens, ws, out):
        pa.cache_write(vals["key"], vals["value"], vals["k_cache"], vals["v_cache"], slots,
                       error_word=err)
        pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens, mx,
                            wl.scale, out=out, workspace=ws, error_word=err)

    ref = {}
    for name, lens in (("a", la), ("b", lb)):
        ref[name] = torch.empty(S, H, D, dtype=torch.float32, device=DEV)
        call(lens, torch.empty(nbytes, dtype=torch.uint8, device=DEV), ref[name])
        torch.cuda.synchronize()
    shared = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    outs = [torch.empty(S, H, D, dtype=torch.float32, device=DEV) for _ in range(40)]
    for i, out in enumerate(outs):
        call(la if i % 2 == 0 else lb, shared, out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i, out in enumerate(outs):
        assert torch.equal(out, ref["a" if i % 2 == 0 else "b"]), i


def _fuzz_case(i):
    """Seeded random shape i: query groups 1..8, KV heads 1..8, head_dim 64 /
    128 / 256, fp16 / bf16, blocks of 8..256 tokens, 1..40 sequences with a
    mix of empty, short and long contexts."""
    rng = np.random.default_rng(7000 + i)
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.integers(1, 9))
    D = int(rng.choice([64, 128, 256]))
    dtype = str(rng.choice(["f16", "bf16"]))
    B = int(rng.choice([8, 16, 16, 32, 64, 128, 256]))
    S = int(rng.integers(1, 41))
    kind = rng.integers(0, 4, S)
    lens = np.where(kind == 0, 0, np.where(kind == 1, rng.integers(1, 40, S),
                                           rng.integers(40, 3000, S)))
    if not lens.any():
        lens[0] = int(rng.integers(1, 3000))
    return lens, G * hkv, hkv, D, dtype, B


@pytest.mark.parametrize("i", range(24))
def test_random_shapes(i):
    lens, H, Hkv, D, dtype, B = _fuzz_case(i)
    wl = custom_workload(lens, H, Hkv, D, dtype, seed=7000 + i, block_size=B)
    got, want = _run_and_check(wl, poison=True)
    for s, L in enumerate(lens):
        if L == 0:
            assert np.all(got[s] == 0)
    assert max_abs(got, want) <= ATOL, (H, Hkv, D, dtype, B, len(lens))


# ---------------------------------------------------------------------------
# other block sizes (pools of B tokens per block, the *_ex entry points)
# ---------------------------------------------------------------------------

BS_LENS = [1, 7, 8, 9, 15, 16, 17, 31, 33, 63, 64, 65, 100, 255, 257, 511, 513, 700, 1025]


@pytest.mark.parametrize("B", [8, 32, 64, 128, 256])
@pytest.mark.parametrize("H,Hkv,D,dtype", [
    (4, 4, 128, "f16"), (12, 2, 128, "bf16"), (8, 2, 64, "f16"), (6, 2, 256, "bf16"),
    (3, 3, 64, "bf16"),
])
def test_block_sizes_step_parity(B, H, Hkv, D, dtype):
    """The whole step (cache write + attention) over pools of B-token
    blocks, NaN in every uncovered slot: pools bit-exact, attention within
    the bar, both tensor-core (G >= 2, D <= 128) and CUDA-core paths."""
    wl = custom_workload(BS_LENS, H, Hkv, D, dtype, seed=B * 7 + H, block_size=B)
    got, want = _run_and_check(wl, poison=True)
    assert max_abs(got, want) <= ATOL


@pytest.mark.parametrize("B", [8, 64])
def test_block_sizes_partition_edges(B):
    """512-token partitions over 8- and 64-token blocks."""
    lens = ([511, 512, 513, 1023, 1024, 1025, 1536, 1537, 2047, 2048] * 7)[:64]
    wl = custom_workload(lens, 40, 40, 128, "f16", seed=B, block_size=B)
    got, want = _run_and_check(wl)
    assert max_abs(got, want) <= ATOL


@pytest.mark.parametrize("B", [8, 128])
def test_block_sizes_gqa_workload(B):
    """The GQA workload (12 query heads on 2 KV heads, bf16) re-laid with
    other block sizes."""
    wl = synthetic.relayout(synthetic.make("gqa"), B)
    got, want = _run_and_check(wl)
    assert max_abs(got, want) <= ATOL


@pytest.mark.parametrize("B", [8, 64, 256])
def test_copy_blocks_block_sizes_bit_exact(B):
    import oracle
    L, NB, Hkv, D = 3, 12, 2, 128
    g = torch.Generator(device=DEV).manual_seed(B)
    ks = [torch.randn(NB, Hkv, B, D, generator=g, device=DEV).bfloat16() for _ in range(L)]
    vs = [torch.randn(NB, Hkv, B, D, generator=g, device=DEV).bfloat16() for _ in range(L)]
    pairs = np.array([[3, 10], [7, 11], [0, 5]], np.int64)
    hk = [codes(k) for k in ks]
    hv = [codes(v) for v in vs]
    oracle.copy_blocks(hk, hv, pairs)
    err = _err_word()
    pa.copy_blocks(ks, vs, torch.as_tensor(pairs, device=DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        assert np.array_equal(codes(ks[l]), hk[l])
        assert np.array_equal(codes(vs[l]), hv[l])


@pytest.mark.parametrize("H,Hkv", [(4, 4), (12, 2)])
def test_eight_token_blocks_second_block_out_of_range(H, Hkv):
    """With 8-token blocks a 16-token chunk spans two table entries; a bad
    id in the second one is flagged and the output stays finite."""
    wl = custom_workload([40, 40, 40], H, Hkv, 128, "bf16", seed=4, block_size=8)
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    tables[1, 3] = wl.num_blocks + 3                   # second block of chunk 1
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    err = _err_word()
    out = pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens, 40,
                              wl.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.ERRBIT_BLOCK_OOB
    assert torch.all(torch.isfinite(out))


def test_unsupported_block_sizes_are_refused():
    q = torch.zeros(2, 4, 128, dtype=torch.float16, device=DEV)
    t = torch.zeros(2, 4, dtype=torch.int32, device=DEV)
    ln = torch.ones(2, dtype=torch.int32, device=DEV)
    for B in (4, 12, 512):
        kc = torch.zeros(4, 4, B, 128, dtype=torch.float16, device=DEV)
        with pytest.raises(pa.PaError) as ei:
            pa.decode_attention(q, kc, kc, t, ln, 1, 0.1)
        assert ei.value.status == 2
        with pytest.raises(pa.PaError) as ei:
            pa.cache_write(q[:, :4], q[:, :4], kc, kc, torch.zeros(2, dtype=torch.int64,
                                                                    device=DEV))
        assert ei.value.status == 2


# ---------------------------------------------------------------------------
# block copy across layers; device-detected errors; host-detected errors
# ---------------------------------------------------------------------------

def test_copy_blocks_all_layers_bit_exact():
    import oracle
    L, NB, Hkv, D = 5, 40, 4, 128
    g = torch.Generator(device=DEV).manual_seed(3)
    ks = [torch.randn(NB, Hkv, 16, D, generator=g, device=DEV).half() for _ in range(L)]
    vs = [torch.randn(NB, Hkv, 16, D, generator=g, device=DEV).half() for _ in range(L)]
    pairs = np.array([[3, 30], [7, 31], [3, 32], [12, 5], [0, 39]], np.int64)
    hk = [codes(k) for k in ks]
    hv = [codes(v) for v in vs]
    oracle.copy_blocks(hk, hv, pairs)
    err = _err_word()
    pa.copy_blocks(ks, vs, torch.as_tensor(pairs, device=DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        assert np.array_equal(codes(ks[l]), hk[l])
        assert np.array_equal(codes(vs[l]), hv[l])


def test_copy_blocks_out_of_range_pair_is_flagged_and_skipped():
    NB = 8
    k = torch.arange(NB * 16 * 64, device=DEV, dtype=torch.float32).half().view(NB, 1, 16, 64)
    v = k.clone()
    k0 = k.clone()
    err = _err_word()
    pairs = torch.tensor([[1, NB], [-1, 2], [3, 3]], device=DEV, dtype=torch.int64)
    pa.copy_blocks([k], [v], pairs, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.ERRBIT_BLOCK_OOB
    assert torch.equal(k, k0)


def test_cache_write_out_of_range_slot_is_flagged_and_skipped():
    NB, Hkv, D = 4, 2, 64
    kc = torch.zeros(NB, Hkv, 16, D, dtype=torch.float16, device=DEV)
    vc = kc.clone()
    key = torch.ones(3, Hkv, D, dtype=torch.float16, device=DEV)
    slots = torch.tensor([NB * 16, -1, 5], device=DEV, dtype=torch.int64)
    err = _err_word()
    pa.cache_write(key, key, kc, vc, slots, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.ERRBIT_SLOT_OOB
    assert int((kc != 0).sum()) == Hkv * D          # only slot 5 written
    assert torch.equal(kc[0, :, 5], key[2])


def test_bad_table_entry_and_context_len_are_flagged():
    wl = custom_workload([40, 40, 40], 4, 4, 128, "f16", seed=2)
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    tables[1, 1] = wl.num_blocks + 7                   # out of range block id
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    lens[2] = 10_000                                   # above max_context_len
    err = _err_word()
    out = pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens, 40,
                              wl.scale, error_word=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.ERRBIT_BLOCK_OOB and e & pa.ERRBIT_CONTEXT_LEN
    assert torch.all(out[2] == 0)
    assert torch.all(torch.isfinite(out))


def test_host_detected_errors():
    q = torch.zeros(2, 8, 128, dtype=torch.float16, device=DEV)
    kc = torch.zeros(4, 1, 16, 128, dtype=torch.float16, device=DEV)
    t = torch.zeros(2, 4, dtype=torch.int32, device=DEV)
    ln = torch.ones(2, dtype=torch.int32, device=DEV)
    with pytest.raises(pa.PaError) as ei:              # 8 query heads per KV head is fine;
        pa.decode_attention(q.view(2, 8, 128).repeat(1, 2, 1), kc, kc, t, ln, 16, 0.1)
    assert ei.value.status == 2                        # 16 per KV head is not
    ws = torch.zeros(8, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PaError) as ei:
        pa.decode_attention(q, kc, kc, t, ln, 16, 0.1, workspace=ws)
    assert ei.value.status == 4
    with pytest.raises(pa.PaError) as ei:              # max_context_len beyond the table
        pa.decode_attention(q, kc, kc, t, ln, 65, 0.1)
    assert ei.value.status == 1
    q96 = torch.zeros(2, 1, 96, dtype=torch.float16, device=DEV)
    k96 = torch.zeros(4, 1, 16, 96, dtype=torch.float16, device=DEV)
    with pytest.raises(pa.PaError) as ei:
        pa.decode_attention(q96, k96, k96, t, ln, 16, 0.1)
    assert ei.value.status == 2


# ---------------------------------------------------------------------------
# swap between the device pool and a CPU swap space in pinned host memory
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,dtype", [(8, torch.float16), (16, torch.bfloat16),
                                     (256, torch.float16)])
def test_swap_out_and_in_bit_exact(B, dtype):
    """Swap-out (device -> pinned host) and swap-in (host -> device, into
    other block ids), all layers in one call each: both pools equal the
    oracle's byte for byte."""
    import oracle
    L, ND, NS, Hkv, D = 3, 24, 16, 4, 128
    g = torch.Generator(device=DEV).manual_seed(B)
    gk = [torch.randn(ND, Hkv, B, D, generator=g, device=DEV).to(dtype) for _ in range(L)]
    gv = [torch.randn(ND, Hkv, B, D, generator=g, device=DEV).to(dtype) for _ in range(L)]
    ck = [torch.randn(NS, Hkv, B, D).to(dtype).pin_memory() for _ in range(L)]
    cv = [torch.randn(NS, Hkv, B, D).to(dtype).pin_memory() for _ in range(L)]
    hgk, hgv = [codes(x) for x in gk], [codes(x) for x in gv]
    hck = [x.view(torch.int16).numpy().view(np.uint16).copy() for x in ck]
    hcv = [x.view(torch.int16).numpy().view(np.uint16).copy() for x in cv]
    rng = np.random.default_rng(B)
    out_pairs = np.stack([rng.choice(ND, 9, replace=False), rng.choice(NS, 9, replace=False)], 1)
    in_pairs = np.stack([out_pairs[:, 1], rng.choice(ND, 9, replace=False)], 1)
    err = _err_word()
    pa.swap_blocks(ck, cv, gk, gv, torch.as_tensor(out_pairs, device=DEV), error_word=err)
    oracle.swap_blocks(hck, hcv, hgk, hgv, out_pairs)
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(ck[l].view(torch.int16).numpy().view(np.uint16), hck[l])
        assert np.array_equal(cv[l].view(torch.int16).numpy().view(np.uint16), hcv[l])
    pa.swap_blocks(gk, gv, ck, cv, torch.as_tensor(in_pairs, device=DEV), error_word=err)
    oracle.swap_blocks(hgk, hgv, hck, hcv, in_pairs)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        assert np.array_equal(codes(gk[l]), hgk[l])
        assert np.array_equal(codes(gv[l]), hgv[l])


def test_swap_bad_pair_is_flagged_and_pageable_memory_refused():
    ND, NS, Hkv, B, D = 4, 4, 1, 16, 64
    gk = torch.zeros(ND, Hkv, B, D, dtype=torch.float16, device=DEV)
    ck = torch.ones(NS, Hkv, B, D, dtype=torch.float16).pin_memory()
    err = _err_word()
    pairs = torch.tensor([[0, NS], [1, 2]], dtype=torch.int64, device=DEV)
    pa.swap_blocks([ck], [ck], [gk], [gk], pairs, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.ERRBIT_BLOCK_OOB
    assert torch.all(ck[2] == 0) and torch.all(ck[0] == 1) and torch.all(ck[3] == 1)
    # a pageable host pool is refused on the host, before any launch
    lib = pa.load_library()
    import ctypes
    pageable = np.zeros((NS, Hkv, B, D), np.uint16)
    arr = (ctypes.c_void_p * 1)(pageable.ctypes.data)
    dev_arr = (ctypes.c_void_p * 1)(gk.data_ptr())
    st = lib.pa_swap_blocks(ctypes.cast(arr, ctypes.c_void_p), ctypes.cast(arr, ctypes.c_void_p),
                            ctypes.cast(dev_arr, ctypes.c_void_p),
                            ctypes.cast(dev_arr, ctypes.c_void_p), 1, pairs.data_ptr(), 1, NS,
                            ND, B, Hkv, D, 0, None, None)
    assert st == 1
    assert np.all(pageable == 0)


# ---------------------------------------------------------------------------
# contiguous (unpaged) cache: the layout the block table replaces
# ---------------------------------------------------------------------------

# "short": every context within one partition and few enough (sequence, KV
# head) pairs that the call runs without the plan, an empty sequence among them
CONTIG_LENS = {"mixed": [1, 15, 16, 17, 100, 513, 1000, 1025],
               "short": [1, 15, 16, 0, 17, 100, 200, 255]}


@pytest.mark.parametrize("lens_kind", sorted(CONTIG_LENS))
@pytest.mark.parametrize("H,Hkv,D,dtype", [(8, 8, 128, "f16"), (12, 2, 128, "bf16"),
                                           (8, 2, 64, "f16"), (4, 4, 256, "bf16")])
def test_contiguous_cache_matches_oracle(H, Hkv, D, dtype, lens_kind):
    import oracle
    lens = np.array(CONTIG_LENS[lens_kind], np.int32)
    S = len(lens)
    direct = pa.decode_kernel_launches(S, H, Hkv, D, int(lens.max())) == 1
    assert direct == (lens_kind == "short")
    rows = int(-(-lens.max() // 16) * 16) + 16
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    g = torch.Generator(device=DEV).manual_seed(H * 31 + D)
    q = torch.randn(S, H, D, generator=g, device=DEV).to(tdt)
    kc = torch.randn(S, Hkv, rows, D, generator=g, device=DEV).to(tdt)
    vc = torch.randn(S, Hkv, rows, D, generator=g, device=DEV).to(tdt)
    pos = torch.arange(rows, device=DEV)
    live = pos[None, :] < torch.as_tensor(lens, device=DEV)[:, None]          # [S][rows]
    nan = torch.tensor(float("nan"), dtype=tdt, device=DEV)
    kc = torch.where(live[:, None, :, None], kc, nan).contiguous()            # poison past L
    vc = torch.where(live[:, None, :, None], vc, nan).contiguous()
    err = _err_word()
    out = pa.decode_attention_contiguous(q, kc, vc, torch.as_tensor(lens, device=DEV),
                                         int(lens.max()), 1.0 / np.sqrt(D), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # host: the same rows as a paged pool (sequence s's block j -> block s*nb + j)
    nb = rows // 16

    def pool(c):
        return codes(c).reshape(S, Hkv, nb, 16, D).transpose(0, 2, 1, 3, 4).reshape(
            S * nb, Hkv, 16, D).copy()
    tables = (np.arange(S)[:, None] * nb + np.arange(nb)[None, :]).astype(np.int32)
    want = oracle.decode_attention(codes(q), pool(kc), pool(vc), tables, lens, 1.0 / np.sqrt(D),
                                   dtype)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.all(got[lens == 0] == 0)
    assert max_abs(got, want) <= ATOL


def test_in_order_placement_gives_the_same_output():
    wl = synthetic.in_order(synthetic.make("gqa"))
    got, want = _run_and_check(wl)
    assert max_abs(got, want) <= ATOL
