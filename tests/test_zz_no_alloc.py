"""pa_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (for example code running inside an engine's
execution phase, where all memory must be planned beforehand).  It uses a
workspace array built into the library instead of a caller-provided one.

Called through the C ABI (ctypes on libpa_gb300.so) and compared, bit for
bit, with the existing pa_decode_attention on the same inputs.  The built-in
array keeps the previous call's contents, so the calls alternate two batches
of different shapes (A, B, A): a work list or partial result left by the
other shape must not leak into a result.  One result is also checked against
the CPU oracle.  This file is collected last on purpose.
"""
import ctypes
from types import SimpleNamespace

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA device", allow_module_level=True)

import paged_kv_cache_pa_gb300 as pa  # noqa: E402
from paged_kv_cache_pa_gb300 import synthetic  # noqa: E402
from paged_kv_cache_pa_gb300.build import build  # noqa: E402

ATOL = 2e-3
NOALLOC_BYTES = 32 << 20
DEV = torch.device("cuda:0")
PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE = 1, 2, 4


def _noalloc_fn():
    build()
    lib = ctypes.CDLL(pa.library_path())
    fn = lib.pa_decode_attention_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.restype = I
    fn.argtypes = [P, I, P, P, P, P, I, P, I, I, I, I, I, I, ctypes.c_float, I, P, P]
    return fn


def _call(fn, out, wl, vals, tables, lens, err):
    code = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}
    return fn(out.data_ptr(), code[out.dtype], vals["q"].data_ptr(), vals["k_cache"].data_ptr(),
              vals["v_cache"].data_ptr(), tables.data_ptr(), tables.shape[1], lens.data_ptr(),
              wl.max_context_len, wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
              wl.num_blocks, wl.scale, code[vals["q"].dtype], err.data_ptr(),
              torch.cuda.current_stream(DEV).cuda_stream)


def _batch(name):
    wl = synthetic.make(name)
    assert pa.decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                    wl.max_context_len) <= NOALLOC_BYTES
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    # the existing entry point, with its own freshly allocated workspace
    ref = pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                              wl.max_context_len, wl.scale)
    torch.cuda.synchronize()
    return SimpleNamespace(wl=wl, vals=vals, tables=tables, lens=lens, ref=ref)


def test_noalloc_alternating_batches_match_decode_attention_bit_for_bit(oracle_mod):
    fn = _noalloc_fn()
    a, b = _batch("gqa"), _batch("opt13b")
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for x in (a, b, a, b):
        out = torch.full_like(x.ref, float("nan"))
        assert _call(fn, out, x.wl, x.vals, x.tables, x.lens, err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, x.ref), float((out - x.ref).abs().max())
        outs.append(out)
    # and the noalloc result against the oracle (grouped-query batch, whole batch)
    from paritylib import host_inputs, max_abs
    h = host_inputs(a.wl, a.vals)
    want = oracle_mod.decode_attention(h["q"], h["k_cache"], h["v_cache"], h["tables"],
                                       a.wl.context_lens, a.wl.scale, a.wl.dtype)
    assert max_abs(outs[2].cpu().numpy(), want) <= ATOL


def test_noalloc_rejects_sizes_beyond_its_array():
    fn = _noalloc_fn()
    # 64 sequences x 64 heads x 256 dims with 32K-token contexts need far more
    # than the built-in array; the call must refuse before enqueuing anything
    wl = SimpleNamespace(max_context_len=32768, num_seqs=64, num_heads=64, num_kv_heads=64,
                         head_dim=256, num_blocks=64 * 2048, scale=0.0625)
    assert pa.decode_workspace_size(64, 64, 64, 256, 32768) > NOALLOC_BYTES
    t = torch.zeros(64, dtype=torch.float16, device=DEV)
    tables = torch.zeros(64, 2048, dtype=torch.int32, device=DEV)
    lens = torch.zeros(64, dtype=torch.int32, device=DEV)
    vals = {"q": t, "k_cache": t, "v_cache": t}
    out = torch.zeros(64, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _call(fn, out, wl, vals, tables, lens, err) == PA_ERR_WORKSPACE


@pytest.mark.parametrize("change, status", [
    ({"head_dim": 512}, PA_ERR_UNSUPPORTED),             # no kernel for this head_dim
    ({"num_heads": 64 * 9, "num_kv_heads": 64}, PA_ERR_UNSUPPORTED),   # group of 9
    ({"num_heads": 65, "num_kv_heads": 64}, PA_ERR_INVALID_ARG),      # not divisible
])
def test_noalloc_reports_argument_errors_before_the_size_limit(change, status):
    """Sizes far beyond the array that are also invalid get the error
    pa_decode_attention would give, not PA_ERR_WORKSPACE."""
    fn = _noalloc_fn()
    base = dict(max_context_len=32768, num_seqs=64, num_heads=64, num_kv_heads=64,
                head_dim=256, num_blocks=64 * 2048, scale=0.0625)
    base.update(change)
    wl = SimpleNamespace(**base)
    t = torch.zeros(64, dtype=torch.float16, device=DEV)
    tables = torch.zeros(64, 2048, dtype=torch.int32, device=DEV)
    lens = torch.zeros(64, dtype=torch.int32, device=DEV)
    vals = {"q": t, "k_cache": t, "v_cache": t}
    out = torch.zeros(64, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _call(fn, out, wl, vals, tables, lens, err) == status
