"""pa_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (for example code running inside an engine's
execution phase, where all memory must be planned beforehand).  It uses a
workspace array built into the library instead of a caller-provided one.

Called through the C ABI (ctypes on libpa_gb300.so) and compared with the
existing pa_decode_attention on the same inputs, on two calls in a row (the
built-in workspace keeps the previous call's contents).  This file is
collected last on purpose.
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


@pytest.mark.parametrize("name", ["gqa", "opt13b"])
def test_noalloc_matches_decode_attention_twice(name):
    fn = _noalloc_fn()
    wl = synthetic.make(name)
    assert pa.decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                    wl.max_context_len) <= NOALLOC_BYTES
    vals = synthetic.make_values(wl, device=DEV)
    tables = torch.as_tensor(wl.block_tables, device=DEV)
    lens = torch.as_tensor(wl.context_lens, device=DEV)
    ref = pa.decode_attention(vals["q"], vals["k_cache"], vals["v_cache"], tables, lens,
                              wl.max_context_len, wl.scale)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call(fn, out, wl, vals, tables, lens, err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.all(torch.isfinite(out))
        assert float((out - ref).abs().max()) <= ATOL


def test_noalloc_rejects_sizes_beyond_its_array():
    fn = _noalloc_fn()
    # 64 sequences x 64 heads x 256 dims with 32K-token contexts need far more
    # than the built-in array; the call must refuse before enqueuing anything
    wl = SimpleNamespace(max_context_len=32768, num_seqs=64, num_heads=64, num_kv_heads=64,
                         head_dim=256, num_blocks=64 * 2048, scale=0.0625)
    assert pa.decode_workspace_size(64, 64, 64, 256, 32768) > NOALLOC_BYTES
    t = torch.zeros(1, dtype=torch.float16, device=DEV)
    tables = torch.zeros(64, 2048, dtype=torch.int32, device=DEV)
    lens = torch.zeros(64, dtype=torch.int32, device=DEV)
    vals = {"q": t, "k_cache": t, "v_cache": t}
    out = torch.zeros(1, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _call(fn, out, wl, vals, tables, lens, err) == 4      # PA_ERR_WORKSPACE
