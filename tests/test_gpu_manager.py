"""The native block manager driving the kernels: a beam-search-like trace
(prompts, forks, appends with copy-on-write) produces the copy pairs, slots,
tables and lengths of a decode step, which runs on the GPU and in the oracle
on the same inputs; then a beam group is swapped out to pinned host memory
and back into other block ids, and the batch's attention output is
unchanged to the bit."""
import numpy as np
import pytest
import torch

from paritylib import ATOL, codes, max_abs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import paged_kv_cache_pa_gb300 as pa  # noqa: E402
from paged_kv_cache_pa_gb300.manager import BlockManager  # noqa: E402

DEV = torch.device("cuda:0")


@pytest.mark.parametrize("B", [16, 8])
def test_manager_trace_drives_a_decode_step_and_a_swap(B):
    NB, NC, Hkv, G, D = 400, 64, 2, 6, 128
    H = Hkv * G
    rng = np.random.default_rng(B)
    bm = BlockManager(NB, num_cpu_blocks=NC, block_size=B)
    groups = []
    for prompt in (37, 100, 250):
        root = bm.new_sequence()
        bm.append(root, prompt)
        groups.append([root] + [bm.fork(root) for _ in range(3)])
    for _ in range(int(rng.integers(3, 9))):          # beams grow, copying shared blocks
        for g in groups:
            for s in g:
                bm.append(s, int(rng.integers(1, 4)))
    seqs = [s for g in groups for s in g]
    slots = np.concatenate([bm.append(s, 1) for s in seqs])      # the measured step
    pairs = bm.take_copies()
    assert len(pairs) > 0
    maxb = max(len(bm.table(s)) for s in seqs)
    tables, lens = bm.build_batch(seqs, maxb)
    S = len(seqs)

    gen = torch.Generator(device=DEV).manual_seed(B)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=DEV).to(torch.bfloat16)
    kc, vc = rnd(NB, Hkv, B, D), rnd(NB, Hkv, B, D)
    q, key, val = rnd(S, H, D), rnd(S, Hkv, D), rnd(S, Hkv, D)
    h = {n: codes(t) for n, t in (("kc", kc), ("vc", vc), ("q", q), ("key", key), ("val", val))}

    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.copy_blocks([kc], [vc], torch.as_tensor(pairs, device=DEV), error_word=err)
    pa.cache_write(key, val, kc, vc, torch.as_tensor(slots, device=DEV), error_word=err)
    t_d, l_d = torch.as_tensor(tables, device=DEV), torch.as_tensor(lens, device=DEV)
    scale = 1.0 / np.sqrt(D)
    out = pa.decode_attention(q, kc, vc, t_d, l_d, int(lens.max()), scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    oracle.copy_blocks([h["kc"]], [h["vc"]], pairs)
    oracle.cache_write(h["key"], h["val"], h["kc"], h["vc"], slots)
    want = oracle.decode_attention(h["q"], h["kc"], h["vc"], tables, lens, scale, "bf16")
    assert np.array_equal(codes(kc), h["kc"]) and np.array_equal(codes(vc), h["vc"])
    assert max_abs(out.cpu().numpy(), want) <= ATOL

    # swap group 1 out, let another sequence reuse and overwrite its blocks, swap it back in
    g1 = groups[1]
    hk = torch.empty(NC, Hkv, B, D, dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    p_out = bm.swap_out(g1)
    pa.swap_blocks([hk], [hv], [kc], [vc], torch.as_tensor(p_out, device=DEV), error_word=err)
    intruder = bm.new_sequence()
    n_free = bm.num_free_gpu
    junk_slots = bm.append(intruder, (n_free - len(p_out)) * B)   # leaves room for g1 only
    kc[torch.as_tensor(junk_slots // B, device=DEV)] = 0   # clobber the reused blocks
    vc[torch.as_tensor(junk_slots // B, device=DEV)] = 0
    p_in = bm.swap_in(g1)
    assert set(p_in[:, 1].tolist()).isdisjoint(set((junk_slots // B).tolist()))
    pa.swap_blocks([kc], [vc], [hk], [hv], torch.as_tensor(p_in, device=DEV), error_word=err)
    tables2, lens2 = bm.build_batch(seqs, maxb)
    assert np.array_equal(lens2, lens)
    assert not np.array_equal(tables2[4:8], tables[4:8])   # other block ids now
    assert np.array_equal(tables2[:4], tables[:4]) and np.array_equal(tables2[8:], tables[8:])
    # the same batch with only block ids changed: the same arithmetic in the
    # same order, so the same bits
    out2 = pa.decode_attention(q, kc, vc, torch.as_tensor(tables2, device=DEV), l_d,
                               int(lens.max()), scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out2, out)
