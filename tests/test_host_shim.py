"""Host block manager and workload recipes, replayed against the worked
examples the pages print (tests/golden/*.txt carry the citations)."""
import math

import numpy as np
import pytest

from conftest import golden
from paged_kv_cache_pa_gb300 import synthetic
from paged_kv_cache_pa_gb300.block_manager import BlockLedger, OutOfBlocks, blocks_for


def _ints(v):
    return [int(x) for x in v]


def test_interleaved_sequences_tables():
    g = golden("interleaved_tables.txt")
    B, NB, steps = int(g["block_size"][0][0]), int(g["pool_blocks"][0][0]), int(g["steps"][0][0])
    rows = {int(r[0]): r for r in g["seq"]}
    prompts = {i: int(r[r.index("prompt") + 1]) for i, r in rows.items()}
    led = BlockLedger(NB, block_size=B)
    seqs = [led.new_sequence() for _ in rows]
    for t in range(steps):
        for i, s in enumerate(seqs):
            led.append(s, prompts[i] if t == 0 else 1)
    for i, r in rows.items():
        assert led.length(seqs[i]) == int(r[r.index("stored") + 1])
        assert led.table(seqs[i]) == _ints(r[r.index("table") + 1:])
    assert led.num_free == int(g["free"][0][0])
    assert led.take_copies() == []


def test_parallel_sampling_copy_on_write():
    g = golden("parallel_sampling.txt")
    B = int(g["block_size"][0][0])
    prompt, samples, new = (int(g[k][0][0]) for k in ("prompt", "samples", "new_tokens"))
    led = BlockLedger(64, block_size=B)
    first = led.new_sequence()
    led.append(first, prompt)
    assert len(led.table(first)) == int(g["prompt_blocks"][0][0])
    assert led.fills(first)[-1][1] == int(g["last_block_fill"][0][0])
    seqs = [first] + [led.fork(first) for _ in range(samples - 1)]
    for _ in range(new - 1):          # the first new token is sampled from the prompt
        for s in seqs:
            led.append(s, 1)
    in_use = led.num_blocks - led.num_free
    assert in_use == int(g["blocks_in_use"][0][0])
    assert samples * blocks_for(led.length(seqs[0]), B) == int(g["blocks_unshared"][0][0])
    copies = led.take_copies()
    assert len(copies) == int(g["cow_copies"][0][0])
    for row in g["table"]:
        assert led.table(seqs[int(row[0])]) == _ints(row[1:])
    # the copies are of the shared partial prompt block into fresh blocks
    assert all(src == 2 for src, _ in copies)


def test_figure6_block_table_walkthrough():
    g = golden("figure6_walkthrough.txt")
    B = int(g["block_size"][0][0])
    led = BlockLedger(8, block_size=B, free_order=_ints(g["free_order"][0]))
    seq = led.new_sequence()

    def fills():
        return [f"{b}:{n}" for b, n in led.fills(seq)]

    led.append(seq, 7)
    assert fills() == g["after_prompt"][0]
    led.append(seq, 1)                               # "fathers"
    assert fills() == g["after_token8"][0]
    slot = led.append(seq, 1)[0]                     # "brought"
    assert fills() == g["after_token9"][0]
    assert slot == int(g["slot_token9"][0][0])


def test_cow_trace_two_samples():
    g = golden("cow_trace.txt")
    led = BlockLedger(16, block_size=int(g["block_size"][0][0]),
                      free_order=_ints(g["free_order"][0]))
    a1 = led.new_sequence()
    led.append(a1, int(g["prompt"][0][0]))
    a2 = led.fork(a1)
    led.append(a1, 1)
    led.append(a2, 1)
    assert [tuple(p) for p in led.take_copies()] == [tuple(_ints(g["copies"][0]))]
    assert led.table(a1) == _ints(g["table_A1"][0])
    assert led.table(a2) == _ints(g["table_A2"][0])
    for item in g["refs"][0]:
        b, r = item.split(":")
        assert led.refcount(int(b)) == int(r)


def test_free_returns_blocks_and_out_of_blocks_changes_nothing():
    led = BlockLedger(4)
    s = led.new_sequence()
    led.append(s, 64)
    t = led.new_sequence()
    with pytest.raises(OutOfBlocks):
        led.append(t, 1)
    assert led.table(t) == [] and led.length(t) == 0 and led.num_free == 0
    led.release(s)
    assert led.num_free == 4 and all(r == 0 for r in led.refcounts())


def test_append_is_all_or_nothing():
    """A shared partial last block plus spill blocks beyond the free count:
    the append raises and leaves tables, counts and the copy list alone."""
    led = BlockLedger(4, block_size=16)
    a = led.new_sequence()
    led.append(a, 40)                                # 3 blocks, the last partial
    b = led.fork(a)
    assert led.blocks_needed(b, 1) == 1              # copy of the shared partial block
    assert led.blocks_needed(b, 40) == 3             # copy + two spill blocks
    before = (led.table(a), led.table(b), led.num_free, led.refcounts())
    with pytest.raises(OutOfBlocks):
        led.append(b, 40)
    assert (led.table(a), led.table(b), led.num_free, led.refcounts()) == before
    assert led.take_copies() == []
    assert led.append(b, 1) == [3 * 16 + 8]          # copy-on-write into block 3
    assert led.table(b) == [0, 1, 3] and led.take_copies() == [(2, 3)]


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", [n for n in synthetic.CONFIGS])
def test_workload_tables_and_slots_are_consistent(name):
    wl = synthetic.make(name)
    S = wl.num_seqs
    assert wl.context_lens.min() >= 1
    used = []
    for s in range(S):
        L = int(wl.context_lens[s])
        nb = blocks_for(L)
        row = wl.block_tables[s]
        assert np.all(row[:nb] >= 0) and np.all(row[:nb] < wl.num_blocks)
        assert np.all(row[nb:] == -1)
        used.extend(row[:nb].tolist())
        # the step's new token is position L-1
        pos = L - 1
        assert wl.slot_mapping[s] == row[pos // 16] * 16 + pos % 16
    if name != "beams":
        assert len(set(used)) == len(used)            # no sharing outside beams
    else:
        assert len(set(used)) < len(used)             # beams share prompt blocks
        # copy-on-write destinations are fresh and distinct; sources are shared
        dst = wl.copy_pairs[:, 1]
        assert len(set(dst.tolist())) == len(dst)
        assert not set(dst.tolist()) & set(wl.copy_pairs[:, 0].tolist())
    slots = wl.slot_mapping
    assert len(set(slots.tolist())) == S              # one slot per new token


def test_workload_recipes_follow_the_stated_shapes():
    t = synthetic.make("tiny")
    assert (t.num_seqs, t.num_heads, t.num_kv_heads, t.head_dim, t.num_blocks) == (4, 8, 8, 64, 64)
    assert t.context_lens.max() <= 128
    o = synthetic.make("opt13b")
    assert (o.num_seqs, o.num_heads, o.head_dim, o.dtype) == (256, 40, 128, "f16")
    assert o.context_lens.max() <= 2048 and o.context_lens.min() >= 2
    assert o.num_blocks == sum(blocks_for(int(L)) for L in o.context_lens)
    q = synthetic.make("gqa")
    assert (q.num_heads, q.num_kv_heads, q.dtype) == (12, 2, "bf16")
    assert 512 <= q.context_lens.min() and q.context_lens.max() <= 4096
    # the GQA shape's KV bytes per token over 28 layers: 28 KiB
    assert 28 * 2 * q.num_kv_heads * q.head_dim * 2 == 28 * 1024
    lg = synthetic.make("long")
    assert lg.num_blocks * 40 * 16 * 128 * 2 * 2 == 60 * (1 << 30)
    assert 16384 <= lg.context_lens.min() and lg.context_lens.max() <= 32768
    b = synthetic.make("beams")
    assert b.num_seqs == 192 and b.context_lens.min() >= 513
    # beams of one group have equal length
    assert all(len(set(b.context_lens[i * 6:(i + 1) * 6].tolist())) == 1 for i in range(32))


def test_lognormal_reading():
    rng = np.random.default_rng(0)
    x = synthetic._lognormal_int(rng, 220.0, 200000, 1, 10 ** 9)
    assert abs(x.mean() / 220.0 - 1) < 0.02


@pytest.mark.parametrize("B", [8, 32, 64, 256])
def test_relayout_keeps_lengths_and_resolves_slots(B):
    """Re-laying a workload in B-token blocks keeps every length; each
    sequence gets ceil(L/B) distinct in-range blocks and the step's slot is
    position L-1 resolved through the new table."""
    wl = synthetic.make("gqa")
    r = synthetic.relayout(wl, B)
    assert r.block_size == B and np.array_equal(r.context_lens, wl.context_lens)
    assert r.num_blocks * B >= wl.num_blocks * wl.block_size
    used = []
    for s in range(r.num_seqs):
        L = int(r.context_lens[s])
        nb = blocks_for(L, B)
        row = r.block_tables[s]
        assert np.all(row[:nb] >= 0) and np.all(row[:nb] < r.num_blocks)
        assert np.all(row[nb:] == -1)
        used.extend(row[:nb].tolist())
        assert r.slot_mapping[s] == row[(L - 1) // B] * B + (L - 1) % B
    assert len(set(used)) == len(used)
    assert r.max_blocks_per_seq * B >= r.max_context_len
    o = synthetic.in_order(r)
    assert o.block_size == B and o.block_tables[0, 0] == 0
