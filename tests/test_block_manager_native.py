"""The native block manager (C++ behind include/pa_bm.h): the pages' printed
worked examples replayed exactly, equivalence with the Python host shim on
seeded random traces, all-or-nothing failures, swap of sequence groups, and
the batch inputs it builds for the kernels.  Host code only: runs on CPU."""
import numpy as np
import pytest

from conftest import golden
from paged_kv_cache_pa_gb300 import PaError
from paged_kv_cache_pa_gb300.block_manager import BlockLedger, OutOfBlocks, blocks_for
from paged_kv_cache_pa_gb300.manager import BlockManager, NoFreeBlocks


def _ints(v):
    return [int(x) for x in v]


# ---------------------------------------------------------------------------
# the pages' worked examples (tests/golden/*.txt carry the citations)
# ---------------------------------------------------------------------------

def test_interleaved_sequences_tables():
    g = golden("interleaved_tables.txt")
    B, NB, steps = int(g["block_size"][0][0]), int(g["pool_blocks"][0][0]), int(g["steps"][0][0])
    rows = {int(r[0]): r for r in g["seq"]}
    prompts = {i: int(r[r.index("prompt") + 1]) for i, r in rows.items()}
    bm = BlockManager(NB, block_size=B)
    seqs = [bm.new_sequence() for _ in rows]
    for t in range(steps):
        for i, s in enumerate(seqs):
            bm.append(s, prompts[i] if t == 0 else 1)
    for i, r in rows.items():
        assert bm.seq_len(seqs[i]) == int(r[r.index("stored") + 1])
        assert bm.table(seqs[i]) == _ints(r[r.index("table") + 1:])
    assert bm.num_free_gpu == int(g["free"][0][0])
    assert len(bm.take_copies()) == 0


def test_parallel_sampling_copy_on_write():
    g = golden("parallel_sampling.txt")
    B = int(g["block_size"][0][0])
    prompt, samples, new = (int(g[k][0][0]) for k in ("prompt", "samples", "new_tokens"))
    bm = BlockManager(64, block_size=B)
    first = bm.new_sequence()
    bm.append(first, prompt)
    assert len(bm.table(first)) == int(g["prompt_blocks"][0][0])
    assert bm.fills(first)[-1][1] == int(g["last_block_fill"][0][0])
    seqs = [first] + [bm.fork(first) for _ in range(samples - 1)]
    for _ in range(new - 1):
        for s in seqs:
            bm.append(s, 1)
    assert 64 - bm.num_free_gpu == int(g["blocks_in_use"][0][0])
    assert samples * blocks_for(bm.seq_len(seqs[0]), B) == int(g["blocks_unshared"][0][0])
    copies = bm.take_copies()
    assert len(copies) == int(g["cow_copies"][0][0])
    for row in g["table"]:
        assert bm.table(seqs[int(row[0])]) == _ints(row[1:])
    assert all(int(src) == 2 for src, _ in copies)


def test_figure6_block_table_walkthrough():
    g = golden("figure6_walkthrough.txt")
    B = int(g["block_size"][0][0])
    bm = BlockManager(8, block_size=B, free_order=_ints(g["free_order"][0]))
    s = bm.new_sequence()

    def fills():
        return [f"{b}:{n}" for b, n in bm.fills(s)]

    bm.append(s, 7)
    assert fills() == g["after_prompt"][0]
    bm.append(s, 1)
    assert fills() == g["after_token8"][0]
    slot = int(bm.append(s, 1)[0])
    assert fills() == g["after_token9"][0]
    assert slot == int(g["slot_token9"][0][0])


def test_cow_trace_two_samples():
    g = golden("cow_trace.txt")
    bm = BlockManager(16, block_size=int(g["block_size"][0][0]),
                      free_order=_ints(g["free_order"][0]))
    a1 = bm.new_sequence()
    bm.append(a1, int(g["prompt"][0][0]))
    a2 = bm.fork(a1)
    bm.append(a1, 1)
    bm.append(a2, 1)
    assert [tuple(p) for p in bm.take_copies().tolist()] == [tuple(_ints(g["copies"][0]))]
    assert bm.table(a1) == _ints(g["table_A1"][0])
    assert bm.table(a2) == _ints(g["table_A2"][0])
    for item in g["refs"][0]:
        b, r = item.split(":")
        assert bm.refcount(int(b)) == int(r)


# ---------------------------------------------------------------------------
# the same behaviour as the Python block ledger on random traces
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,B", [(0, 16), (1, 16), (2, 8), (3, 4), (4, 64)])
def test_random_trace_matches_the_python_ledger(seed, B):
    """Seeded random create / append / fork / free operations on the native
    manager and the Python ledger: identical tables, lengths, slots,
    copy-on-write pairs, free counts and reference counts after every
    operation, including the refused appends when the pool runs dry."""
    rng = np.random.default_rng(seed)
    NB = 96
    bm = BlockManager(NB, block_size=B)
    led = BlockLedger(NB, block_size=B)
    live = {}                                      # native id -> ledger id
    failures = 0
    for _ in range(600):
        op = rng.choice(["new", "append", "append", "append", "fork", "free"])
        if op == "new" or not live:
            s = bm.new_sequence()
            live[s] = led.new_sequence()
            op, n = "append", int(rng.integers(1, 3 * B))
            target = s
        else:
            target = int(rng.choice(list(live)))
            n = int(rng.integers(0, 2 * B)) if rng.random() < 0.3 else 1
        if op == "append":
            try:
                want = led.append(live[target], n)
            except OutOfBlocks:
                # both refuse and both stay as they were
                with pytest.raises(NoFreeBlocks):
                    bm.append(target, n)
                failures += 1
            else:
                got = bm.append(target, n)
                assert got.tolist() == want
        elif op == "fork":
            c = bm.fork(target)
            live[c] = led.fork(live[target])
        elif op == "free":
            bm.free(target)
            led.release(live.pop(target))
        for s, ls in live.items():
            assert bm.table(s) == led.table(ls) and bm.seq_len(s) == led.length(ls)
        assert bm.num_free_gpu == led.num_free
        assert [tuple(p) for p in bm.take_copies().tolist()] == led.take_copies()
        assert [bm.refcount(b) for b in range(NB)] == led.refcounts()
    assert failures > 0                            # the trace ran the pool dry


def test_append_is_all_or_nothing():
    bm = BlockManager(4, block_size=16)
    a = bm.new_sequence()
    bm.append(a, 40)                               # 3 blocks
    b = bm.fork(a)                                 # shares all three
    assert bm.blocks_needed(b, 1) == 1             # copy of the shared partial block
    assert bm.blocks_needed(b, 40) == 3            # copy + two new blocks
    before = (bm.table(a), bm.table(b), bm.num_free_gpu, [bm.refcount(i) for i in range(4)])
    with pytest.raises(NoFreeBlocks):
        bm.append(b, 40)
    assert (bm.table(a), bm.table(b), bm.num_free_gpu,
            [bm.refcount(i) for i in range(4)]) == before
    assert len(bm.take_copies()) == 0
    slots = bm.append(b, 1)                        # fits: copy-on-write into block 3
    assert bm.table(b) == [0, 1, 3] and slots.tolist() == [3 * 16 + 8]
    assert bm.take_copies().tolist() == [[2, 3]]


def test_errors_leave_the_manager_unchanged():
    bm = BlockManager(8, block_size=16)
    with pytest.raises(PaError):
        bm.append(12345, 1)
    with pytest.raises(PaError):
        bm.fork(7)
    with pytest.raises(PaError):
        BlockManager(0)
    with pytest.raises(PaError):
        BlockManager(8, free_order=[1, 1])
    s = bm.new_sequence()
    bm.append(s, 3)
    with pytest.raises(PaError):
        bm.build_batch([s, 99], 4)
    with pytest.raises(PaError):
        bm.build_batch([s], 0)
    assert bm.num_free_gpu == 7


# ---------------------------------------------------------------------------
# swap of sequence groups to the CPU space and back
# ---------------------------------------------------------------------------

def test_swap_group_out_and_in():
    """A group (a prompt and two forks sharing it) moves to the CPU space:
    one CPU block per distinct GPU block, reference counts carried over,
    GPU blocks freed; swapping in gives new GPU ids and (cpu, gpu) pairs
    that map every block back; tables stay consistent throughout."""
    bm = BlockManager(16, num_cpu_blocks=8, block_size=4)
    a = bm.new_sequence()
    bm.append(a, 10)                               # blocks 0,1,2 (2 half full)
    b, c = bm.fork(a), bm.fork(a)
    bm.append(b, 1)                                # b copies block 2 -> 3
    bm.take_copies()
    other = bm.new_sequence()
    bm.append(other, 5)                            # blocks 4, 5: not in the group
    free_gpu = bm.num_free_gpu
    ta, tb, tc = bm.table(a), bm.table(b), bm.table(c)
    pairs = bm.swap_out([a, b, c])
    gpu_ids = [int(x) for x in pairs[:, 0]]
    assert gpu_ids == [0, 1, 2, 3]                 # distinct blocks, first use order
    assert bm.num_free_gpu == free_gpu + 4 and bm.num_free_cpu == 4
    m = {int(g): int(h) for g, h in pairs}
    assert bm.table(a) == [m[x] for x in ta] and bm.table(b) == [m[x] for x in tb]
    assert bm.refcount(m[0], on_cpu=True) == 3 and bm.refcount(m[3], on_cpu=True) == 1
    assert bm.on_cpu(a) and not bm.on_cpu(other)
    with pytest.raises(PaError):
        bm.append(a, 1)                            # swapped out: no appends
    with pytest.raises(PaError):
        bm.build_batch([a], 4)
    bm.append(other, 20)                           # the freed GPU blocks are reused
    back = bm.swap_in([a, b, c])
    assert [int(x) for x in back[:, 0]] == [m[x] for x in gpu_ids]
    n = {int(h): int(g) for h, g in back}
    assert bm.table(a) == [n[m[x]] for x in ta]
    assert bm.table(c) == [n[m[x]] for x in tc]
    assert bm.num_free_cpu == 8 and not bm.on_cpu(b)
    assert bm.refcount(bm.table(a)[0]) == 3
    tables, lens = bm.build_batch([a, b, c, other], 8)
    assert lens.tolist() == [10, 11, 10, 25]
    assert tables[1, :3].tolist() == bm.table(b) and tables[1, 3] == -1


def test_swap_refuses_partial_groups_and_full_space():
    bm = BlockManager(8, num_cpu_blocks=2, block_size=4)
    a = bm.new_sequence()
    bm.append(a, 8)
    b = bm.fork(a)
    with pytest.raises(PaError):                   # b still holds a's blocks
        bm.swap_out([a])
    bm.append(a, 4)                                # a: 3 blocks, 2 shared with b
    with pytest.raises(NoFreeBlocks):              # 3 distinct blocks, space for 2
        bm.swap_out([a, b])
    assert not bm.on_cpu(a) and bm.num_free_cpu == 2
    bm.free(b)
    c = bm.new_sequence()
    bm.append(c, 8)
    assert bm.swap_out([c]).shape == (2, 2)
    bm.free(c)                                     # freeing a swapped sequence frees CPU blocks
    assert bm.num_free_cpu == 2


def test_build_batch_pads_tables():
    bm = BlockManager(32, block_size=16)
    seqs = []
    for L in (1, 16, 17, 100):
        s = bm.new_sequence()
        bm.append(s, L)
        seqs.append(s)
    tables, lens = bm.build_batch(seqs, 8)
    assert lens.tolist() == [1, 16, 17, 100]
    for i, s in enumerate(seqs):
        t = bm.table(s)
        assert tables[i, :len(t)].tolist() == t and np.all(tables[i, len(t):] == -1)
