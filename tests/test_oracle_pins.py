"""Pins for the CPU oracle: each check ties it to something other than itself
(a library routine, a closed form, an invariant the pages state, brute force
at high precision), chosen so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them."""
import math

import numpy as np
import pytest
import torch

from conftest import golden

BLOCK = 16


# ---------------------------------------------------------------------------
# 16-bit float codes
# ---------------------------------------------------------------------------

def test_f16_decode_all_codes_match_numpy(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint16)
    got = oracle_mod.half_to_double(codes, "f16")
    want = codes.view(np.float16).astype(np.float64)
    assert np.array_equal(got, want, equal_nan=True)


def test_bf16_decode_all_codes_match_torch(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint16)
    got = oracle_mod.half_to_double(codes, "bf16")
    want = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want, equal_nan=True)


def _encode_cases(rng):
    base = [0.0, -0.0, 1.0, -1.0, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504.0, 65519.99, 65520.0,
            1e6, -1e6, 2 ** -24, 2 ** -25, 2 ** -25 * 1.0000001, 3 * 2 ** -26, 6e-8, 2 ** -14,
            2 ** -14 * (1 - 2 ** -11), math.inf, -math.inf, 3.0e38, 3.4e38, 1e-40, 1e-45]
    r = np.concatenate([rng.standard_normal(20000), rng.standard_normal(20000) * 1e-5,
                        rng.standard_normal(20000) * 1e4, np.array(base)])
    return r


def test_f16_encode_matches_numpy_rne(oracle_mod):
    x = _encode_cases(np.random.default_rng(0))
    got = oracle_mod.double_to_half(x, "f16")
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_encode_matches_torch_rne(oracle_mod):
    # float32-representable inputs, so torch's float32 -> bfloat16 rounding is
    # the only rounding on both sides
    x = _encode_cases(np.random.default_rng(1)).astype(np.float32).astype(np.float64)
    got = oracle_mod.double_to_half(x, "bf16")
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(got, want.view(np.uint16))


def test_encode_of_nan_is_nan(oracle_mod):
    for dt in ("f16", "bf16"):
        c = oracle_mod.double_to_half(np.array([np.nan]), dt)
        assert np.isnan(oracle_mod.half_to_double(c, dt))[0]


# ---------------------------------------------------------------------------
# helpers: small paged problems built by hand
# ---------------------------------------------------------------------------

def _codes(x, dtype):
    t = torch.as_tensor(np.asarray(x, np.float32))
    t = t.to(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _paged_problem(rng, lens, H, Hkv, D, dtype="f16", extra_blocks=3):
    """Random q/K/V for the given lengths, blocks scattered over a pool."""
    lens = np.asarray(lens, np.int32)
    nbs = [-(-int(L) // BLOCK) for L in lens]
    NB = sum(nbs) + extra_blocks
    perm = rng.permutation(NB)
    maxb = max(max(nbs), 1)
    tables = np.full((len(lens), maxb), -1, np.int32)
    pos = 0
    for s, n in enumerate(nbs):
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    q = _codes(rng.standard_normal((len(lens), H, D)), dtype)
    kc = _codes(rng.standard_normal((NB, Hkv, BLOCK, D)), dtype)
    vc = _codes(rng.standard_normal((NB, Hkv, BLOCK, D)), dtype)
    return q, kc, vc, tables, lens


def _gather(oracle_mod, pool, tables, lens, s, dtype):
    """[Hkv][L][D] float64 rows of sequence s, gathered by plain indexing."""
    L = int(lens[s])
    rows = [pool[tables[s, t // BLOCK], :, t % BLOCK, :] for t in range(L)]
    return oracle_mod.half_to_double(np.stack(rows, axis=1), dtype)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,Hkv,D,dtype", [(4, 4, 8, "f16"), (6, 2, 16, "bf16"),
                                           (8, 1, 32, "f16")])
def test_attention_matches_sdpa_on_gathered_kv(oracle_mod, H, Hkv, D, dtype):
    """Paged gather == dense attention: torch SDPA on CPU float64, with the KV
    heads repeated to the query heads consecutively (the grouped-query
    reading), and the caller's scale."""
    rng = np.random.default_rng(H * 100 + D)
    lens = [1, 15, 16, 17, 33, 50]
    q, kc, vc, tables, lens = _paged_problem(rng, lens, H, Hkv, D, dtype)
    scale = 0.37
    got = oracle_mod.decode_attention(q, kc, vc, tables, lens, scale, dtype)
    G = H // Hkv
    for s in range(len(lens)):
        K = torch.from_numpy(_gather(oracle_mod, kc, tables, lens, s, dtype))
        V = torch.from_numpy(_gather(oracle_mod, vc, tables, lens, s, dtype))
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        Q = torch.from_numpy(oracle_mod.half_to_double(q[s], dtype))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)[:, 0, :]
        np.testing.assert_allclose(got[s], ref.numpy(), rtol=0, atol=1e-12)


def test_paged_equals_contiguous_bitwise(oracle_mod):
    """Same K/V stored in scattered blocks vs in identity order: identical bits
    (the attention depends only on the tokens, not on where they live)."""
    rng = np.random.default_rng(7)
    H, Hkv, D = 4, 2, 16
    q, kc, vc, tables, lens = _paged_problem(rng, [5, 40, 64, 17], H, Hkv, D, extra_blocks=0)
    maxb = tables.shape[1]
    S = len(lens)
    # identity layout: sequence s owns blocks s*maxb .. s*maxb+maxb-1
    kc2 = np.zeros((S * maxb, Hkv, BLOCK, D), np.uint16)
    vc2 = np.zeros_like(kc2)
    t2 = np.full_like(tables, -1)
    for s in range(S):
        n = -(-int(lens[s]) // BLOCK)
        for j in range(n):
            kc2[s * maxb + j] = kc[tables[s, j]]
            vc2[s * maxb + j] = vc[tables[s, j]]
            t2[s, j] = s * maxb + j
    a = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.25, "f16")
    b = oracle_mod.decode_attention(q, kc2, vc2, t2, lens, 0.25, "f16")
    assert np.array_equal(a, b)


def _relayout(rows_k, rows_v, lens, B, rng):
    """Store per-sequence token rows ([Hkv][L][D] codes) into a pool of
    B-token blocks at scattered places; returns (kc, vc, tables)."""
    S = len(lens)
    Hkv, D = rows_k[0].shape[0], rows_k[0].shape[2]
    nbs = [-(-int(L) // B) for L in lens]
    NB = sum(nbs) + 2
    perm = rng.permutation(NB)
    tables = np.full((S, max(max(nbs), 1)), -1, np.int32)
    kc = rng.integers(0, 1 << 16, (NB, Hkv, B, D), dtype=np.uint16)   # junk outside contexts
    vc = rng.integers(0, 1 << 16, (NB, Hkv, B, D), dtype=np.uint16)
    pos = 0
    for s in range(S):
        tables[s, :nbs[s]] = perm[pos:pos + nbs[s]]
        pos += nbs[s]
        for t in range(int(lens[s])):
            kc[tables[s, t // B], :, t % B, :] = rows_k[s][:, t, :]
            vc[tables[s, t // B], :, t % B, :] = rows_v[s][:, t, :]
    return kc, vc, tables


def test_block_size_does_not_change_the_output(oracle_mod):
    """The block size B is a storage parameter: the same tokens stored in
    blocks of 1, 3, 8, 16, 32, 64 or 256 tokens give bit-identical outputs
    (same tokens, same summation order), and match SDPA on the dense rows.
    A block size hard-coded anywhere (t / 16) fails every B but 16; junk
    outside the contexts makes a read past L visible."""
    rng = np.random.default_rng(21)
    H, Hkv, D, dtype = 6, 2, 16, "bf16"
    lens = np.array([1, 7, 8, 9, 31, 64, 100, 257], np.int32)
    q = _codes(rng.standard_normal((len(lens), H, D)), dtype)
    rows_k = [_codes(rng.standard_normal((Hkv, int(L), D)), dtype) for L in lens]
    rows_v = [_codes(rng.standard_normal((Hkv, int(L), D)), dtype) for L in lens]
    outs = {}
    for B in (1, 3, 8, 16, 32, 64, 256):
        kc, vc, tables = _relayout(rows_k, rows_v, lens, B, np.random.default_rng(B))
        outs[B] = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.3, dtype)
        bw = oracle_mod.decode_attention_blockwise(q, kc, vc, tables, lens, 0.3, dtype)
        np.testing.assert_allclose(bw, outs[B], rtol=0, atol=1e-12)
    for B, o in outs.items():
        assert np.array_equal(o, outs[16]), B
    G = H // Hkv
    for s in range(len(lens)):
        K = torch.from_numpy(oracle_mod.half_to_double(rows_k[s], dtype)).repeat_interleave(G, 0)
        V = torch.from_numpy(oracle_mod.half_to_double(rows_v[s], dtype)).repeat_interleave(G, 0)
        Q = torch.from_numpy(oracle_mod.half_to_double(q[s], dtype))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=0.3)[:, 0, :]
        np.testing.assert_allclose(outs[8][s], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("B", [8, 64])
def test_cache_write_at_other_block_sizes(oracle_mod, B):
    """slot -> (slot // B, slot % B): the written rows are found there, and
    nothing else in the pool changes."""
    rng = np.random.default_rng(B)
    NB, Hkv, D, T = 7, 3, 8, 12
    kc = rng.integers(0, 1 << 16, (NB, Hkv, B, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, (NB, Hkv, B, D), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    key = rng.integers(0, 1 << 16, (T, Hkv, D), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, (T, Hkv, D), dtype=np.uint16)
    slots = rng.choice(NB * B, T, replace=False).astype(np.int64)
    slots[3] = -1
    oracle_mod.cache_write(key, val, kc, vc, slots)
    touched = np.zeros((NB, B), bool)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        b, o = divmod(int(sl), B)
        assert np.array_equal(kc[b, :, o], key[t]) and np.array_equal(vc[b, :, o], val[t])
        touched[b, o] = True
    keep = ~touched[:, None, :, None].repeat(Hkv, 1).repeat(D, 3)
    assert np.array_equal(kc[keep], k0[keep]) and np.array_equal(vc[keep], v0[keep])


def test_copy_blocks_at_block_size_32(oracle_mod):
    rng = np.random.default_rng(32)
    NB, Hkv, B, D = 9, 2, 32, 8
    ks = [rng.integers(0, 1 << 16, (NB, Hkv, B, D), dtype=np.uint16) for _ in range(2)]
    vs = [rng.integers(0, 1 << 16, (NB, Hkv, B, D), dtype=np.uint16) for _ in range(2)]
    before = [x.copy() for x in ks + vs]
    pairs = np.array([[1, 4], [2, 7]], np.int64)
    oracle_mod.copy_blocks(ks, vs, pairs)
    for x, x0 in zip(ks + vs, before):
        want = x0.copy()
        want[4], want[7] = x0[1], x0[2]
        assert np.array_equal(x, want)


def test_context_of_one_returns_v0(oracle_mod):
    rng = np.random.default_rng(3)
    q, kc, vc, tables, lens = _paged_problem(rng, [1, 1, 1], 6, 3, 32, "bf16")
    out = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.125, "bf16")
    for s in range(3):
        v0 = oracle_mod.half_to_double(vc[tables[s, 0], :, 0, :], "bf16")
        assert np.array_equal(out[s], np.repeat(v0, 2, axis=0))


def test_empty_context_is_zero(oracle_mod):
    rng = np.random.default_rng(4)
    q, kc, vc, tables, lens = _paged_problem(rng, [0, 3], 2, 2, 8)
    out = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.5, "f16")
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.all(np.isfinite(out))


def test_weights_are_a_convex_combination(oracle_mod):
    rng = np.random.default_rng(5)
    lens = [1, 7, 16, 31, 100]
    q, kc, vc, tables, lens = _paged_problem(rng, lens, 4, 4, 16)
    out, w = oracle_mod.attention_weights(q, kc, vc, tables, lens, 0.25, "f16")
    for s, L in enumerate(lens):
        ws = w[s, :, :L]
        assert np.all(ws >= 0)
        np.testing.assert_allclose(ws.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        # and the output is that combination of the V rows
        V = _gather(oracle_mod, vc, tables, lens, s, "f16")
        np.testing.assert_allclose(out[s], np.einsum("ht,htd->hd", ws, V), atol=1e-12)


def test_zero_scale_gives_mean_of_values(oracle_mod):
    rng = np.random.default_rng(6)
    q, kc, vc, tables, lens = _paged_problem(rng, [9, 48, 70], 4, 2, 16)
    out = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.0, "f16")
    for s in range(3):
        V = _gather(oracle_mod, vc, tables, lens, s, "f16")
        np.testing.assert_allclose(out[s], np.repeat(V.mean(axis=1), 2, axis=0), atol=1e-13)


def test_constant_keys_give_mean_of_values(oracle_mod):
    rng = np.random.default_rng(8)
    q, kc, vc, tables, lens = _paged_problem(rng, [20, 33], 2, 2, 8)
    kc[:] = kc[0, 0, 0]                        # every key row identical
    out = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.9, "f16")
    for s in range(2):
        V = _gather(oracle_mod, vc, tables, lens, s, "f16")
        np.testing.assert_allclose(out[s], V.mean(axis=1), atol=1e-13)


def test_dominant_key_selects_its_value(oracle_mod):
    rng = np.random.default_rng(9)
    D = 16
    q, kc, vc, tables, lens = _paged_problem(rng, [37], 1, 1, D)
    q[:] = _codes(np.eye(D)[0] * 8.0, "f16")[None, None, :]
    kc[:] = _codes(np.zeros(D), "f16")
    j = 29
    kc[tables[0, j // BLOCK], 0, j % BLOCK, 0] = _codes([64.0], "f16")[0]
    out = oracle_mod.decode_attention(q, kc, vc, tables, lens, 1.0, "f16")  # gap 512
    vj = oracle_mod.half_to_double(vc[tables[0, j // BLOCK], 0, j % BLOCK], "f16")
    np.testing.assert_allclose(out[0, 0], vj, rtol=0, atol=1e-15)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_blockwise_form_equals_tokenwise(oracle_mod, dtype):
    """The block-wise reformulation (per-block partial max / sum / weighted
    values, then a rescaling merge) computes the same output."""
    rng = np.random.default_rng(10)
    q, kc, vc, tables, lens = _paged_problem(rng, [1, 16, 17, 100, 250], 6, 3, 32, dtype)
    a = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.2, dtype)
    b = oracle_mod.decode_attention_blockwise(q, kc, vc, tables, lens, 0.2, dtype)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_token_permutation_invariance(oracle_mod):
    """Blocks may be processed in any order: permuting (k_t, v_t) jointly
    within the context leaves the output unchanged."""
    rng = np.random.default_rng(11)
    q, kc, vc, tables, lens = _paged_problem(rng, [45, 80], 4, 4, 16)
    a = oracle_mod.decode_attention(q, kc, vc, tables, lens, 0.3, "f16")
    kc2, vc2 = kc.copy(), vc.copy()
    for s, L in enumerate(lens):
        pos = [(tables[s, t // BLOCK], t % BLOCK) for t in range(L)]
        perm = rng.permutation(L)
        for t, u in enumerate(perm):
            kc2[pos[t][0], :, pos[t][1]] = kc[pos[u][0], :, pos[u][1]]
            vc2[pos[t][0], :, pos[t][1]] = vc[pos[u][0], :, pos[u][1]]
    b = oracle_mod.decode_attention(q, kc2, vc2, tables, lens, 0.3, "f16")
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_tiny_brute_force_high_precision(oracle_mod):
    """L <= 4, D = 4, integer-valued inputs; expected output from the
    definition evaluated with 50-digit arithmetic."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(12)
    for L in (1, 2, 3, 4):
        qv = rng.integers(-3, 4, 4)
        K = rng.integers(-3, 4, (L, 4))
        V = rng.integers(-5, 6, (L, 4))
        kc = np.zeros((1, 1, BLOCK, 4), np.uint16)
        vc = np.zeros_like(kc)
        kc[0, 0, :L] = _codes(K, "f16")
        vc[0, 0, :L] = _codes(V, "f16")
        q = _codes(qv, "f16")[None, None, :]
        tables = np.zeros((1, 1), np.int32)
        scale = 0.5
        out = oracle_mod.decode_attention(q, kc, vc, tables, np.array([L], np.int32), scale, "f16")
        x = [mp.mpf(scale) * sum(mp.mpf(int(qv[d])) * int(K[t, d]) for d in range(4)) for t in range(L)]
        w = [mp.e ** xt for xt in x]
        Z = sum(w)
        want = [sum(w[t] * int(V[t, d]) for t in range(L)) / Z for d in range(4)]
        np.testing.assert_allclose(out[0, 0], [float(v) for v in want], rtol=0, atol=1e-15)


def test_bad_block_id_is_reported(oracle_mod):
    rng = np.random.default_rng(13)
    q, kc, vc, tables, lens = _paged_problem(rng, [20], 1, 1, 8)
    tables[0, 1] = kc.shape[0]
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.decode_attention(q, kc, vc, tables, lens, 1.0, "f16")


# ---------------------------------------------------------------------------
# cache write and block copy
# ---------------------------------------------------------------------------

def test_cache_write_places_rows_and_touches_nothing_else(oracle_mod):
    rng = np.random.default_rng(20)
    NB, Hkv, D, T = 6, 3, 16, 7
    kc = rng.integers(0, 1 << 16, (NB, Hkv, BLOCK, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, (NB, Hkv, BLOCK, D), dtype=np.uint16)
    key = rng.integers(0, 1 << 16, (T, Hkv, D), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, (T, Hkv, D), dtype=np.uint16)
    slots = np.array([0, 17, 95, -1, 33, 48, 15], np.int64)
    k0, v0 = kc.copy(), vc.copy()
    oracle_mod.cache_write(key, val, kc, vc, slots)
    touched = np.zeros((NB, BLOCK), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        b, o = divmod(int(s), BLOCK)           # the page table's resolve()
        assert np.array_equal(kc[b, :, o, :], key[t])
        assert np.array_equal(vc[b, :, o, :], val[t])
        touched[b, o] = True
    by_slot = lambda a: a.transpose(0, 2, 1, 3)          # [block][offset][head][dim]
    assert np.array_equal(by_slot(kc)[~touched], by_slot(k0)[~touched])
    assert np.array_equal(by_slot(vc)[~touched], by_slot(v0)[~touched])


def test_cache_write_rejects_out_of_range_slot(oracle_mod):
    kc = np.zeros((2, 1, BLOCK, 8), np.uint16)
    vc = kc.copy()
    key = np.ones((1, 1, 8), np.uint16)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.cache_write(key, key, kc, vc, np.array([32], np.int64))
    assert not kc.any()


def test_copy_blocks_copies_every_layer_and_keeps_source(oracle_mod):
    rng = np.random.default_rng(21)
    NB, Hkv, D, layers = 9, 2, 8, 3
    ks = [rng.integers(0, 1 << 16, (NB, Hkv, BLOCK, D), dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 1 << 16, (NB, Hkv, BLOCK, D), dtype=np.uint16) for _ in range(layers)]
    k0 = [k.copy() for k in ks]
    v0 = [v.copy() for v in vs]
    pairs = np.array([[1, 4], [7, 2], [1, 8]], np.int64)
    oracle_mod.copy_blocks(ks, vs, pairs)
    dsts = set(pairs[:, 1].tolist())
    for l in range(layers):
        for src, dst in pairs:
            assert np.array_equal(ks[l][dst], k0[l][src])
            assert np.array_equal(vs[l][dst], v0[l][src])
        for b in range(NB):
            if b not in dsts:                     # sources and bystanders unchanged
                assert np.array_equal(ks[l][b], k0[l][b])
                assert np.array_equal(vs[l][b], v0[l][b])


def test_copy_blocks_rejects_out_of_range_pair(oracle_mod):
    ks = [np.zeros((2, 1, BLOCK, 8), np.uint16)]
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.copy_blocks(ks, [k.copy() for k in ks], np.array([[0, 2]], np.int64))


# ---------------------------------------------------------------------------
# pool layout against the pages' KV-size closed forms
# ---------------------------------------------------------------------------

def test_pool_layout_matches_kv_size_closed_forms():
    """Bytes per token per layer of the [blocks][kv_heads][16][head_dim] K and
    V pools, times the layers, equal the figures the pages print."""
    g = golden("kv_bytes_closed_forms.txt")
    for name, layers, hkv, d, elt, value, unit in (
            [k] + v for k, vs in g.items() for v in vs):
        layers, hkv, d, elt = int(layers), int(hkv), int(d), int(elt)
        nb = 3
        dt = torch.float16 if elt == 2 else None
        k = torch.empty(nb, hkv, BLOCK, d, dtype=dt)
        v = torch.empty(nb, hkv, BLOCK, d, dtype=dt)
        per_token = (k.nbytes + v.nbytes) // (nb * BLOCK) * layers
        if unit == "KiB_per_token":
            assert per_token / 1024 == float(value)
        elif unit == "GB_per_2048_tokens_rounded_2dp":
            assert round(per_token * 2048 / 1e9, 2) == float(value)
        elif unit == "bytes_per_16_token_block":
            assert per_token * BLOCK == int(value)
        else:  # pragma: no cover
            raise AssertionError(unit)
    # the paper summary's own arithmetic: 2 x 5120 x 40 x 2 bytes
    assert 2 * 5120 * 40 * 2 == 40 * (2 * 40 * 128 * 2) == 819200


# ---------------------------------------------------------------------------
# swap between two pools
# ---------------------------------------------------------------------------

def test_swap_out_and_back_in_restores_the_pool(oracle_mod):
    """Swap-out copies the named device blocks into free swap blocks, and
    swap-in of the same pairs reversed brings them back byte for byte; other
    blocks of both pools are untouched; the pairs map layer by layer."""
    rng = np.random.default_rng(19)
    L, ND, NS, Hkv, B, D = 3, 10, 7, 2, 8, 16
    gk = [rng.integers(0, 1 << 16, (ND, Hkv, B, D), dtype=np.uint16) for _ in range(L)]
    gv = [rng.integers(0, 1 << 16, (ND, Hkv, B, D), dtype=np.uint16) for _ in range(L)]
    ck = [rng.integers(0, 1 << 16, (NS, Hkv, B, D), dtype=np.uint16) for _ in range(L)]
    cv = [rng.integers(0, 1 << 16, (NS, Hkv, B, D), dtype=np.uint16) for _ in range(L)]
    g0 = [x.copy() for x in gk + gv]
    c0 = [x.copy() for x in ck + cv]
    out_pairs = np.array([[9, 0], [2, 5], [4, 3]], np.int64)          # (gpu, cpu)
    oracle_mod.swap_blocks(ck, cv, gk, gv, out_pairs)
    for l in range(L):
        for g, c in out_pairs:
            assert np.array_equal(ck[l][c], gk[l][g]) and np.array_equal(cv[l][c], gv[l][g])
        for c in set(range(NS)) - set(out_pairs[:, 1].tolist()):
            assert np.array_equal(ck[l][c], c0[l][c]) and np.array_equal(cv[l][c], c0[L + l][c])
    # the GPU blocks are freed and overwritten, then swapped back into other ids
    for x in gk + gv:
        x[[9, 2, 4]] = 0
    in_pairs = np.array([[0, 1], [5, 6], [3, 8]], np.int64)           # (cpu, new gpu)
    oracle_mod.swap_blocks(gk, gv, ck, cv, in_pairs)
    for l in range(L):
        for (g_old, _), (_, g_new) in zip(out_pairs, in_pairs):
            assert np.array_equal(gk[l][g_new], g0[l][g_old])
            assert np.array_equal(gv[l][g_new], g0[L + l][g_old])
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.swap_blocks(ck, cv, gk, gv, np.array([[0, NS]], np.int64))


# ---------------------------------------------------------------------------
# prefill (chunked prefill) attention
# ---------------------------------------------------------------------------

def _prefill_problem(rng, cases, H, Hkv, D, B, dtype):
    """(cached, new) token counts per sequence -> paged pools holding every
    sequence's full context, q rows of the new tokens, tables, qsl, lens."""
    S = len(cases)
    lens = np.array([c + n for c, n in cases], np.int32)
    qsl = np.concatenate([[0], np.cumsum([n for _, n in cases])]).astype(np.int32)
    rows_k = [_codes(rng.standard_normal((Hkv, int(L), D)), dtype) for L in lens]
    rows_v = [_codes(rng.standard_normal((Hkv, int(L), D)), dtype) for L in lens]
    kc, vc, tables = _relayout(rows_k, rows_v, lens, B, rng)
    q = _codes(rng.standard_normal((int(qsl[-1]), H, D)), dtype)
    return q, kc, vc, tables, qsl, lens, rows_k, rows_v


@pytest.mark.parametrize("H,Hkv,D,B,dtype", [(4, 4, 16, 16, "f16"), (6, 2, 32, 8, "bf16"),
                                             (8, 1, 16, 64, "f16")])
def test_prefill_matches_causal_sdpa(oracle_mod, H, Hkv, D, B, dtype):
    """Each sequence's new tokens against torch SDPA (CPU float64) on the
    gathered rows with an explicit causal mask: new token i at position
    c + i sees keys 0 .. c + i; grouped query heads repeated consecutively."""
    rng = np.random.default_rng(H * 10 + B)
    cases = [(0, 1), (0, 37), (20, 16), (100, 33), (5, 70), (64, 1)]
    q, kc, vc, tables, qsl, lens, rows_k, rows_v = _prefill_problem(rng, cases, H, Hkv, D, B,
                                                                    dtype)
    got = oracle_mod.prefill_attention(q, kc, vc, tables, qsl, lens, 0.21, dtype)
    G = H // Hkv
    for s, (c, n) in enumerate(cases):
        K = torch.from_numpy(oracle_mod.half_to_double(rows_k[s], dtype)).repeat_interleave(G, 0)
        V = torch.from_numpy(oracle_mod.half_to_double(rows_v[s], dtype)).repeat_interleave(G, 0)
        Q = torch.from_numpy(oracle_mod.half_to_double(q[qsl[s]:qsl[s + 1]], dtype))
        Q = Q.permute(1, 0, 2)                                     # [H][n][D]
        mask = torch.arange(c + n)[None, :] <= (c + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                               scale=0.21)
        np.testing.assert_allclose(got[qsl[s]:qsl[s + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def test_prefill_in_two_chunks_equals_one(oracle_mod):
    """Chunked prefill: the same new tokens prefilled in one call, or in two
    calls whose first covers only the earlier tokens (the cache then holds
    fewer tokens), give identical rows."""
    rng = np.random.default_rng(5)
    H, Hkv, D, B = 4, 2, 16, 16
    cases = [(10, 50), (0, 33)]
    q, kc, vc, tables, qsl, lens, _, _ = _prefill_problem(rng, cases, H, Hkv, D, B, "f16")
    whole = oracle_mod.prefill_attention(q, kc, vc, tables, qsl, lens, 0.3, "f16")
    first = [20, 12]                                   # new tokens in the first chunk
    q1 = np.concatenate([q[qsl[s]:qsl[s] + first[s]] for s in range(2)])
    qsl1 = np.array([0, first[0], first[0] + first[1]], np.int32)
    lens1 = np.array([cases[s][0] + first[s] for s in range(2)], np.int32)
    part1 = oracle_mod.prefill_attention(q1, kc, vc, tables, qsl1, lens1, 0.3, "f16")
    q2 = np.concatenate([q[qsl[s] + first[s]:qsl[s + 1]] for s in range(2)])
    qsl2 = np.array([0, cases[0][1] - first[0], q2.shape[0]], np.int32)
    part2 = oracle_mod.prefill_attention(q2, kc, vc, tables, qsl2, lens, 0.3, "f16")
    for s in range(2):
        a = np.concatenate([part1[qsl1[s]:qsl1[s + 1]], part2[qsl2[s]:qsl2[s + 1]]])
        assert np.array_equal(a, whole[qsl[s]:qsl[s + 1]])
