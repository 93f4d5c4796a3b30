"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test here is chosen so that a plausible slip in the oracle (a dropped scale,
a transposed operand, an off-by-one causal diagonal, a wrong GQA head map, a
wrong rotation direction, a log base mix-up) fails at least one of them.
"""

import json
import os

import numpy as np
import pytest
import scipy.special as sps

import oracle
from oracle import (CONTIGUOUS, STRIPED, ZIGZAG, causal_pair_counts, full_attention,
                    full_attention_rows, layout_positions, merge_partials, ring_partials,
                    ring_sim, tile_classes_bruteforce, tile_counts)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Layouts and causal pair counts
# ---------------------------------------------------------------------------

def test_printed_causal_pair_counts(golden_dir):
    g = _load(golden_dir, "causal_pair_counts.json")
    c = causal_pair_counts(g["num_devices"], g["block_size"], CONTIGUOUS)
    s = causal_pair_counts(g["num_devices"], g["block_size"], STRIPED)
    assert c["work"] == g["contiguous"]["work"]
    assert s["work"] == g["striped"]["work"]
    assert f"{c['imbalance']:.2f}" == g["contiguous"]["imbalance_2dp"]
    assert f"{s['imbalance']:.2f}" == g["striped"]["imbalance_2dp"]
    assert (c["total"] == s["total"]) is g["same_total"]


@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
@pytest.mark.parametrize("seq,n", [(8, 2), (12, 4), (128, 8), (4096, 32), (96, 8)])
def test_layout_is_a_permutation(layout, seq, n):
    if layout == ZIGZAG and seq % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    pos = layout_positions(layout, seq, n)
    assert sorted(pos.tolist()) == list(range(seq))
    s_n = seq // n
    for p in range(n):   # positions increase inside every shard
        assert np.all(np.diff(pos[p * s_n:(p + 1) * s_n]) > 0)


def test_layout_small_tables():
    # written out by hand from the three definitions
    assert layout_positions(CONTIGUOUS, 8, 2).tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    assert layout_positions(STRIPED, 8, 2).tolist() == [0, 2, 4, 6, 1, 3, 5, 7]
    assert layout_positions(ZIGZAG, 8, 2).tolist() == [0, 1, 6, 7, 2, 3, 4, 5]
    z = layout_positions(ZIGZAG, 12, 3)      # chunks of 2: p0={0,1,10,11}
    assert z[:4].tolist() == [0, 1, 10, 11]
    assert z[4:8].tolist() == [2, 3, 8, 9]
    assert z[8:].tolist() == [4, 5, 6, 7]


def test_zigzag_exact_balance():
    for n, blk in [(8, 16), (4, 8), (2, 64)]:
        z = causal_pair_counts(n, blk, ZIGZAG)
        assert len(set(z["work"])) == 1
        assert z["total"] == n * blk * (n * blk + 1) // 2


def test_layout_rejects_uneven():
    with pytest.raises(ValueError):
        layout_positions(CONTIGUOUS, 10, 4)
    with pytest.raises(ValueError):
        layout_positions(ZIGZAG, 12, 4)


# ---------------------------------------------------------------------------
# Plain attention
# ---------------------------------------------------------------------------

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_full_attention_matches_scipy():
    q, k, v = _rand((1, 2, 20, 8), 1), _rand((1, 2, 20, 8), 2), _rand((1, 2, 20, 8), 3)
    o, lse = full_attention(q, k, v)
    for h in range(2):
        s = q[0, h] @ k[0, h].T / np.sqrt(8)
        np.testing.assert_allclose(o[0, h], sps.softmax(s, axis=1) @ v[0, h], atol=1e-13)
        np.testing.assert_allclose(lse[0, h], sps.logsumexp(s, axis=1), atol=1e-13)


def test_full_attention_causal_matches_scipy():
    q, k, v = _rand((1, 1, 17, 4), 4), _rand((1, 1, 17, 4), 5), _rand((1, 1, 17, 4), 6)
    o, lse = full_attention(q, k, v, causal=True, scale=0.3)
    s = q[0, 0] @ k[0, 0].T * 0.3
    s[np.triu_indices(17, 1)] = -np.inf
    np.testing.assert_allclose(o[0, 0], sps.softmax(s, axis=1) @ v[0, 0], atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], sps.logsumexp(s, axis=1), atol=1e-13)
    # causal row 0 sees only key 0
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], 0.3 * q[0, 0, 0] @ k[0, 0, 0], atol=1e-14)


def test_full_attention_closed_forms():
    d = 16
    q = _rand((1, 1, 5, d), 7)
    kv = _rand((1, 1, 1, d), 8)
    k = np.repeat(kv, 9, axis=2)                # 9 identical keys
    v = _rand((1, 1, 9, d), 9)
    o, lse = full_attention(q, k, v)
    np.testing.assert_allclose(o[0, 0], np.repeat(v[0, 0].mean(0, keepdims=True), 5, 0), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.log(9) + (q[0, 0] @ kv[0, 0, 0]) / np.sqrt(d), atol=1e-13)


def test_full_attention_rows_sum_to_one():
    q, k = _rand((1, 1, 30, 8), 10), _rand((1, 1, 30, 8), 11)
    eye = np.eye(30)[None, None]                 # V = identity exposes the probabilities
    vv = np.zeros((1, 1, 30, 30)); vv[:] = eye
    qq = np.concatenate([q, np.zeros((1, 1, 30, 22))], axis=3)
    kk = np.concatenate([k, np.zeros((1, 1, 30, 22))], axis=3)
    for causal in (False, True):
        o, _ = full_attention(qq, kk, vv, causal=causal, scale=1 / np.sqrt(8))
        np.testing.assert_allclose(o[0, 0].sum(1), 1.0, atol=1e-14)
        assert np.all(o >= 0)


def test_gqa_head_mapping():
    q = _rand((2, 6, 11, 4), 12)
    k, v = _rand((2, 3, 11, 4), 13), _rand((2, 3, 11, 4), 14)
    o, lse = full_attention(q, k, v, causal=True)
    for b in range(2):
        for h in range(6):
            g = h // 2
            o1, l1 = full_attention(q[b:b + 1, h:h + 1], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1], causal=True)
            np.testing.assert_allclose(o[b, h], o1[0, 0], atol=1e-15)
            np.testing.assert_allclose(lse[b, h], l1[0, 0], atol=1e-15)


def test_full_attention_rows_equals_full():
    q = _rand((1, 4, 40, 8), 15)
    k, v = _rand((1, 2, 40, 8), 16), _rand((1, 2, 40, 8), 17)
    pos = layout_positions(ZIGZAG, 40, 4)
    o, lse = full_attention(q, k, v, causal=True, positions=pos)
    picks = [(0, h, r) for h in range(4) for r in (0, 1, 9, 10, 22, 39)]
    o2, l2 = full_attention_rows(q, k, v, picks, causal=True, positions=pos, chunk=5)
    for n, (b, h, r) in enumerate(picks):
        np.testing.assert_allclose(o2[n], o[b, h, r], atol=1e-14)
        np.testing.assert_allclose(l2[n], lse[b, h, r], atol=1e-14)


# ---------------------------------------------------------------------------
# The ring
# ---------------------------------------------------------------------------

def test_toy_ring_equals_attention(golden_dir):
    g = _load(golden_dir, "toy_ring.json")
    n, blk, d = g["n_devices"], g["tokens_per_device"], g["head_dim"]
    rng = np.random.default_rng(1)
    Q, K, V = (rng.normal(size=(n * blk, d)) for _ in range(3))
    o, lse = ring_sim(Q[None, None], K[None, None], V[None, None], n)
    s = Q @ K.T / np.sqrt(d)
    ref = sps.softmax(s, axis=1) @ V
    assert np.allclose(o[0, 0], ref)                      # the page's own check
    np.testing.assert_allclose(o[0, 0], ref, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], sps.logsumexp(s, axis=1), atol=1e-13)


def test_module23_example(golden_dir):
    torch = pytest.importorskip("torch")
    g = _load(golden_dir, "module23_exact.json")
    torch.manual_seed(0)
    q, k, v = (torch.randn(*g["shape_bhsd"]) for _ in range(3))
    q, k, v = q.double().numpy(), k.double().numpy(), v.double().numpy()
    d = q.shape[-1]
    ring, _ = ring_sim(q, k, v, g["num_devices"])
    s = q @ np.swapaxes(k, -1, -2) / np.sqrt(d)
    ref = sps.softmax(s, axis=-1) @ v
    assert np.abs(ring - ref).max() <= g["atol"]
    tri = np.triu(np.ones((96, 96), bool), 1)
    ref_c = sps.softmax(np.where(tri, np.finfo(np.float64).min, s), axis=-1) @ v
    ring_c, _ = ring_sim(q, k, v, g["num_devices"], causal=True)
    assert np.abs(ring_c - ref_c).max() <= g["atol"]
    np.testing.assert_allclose(ring_c, ref_c, atol=1e-12)


@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
def test_ring_layout_invariance(layout):
    # natural-order inputs, permuted into the layout, ringed, then un-permuted
    B, Hq, Hkv, S, d, n = 1, 4, 2, 48, 8, 4
    q, k, v = _rand((B, Hq, S, d), 20), _rand((B, Hkv, S, d), 21), _rand((B, Hkv, S, d), 22)
    pos = layout_positions(layout, S, n)
    o_ref, l_ref = full_attention(q, k, v, causal=True)
    o_l, l_l = ring_sim(q[:, :, pos], k[:, :, pos], v[:, :, pos], n, positions=pos, causal=True)
    back_o = np.empty_like(o_l); back_o[:, :, pos] = o_l
    back_l = np.empty_like(l_l); back_l[:, :, pos] = l_l
    np.testing.assert_allclose(back_o, o_ref, atol=1e-13)
    np.testing.assert_allclose(back_l, l_ref, atol=1e-13)


def test_ring_one_shard_is_attention():
    q, k, v = _rand((1, 2, 9, 4), 23), _rand((1, 1, 9, 4), 24), _rand((1, 1, 9, 4), 25)
    for causal in (False, True):
        a = ring_sim(q, k, v, 1, causal=causal)
        b = full_attention(q, k, v, causal=causal)
        np.testing.assert_allclose(a[0], b[0], atol=1e-14)
        np.testing.assert_allclose(a[1], b[1], atol=1e-14)


def test_ring_large_logits():
    # Q scaled so the running max moves a lot between blocks
    q = 4 * _rand((1, 1, 64, 16), 26)
    k, v = _rand((1, 1, 64, 16), 27), _rand((1, 1, 64, 16), 28)
    for causal in (False, True):
        a = ring_sim(q, k, v, 8, causal=causal, scale=1.0)
        b = full_attention(q, k, v, causal=causal, scale=1.0)
        np.testing.assert_allclose(a[0], b[0], atol=1e-12)
        np.testing.assert_allclose(a[1], b[1], rtol=1e-13)


# ---------------------------------------------------------------------------
# Partials and merging
# ---------------------------------------------------------------------------

def test_merge_of_halves_is_attention():
    q = _rand((1, 2, 10, 8), 30)
    k, v = _rand((1, 2, 14, 8), 31), _rand((1, 2, 14, 8), 32)
    oa, la = full_attention(q, k[:, :, :5], v[:, :, :5], scale=0.35)
    ob, lb = full_attention(q, k[:, :, 5:], v[:, :, 5:], scale=0.35)
    o, l = merge_partials(np.stack([oa, ob]), np.stack([la, lb]))
    # single-call reference on all 14 keys (q and keys have different lengths)
    s = np.einsum("bhqd,bhkd->bhqk", q, k) * 0.35
    np.testing.assert_allclose(o, np.einsum("bhqk,bhkd->bhqd", sps.softmax(s, -1), v), atol=1e-14)
    np.testing.assert_allclose(l, sps.logsumexp(s, -1), atol=1e-14)


def test_merge_ignores_empty_parts():
    o = _rand((3, 4, 6), 33)
    l = _rand((3, 4), 34)
    l[1] = -np.inf
    m1, l1 = merge_partials(o, l)
    m2, l2 = merge_partials(o[[0, 2]], l[[0, 2]])
    np.testing.assert_allclose(m1, m2, atol=1e-15)
    np.testing.assert_allclose(l1, l2, atol=1e-15)
    m3, l3 = merge_partials(o[:1], np.full((1, 4), -np.inf))
    assert np.all(m3 == 0) and np.all(np.isneginf(l3))


@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_partials_merge_to_ring(layout, causal):
    B, Hq, Hkv, S, d, n = 1, 2, 1, 24, 4, 3
    q, k, v = _rand((B, Hq, S, d), 40), _rand((B, Hkv, S, d), 41), _rand((B, Hkv, S, d), 42)
    pos = layout_positions(layout, S, n)
    op, lp = ring_partials(q, k, v, n, positions=pos, causal=causal)
    o, l = merge_partials(op, lp)
    o2, l2 = ring_sim(q, k, v, n, positions=pos, causal=causal)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(l, l2, atol=1e-13)
    # order independence: merging the steps in reverse order changes nothing
    o3, l3 = merge_partials(op[::-1], lp[::-1])
    np.testing.assert_allclose(o3, o2, atol=1e-13)
    if causal and layout == CONTIGUOUS:
        # shard 0 at step 1 holds the last block: strictly in the future
        assert np.all(np.isneginf(lp[1, :, :, : S // n]))


# ---------------------------------------------------------------------------
# Tile classification
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
@pytest.mark.parametrize("seq,n,tile", [(96, 4, 8), (64, 4, 5), (120, 3, 16), (64, 8, 4)])
def test_tile_counts_bruteforce(layout, seq, n, tile):
    if layout == ZIGZAG and seq % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    for causal in (True, False):
        a = tile_counts(layout, seq, n, causal=causal, tile=tile)
        b = tile_classes_bruteforce(layout, seq, n, causal=causal, tile=tile)
        for x, y in zip(a, b):
            assert x.tolist() == y.tolist()


def test_tile_counts_unit_tiles_are_pair_counts(golden_dir):
    # with 1x1 tiles, FULL counts are exactly the causal pairs of each device
    g = _load(golden_dir, "causal_pair_counts.json")
    for layout in (CONTIGUOUS, STRIPED):
        full, part, skip = tile_counts(layout, 128, 8, causal=True, tile=1)
        assert full.tolist() == g[layout]["work"]
        assert part.sum() == 0
        assert (full + skip).tolist() == [128 * 16] * 8


def test_tile_counts_closed_forms_seq32k():
    # 32768 tokens, 8 shards, 128x128 tiles: global tile a meets tiles b<a FULL,
    # b=a PARTIAL, b>a SKIP (both layouts keep tiles 128-aligned in position)
    full, part, skip = tile_counts(CONTIGUOUS, 32768, 8)
    for p in range(8):
        assert (full[p], part[p], skip[p]) == (1024 * p + 496, 32, 1024 * (7 - p) + 496)
    full, part, skip = tile_counts(ZIGZAG, 32768, 8)
    assert full.tolist() == [4080] * 8 and part.tolist() == [32] * 8 and skip.tolist() == [4080] * 8


def test_tile_counts_closed_forms_striped_131k():
    full, part, skip = tile_counts(STRIPED, 131072, 32)
    assert full.tolist() == [32 * 496] * 32
    assert part.tolist() == [32 * 32] * 32
    assert skip.tolist() == [32 * 496] * 32


def test_oracle_exports():
    for name in oracle.__all__:
        assert hasattr(oracle, name)


def test_attention_rows_equals_full():
    q = _rand((1, 2, 50, 8), 50)
    k, v = _rand((1, 1, 50, 8), 51), _rand((1, 1, 50, 8), 52)
    pos = layout_positions(STRIPED, 50, 5)
    o, lse = full_attention(q, k, v, causal=True)            # natural order
    rows = np.array([0, 3, 17, 49, 25])
    o2, l2 = oracle.attention_rows(q[0, 1, rows], k[0, 0], v[0, 0], q_positions=rows, causal=True, chunk=2)
    np.testing.assert_allclose(o2, o[0, 1, rows], atol=1e-14)
    np.testing.assert_allclose(l2, lse[0, 1, rows], atol=1e-14)
    # keys handed over in layout order with their positions give the same rows
    o3, l3 = oracle.attention_rows(q[0, 1, rows], k[0, 0, pos], v[0, 0, pos], q_positions=rows,
                                   k_positions=pos, causal=True)
    np.testing.assert_allclose(o3, o2, atol=1e-14)
    np.testing.assert_allclose(l3, l2, atol=1e-14)


# ---------------------------------------------------------------------------
# The K/V exchange (what each device holds at each step)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_pass_blocks_closed_form(n):
    # rows labelled by their starting position: after t exchanges, the rows of
    # slot p are those that started in slot (p - t) mod N, in their own order
    s_n, S = 4, 4 * n
    x = np.arange(2 * S, dtype=np.float64).reshape(1, 2, S, 1).repeat(3, axis=-1)
    for t in range(2 * n + 1):
        y = oracle.held_blocks(x, n, t)
        for p in range(n):
            src = (p - t) % n
            np.testing.assert_array_equal(y[..., p * s_n:(p + 1) * s_n, :], x[..., src * s_n:(src + 1) * s_n, :])
    np.testing.assert_array_equal(oracle.held_blocks(x, n, n), x)
    if n > 1:  # direction: device i sends to i+1, so slot 1 now holds slot 0's rows
        np.testing.assert_array_equal(oracle.pass_blocks(x, n)[..., s_n:2 * s_n, :], x[..., :s_n, :])


@pytest.mark.parametrize("layout", [CONTIGUOUS, ZIGZAG])
def test_held_blocks_give_ring_partials(layout):
    # attention of each device's rows over the block it holds at step t, with that
    # block's positions, is partial t of ring_partials
    B, Hq, Hkv, S, d, n = 1, 2, 1, 24, 4, 3
    q, k, v = _rand((B, Hq, S, d), 60), _rand((B, Hkv, S, d), 61), _rand((B, Hkv, S, d), 62)
    pos = layout_positions(layout, S, n)
    op, lp = ring_partials(q, k, v, n, positions=pos, causal=True)
    s_n = S // n
    for t in range(n):
        kh, vh = oracle.held_blocks(k, n, t), oracle.held_blocks(v, n, t)
        ph = oracle.held_blocks(pos.reshape(S, 1), n, t)[:, 0]
        for p in range(n):
            rows = slice(p * s_n, (p + 1) * s_n)
            for h in range(Hq):
                allowed = ph[rows][None, :] <= pos[rows][:, None]
                if not allowed.any():
                    assert np.all(np.isneginf(lp[t, 0, h, rows]))
                    continue
                o, l = oracle.attention_rows(q[0, h, rows], kh[0, 0, rows], vh[0, 0, rows],
                                             q_positions=pos[rows], k_positions=ph[rows], causal=True)
                ok = np.isfinite(l)
                np.testing.assert_allclose(o[ok], op[t, 0, h, rows][ok], atol=1e-13)
                np.testing.assert_allclose(l, lp[t, 0, h, rows], atol=1e-13)


# ---------------------------------------------------------------------------
# Backward pass
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(causal):
    # L = sum(O * dO); its gradient by central differences of full_attention
    B, Hq, Hkv, S, d = 1, 2, 1, 6, 3
    q, k, v, do = _rand((B, Hq, S, d), 70), _rand((B, Hkv, S, d), 71), _rand((B, Hkv, S, d), 72), _rand((B, Hq, S, d), 73)
    pos = layout_positions(ZIGZAG, S, 3)            # rows in a layout order, masked by position
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=causal, positions=pos)

    def loss(q_, k_, v_):
        o, _ = full_attention(q_, k_, v_, causal=causal, positions=pos)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{a + "_": t for a, t in args_p.items()}) -
                        loss(**{a + "_": t for a, t in args_m.items()})) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=1e-7, rtol=1e-6, err_msg=name)


def test_backward_special_cases():
    # one key: O = v, so dV = dO and nothing flows to q or k
    q, k, v, do = _rand((1, 1, 1, 4), 80), _rand((1, 1, 1, 4), 81), _rand((1, 1, 1, 4), 82), _rand((1, 1, 1, 4), 83)
    dq, dk, dv = oracle.attention_backward(q, k, v, do)
    np.testing.assert_allclose(dv, do, atol=1e-15)
    assert np.all(dq == 0) and np.all(dk == 0)
    # softmax rows sum to one, so each row of dS sums to zero and the rows of dK sum to zero
    q, k, v, do = _rand((1, 2, 16, 4), 84), _rand((1, 1, 16, 4), 85), _rand((1, 1, 16, 4), 86), _rand((1, 2, 16, 4), 87)
    for causal in (False, True):
        _, dk, _ = oracle.attention_backward(q, k, v, do, causal=causal)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_backward_equals_attention_backward(layout, causal):
    B, Hq, Hkv, S, d, n = 1, 4, 2, 24, 4, 3
    q, k, v, do = _rand((B, Hq, S, d), 90), _rand((B, Hkv, S, d), 91), _rand((B, Hkv, S, d), 92), _rand((B, Hq, S, d), 93)
    pos = layout_positions(layout, S, n)
    o, lse = full_attention(q, k, v, causal=causal, positions=pos)
    want = oracle.attention_backward(q, k, v, do, causal=causal, positions=pos)
    got = oracle.ring_backward(q, k, v, do, o, lse, n, positions=pos, causal=causal)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, atol=1e-12)


@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
def test_to_natural_inverts_the_layout(layout):
    S, n = 48, 4
    x = _rand((2, 3, S, 5), 100)
    pos = layout_positions(layout, S, n)
    np.testing.assert_array_equal(oracle.to_natural(x[..., pos, :], pos), x)
    lab = oracle.to_natural(np.arange(S, dtype=np.float64)[:, None][pos], pos)
    np.testing.assert_array_equal(lab[:, 0], np.arange(S))
    if layout == CONTIGUOUS:
        np.testing.assert_array_equal(oracle.to_natural(x, pos), x)


# ---------------------------------------------------------------------------
# Ulysses' all-to-all
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("layout", [CONTIGUOUS, STRIPED, ZIGZAG])
def test_ulysses_exchange(layout):
    N, B, H, S = 4, 2, 8, 32
    hl = H // N
    pos = layout_positions(layout, S, N)
    # label = (b, h, position) on the layout-ordered sequence side
    x = np.zeros((B, H, S, 3))
    x[..., 0] = np.arange(B)[:, None, None]
    x[..., 1] = np.arange(H)[None, :, None]
    x[..., 2] = pos[None, None, :]
    y = oracle.ulysses_seq_to_head(x, pos, N)
    for q in range(N):            # device q holds heads q*hl.., every position in order
        for hh in range(hl):
            np.testing.assert_array_equal(y[q, :, hh, :, 1], q * hl + hh)
            np.testing.assert_array_equal(y[q, :, hh, :, 2], np.broadcast_to(np.arange(S), (B, S)))
            np.testing.assert_array_equal(y[q, :, hh, :, 0], np.broadcast_to(np.arange(B)[:, None], (B, S)))
    np.testing.assert_array_equal(oracle.ulysses_head_to_seq(y, pos, N), x)


def test_ulysses_attention_equals_full():
    # exchange, ordinary causal attention per device (its heads, all tokens), exchange back
    N, B, Hq, Hkv, S, d = 2, 1, 4, 2, 16, 4
    pos = layout_positions(ZIGZAG, S, N)
    q, k, v = _rand((B, Hq, S, d), 110), _rand((B, Hkv, S, d), 111), _rand((B, Hkv, S, d), 112)
    ql, kl, vl = q[..., pos, :], k[..., pos, :], v[..., pos, :]        # layout order
    qh, kh, vh = (oracle.ulysses_seq_to_head(t, pos, N) for t in (ql, kl, vl))
    outs, lses = zip(*(full_attention(qh[p], kh[p], vh[p], causal=True) for p in range(N)))
    o = oracle.ulysses_head_to_seq(np.stack(outs), pos, N)
    lse = oracle.ulysses_head_to_seq(np.stack(lses)[..., None], pos, N)[..., 0]
    ow, lw = full_attention(ql, kl, vl, causal=True, positions=pos)
    np.testing.assert_allclose(o, ow, atol=1e-12)
    np.testing.assert_allclose(lse, lw, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_row_blocks(causal):
    B, Hq, Hkv, S, d = 1, 4, 2, 40, 8
    q, k, v, do = _rand((B, Hq, S, d), 120), _rand((B, Hkv, S, d), 121), _rand((B, Hkv, S, d), 122), _rand((B, Hq, S, d), 123)
    pos = layout_positions(STRIPED, S, 4)
    whole = oracle.attention_backward(q, k, v, do, causal=causal, positions=pos)
    blocked = oracle.attention_backward(q, k, v, do, causal=causal, positions=pos, block=7)
    for a, b in zip(whole, blocked):
        np.testing.assert_allclose(b, a, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_finite_differences(causal):
    # L = sum over the chosen rows of O_i . dO_i, by central differences of attention_rows
    S, d = 7, 3
    q_rows, do_rows = _rand((3, d), 130), _rand((3, d), 131)
    k, v = _rand((S, d), 132), _rand((S, d), 133)
    q_pos = np.array([5, 2, 4])
    key_idx = np.array([0, 2, 3, 5])
    dq, dk_part, dv_part = oracle.attention_backward_rows(q_rows, do_rows, q_pos, k, v, causal=causal,
                                                          key_idx=key_idx)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_rows(q_, k_, v_, q_positions=q_pos, causal=causal)
        return float((o * do_rows).sum())

    eps = 1e-6

    def num_grad(x, f, rows):
        g = np.zeros((len(rows), x.shape[1]))
        for a, r in enumerate(rows):
            for c in range(x.shape[1]):
                xp, xm = x.copy(), x.copy()
                xp[r, c] += eps
                xm[r, c] -= eps
                g[a, c] = (f(xp) - f(xm)) / (2 * eps)
        return g

    np.testing.assert_allclose(dq, num_grad(q_rows, lambda x: loss(x, k, v), range(3)), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dk_part, num_grad(k, lambda x: loss(q_rows, x, v), key_idx), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dv_part, num_grad(v, lambda x: loss(q_rows, k, x), key_idx), atol=1e-7, rtol=1e-6)
    if causal:   # keys after every chosen row get nothing
        _, dk_late, dv_late = oracle.attention_backward_rows(q_rows, do_rows, q_pos, k, v, causal=True,
                                                             key_idx=[S - 1])
        assert np.all(dk_late == 0) and np.all(dv_late == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_subsets_add_up(causal):
    # rows in a layout order, keys given by position; split the query rows into
    # interleaved subsets: dQ rows match, and the key-row parts add up to dK, dV
    B, Hq, Hkv, S, d = 1, 2, 1, 30, 4
    q, k, v, do = _rand((B, Hq, S, d), 140), _rand((B, Hkv, S, d), 141), _rand((B, Hkv, S, d), 142), _rand((B, Hq, S, d), 143)
    pos = layout_positions(ZIGZAG, S, 3)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=causal, positions=pos)
    keys = np.array([0, 7, 13, 29])
    dk_sum, dv_sum = np.zeros((len(keys), d)), np.zeros((len(keys), d))
    for h in range(Hq):
        for sub in (np.arange(0, S, 3), np.arange(1, S, 3), np.arange(2, S, 3)):
            dq_s, dk_p, dv_p = oracle.attention_backward_rows(q[0, h, sub], do[0, h, sub], pos[sub], k[0, 0], v[0, 0],
                                                              k_pos=pos, causal=causal, key_idx=keys)
            np.testing.assert_allclose(dq_s, dq[0, h, sub], atol=1e-13)
            dk_sum += dk_p
            dv_sum += dv_p
    np.testing.assert_allclose(dk_sum, dk[0, 0, keys], atol=1e-12)
    np.testing.assert_allclose(dv_sum, dv[0, 0, keys], atol=1e-12)
