"""GPU parity of the bf16 tensor-core forward on shapes the oracle computes in full.

Shapes span several 128-row tiles with ragged tails (shards not a multiple of
128), every layout, causal and not, GQA groups of even size (query heads paired
per CTA), odd size and 1 (row tiles paired per CTA), and the per-step partials.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bf16_close, assert_f32_close, to64, to_layout, to_natural

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def _run(B, S, Hq, Hkv, n, layout, causal, seed, q_scale=1.0, scale=0.0):
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=seed, device="cuda", dtype="bf16",
                                     q_scale=q_scale)
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, layout, causal, "bf16", scale)
    pos = oracle.layout_positions(layout, S, n)
    pos_t = torch.from_numpy(pos).cuda()
    ql, kl, vl = (to_layout(t, pos_t) for t in (q, k, v))
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=causal, scale=scale or None)
    assert_bf16_close(to64(to_natural(o, pos_t)), ow, to64(to_natural(lse, pos_t)), lw,
                      f"{layout} causal={causal} S={S} N={n} Hq={Hq} Hkv={Hkv}")
    return plan, (ql, kl, vl), (o, lse), pos


SHAPES = [
    # B, S, Hq, Hkv, N     (S/N rows per shard)
    (1, 1024, 4, 2, 2),    # 512 per shard: 4 full tiles
    (1, 900, 4, 2, 3),     # 300 per shard: 2 tiles + 44-row tail
    (2, 640, 2, 2, 4),     # G = 1: row tiles paired, 160 per shard (1 tile + 32 tail)
    (1, 768, 6, 2, 2),     # G = 3 (odd): row tiles paired, 384 per shard (3 tiles: one single)
    (1, 256, 8, 1, 1),     # N = 1: plain attention, G = 8
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_fused_matches_oracle(shape, layout, causal):
    B, S, Hq, Hkv, n = shape
    if layout == "zigzag" and S % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    _run(B, S, Hq, Hkv, n, layout, causal, seed=sum(shape))


def test_bf16_short_shards():
    # 40 rows per shard: every tile is a ragged tail
    _run(1, 320, 2, 1, 8, "zigzag", True, seed=5)
    _run(1, 320, 2, 2, 8, "striped", False, seed=6)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_large_logits(causal):
    # Q x4: the running max moves by many units between tiles (lazy rescale path)
    _run(1, 1024, 4, 4, 4, "contiguous", causal, seed=9, q_scale=4.0)
    _run(1, 1024, 4, 2, 4, "zigzag", causal, seed=10, q_scale=4.0, scale=0.3)


@pytest.mark.parametrize("n", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_dominant_key_in_last_columns(n, causal):
    # One key (position 124, column 124 of its 128-key tile) scores about 260 log2
    # units above every other key for the queries at positions 120..127.  The row max
    # must include the tile's last columns: a reference that missed that key would put
    # 2^260 into float32 and turn those rows into inf / NaN.  Rows 124..126 see the key
    # through a causal diagonal tile (limit 125..127), rows 127 and up through a full one.
    B, S, H, d = 1, 256, 1, 128
    q, k, v = workloads.small_inputs(B, S, H, H, d, seed=31, device="cuda", dtype="bf16")
    q[0, 0, 120:128] = 0
    q[0, 0, 120:128, 0] = 16.0
    k[0, 0, 124] = 0
    k[0, 0, 124, 0] = 128.0
    plan = ra.ra_plan(B, S, H, H, d, n, "contiguous", causal, "bf16")
    o, lse = ra.ra_fwd(plan, q, k, v)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=causal)
    assert np.isfinite(to64(o)).all() and np.isfinite(to64(lse)).all()
    # where the key is visible its weight is 1: the row is V's row 124, the LSE its score
    seen = slice(124, 128) if causal else slice(120, 128)
    assert np.array_equal(to64(o)[0, 0, seen], np.broadcast_to(to64(v)[0, 0, 124], to64(o)[0, 0, seen].shape))
    assert_bf16_close(to64(o), ow, to64(lse), lw, f"dominant key causal={causal} N={n}")


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_partials_and_merge(layout, causal):
    B, S, Hq, Hkv, n = 1, 768, 4, 2, 3
    plan, (ql, kl, vl), (o, lse), pos = _run(B, S, Hq, Hkv, n, layout, causal, seed=21)
    op, lp = ra.ra_fwd(plan, ql, kl, vl, partials=True)
    ra.ra_sync_status(plan)
    owp, lwp = oracle.ring_partials(to64(ql), to64(kl), to64(vl), n, positions=pos, causal=causal)
    for t in range(n):
        live = np.isfinite(lwp[t])
        assert np.array_equal(np.isneginf(to64(lp[t])), ~live), f"step {t}: skipped rows differ"
        if live.any():
            assert_bf16_close(to64(op[t])[live], owp[t][live], to64(lp[t])[live], lwp[t][live], f"step {t}")
        assert np.all(to64(op[t])[~live] == 0)
    om, lm = ra.ra_merge_partials(op, lp, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ow, lw = oracle.full_attention(to64(ql), to64(kl), to64(vl), causal=causal, positions=pos)
    assert_bf16_close(to64(om), ow, to64(lm), lw, "merged partials")


def test_bf16_deterministic():
    q, k, v = workloads.small_inputs(1, 2048, 8, 2, 128, seed=3, device="cuda", dtype="bf16")
    plan = ra.ra_plan(1, 2048, 8, 2, 128, 4, "zigzag", True, "bf16")
    o1, l1 = ra.ra_fwd(plan, q, k, v)
    o2, l2 = ra.ra_fwd(plan, q, k, v)
    ra.ra_sync_status(plan)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bf16_pipeline_through_layout_kernels():
    """Natural-order inputs -> ra_layout_perm -> ra_fwd -> inverse ra_layout_perm."""
    B, S, Hq, Hkv, n = 1, 1536, 4, 2, 4
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=33, device="cuda", dtype="bf16")
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, "zigzag", True, "bf16")
    ql, kl, vl = (ra.ra_layout_perm(t, "zigzag", n) for t in (q, k, v))
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    on = ra.ra_layout_perm(o, "zigzag", n, inverse=True)
    ln = ra.ra_layout_perm(lse, "zigzag", n, inverse=True)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=True)
    assert_bf16_close(to64(on), ow, to64(ln), lw, "pipeline")


def test_bf16_row_sums_property():
    """exp(s - LSE) summed over a row's causal keys is 1 (checked in fp64 on sampled rows)."""
    B, S, Hq, Hkv, n = 1, 2048, 2, 1, 4
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=44, device="cuda", dtype="bf16")
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, "striped", True, "bf16")
    pos = oracle.layout_positions("striped", S, n)
    pos_t = torch.from_numpy(pos).cuda()
    _, lse = ra.ra_fwd(plan, *(to_layout(t, pos_t) for t in (q, k, v)))
    ra.ra_sync_status(plan)
    lse_n = to64(to_natural(lse, pos_t))
    qn, kn = to64(q), to64(k)
    for h in range(Hq):
        for x in (0, 1, 127, 128, 1000, S - 1):
            s = kn[0, 0, : x + 1] @ qn[0, h, x] / np.sqrt(128)
            assert abs(np.exp(s - lse_n[0, h, x]).sum() - 1.0) < 5e-3


@pytest.mark.parametrize("s_n", [1, 2, 3])
@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_shards_of_a_few_rows(s_n, layout, causal):
    # N = 16 shards of 1-3 rows: every 128-row tile box spans many shards, and every
    # query and key tile is a ragged tail of a few rows
    n = 16
    if layout == "zigzag" and s_n % 2:
        pytest.skip("zigzag needs 2N | S")
    _run(1, n * s_n, 4, 2, n, layout, causal, seed=70 + s_n)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_several_dominant_keys_at_rounding_midpoints(causal):
    # Rows 64..127 see four dominant keys (positions 3, 10, 40, 60) whose weights
    # relative to the largest are about 1, 1 - 2^-9, 1 - 3*2^-9 and 1 - 5*2^-9: the
    # last three sit at or beside midpoints of bf16 rounding, where P's rounding error
    # is largest, and the row-sum correction covers only the largest key.  Their values
    # are +4, -4, +4, -4 in every column, so that O is near zero and its own bf16
    # rounding negligible; every other key is 28 natural-log units below them.  The
    # bf16 rounding of the three weights moves O by at most 3 * 2^-9 * 4 / 4 (about
    # 6e-3), inside the 2e-2 tolerance.
    B, S, H, d = 1, 128, 1, 128
    q, k, v = workloads.small_inputs(B, S, H, H, d, seed=37, device="cuda", dtype="bf16")
    scale = 1.0 / np.sqrt(d)
    q[0, 0, 64:] = 0
    q[0, 0, 64:, 0] = 8.0    # base score 8 * 40 * scale = 28.3 for the dominant keys
    q[0, 0, 64:, 1] = 64.0   # carries the small offsets ln(ratio) through k[:, 1]
    k[0, 0] = 0
    dominant = ((3, 1.0, 4.0), (10, 1 - 2.0 ** -9, -4.0), (40, 1 - 3 * 2.0 ** -9, 4.0), (60, 1 - 5 * 2.0 ** -9, -4.0))
    for pos, ratio, value in dominant:
        k[0, 0, pos, 0] = 40.0
        k[0, 0, pos, 1] = np.log(ratio) / (64.0 * scale)
        v[0, 0, pos] = value
    plan = ra.ra_plan(B, S, H, H, d, 1, "contiguous", causal, "bf16")
    o, lse = ra.ra_fwd(plan, q, k, v)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=causal)
    err = np.abs(to64(o)[0, 0, 64:] - ow[0, 0, 64:]).max()
    print(f"several dominant keys, causal={causal}: max-abs error {err:.3e} on rows 64..127")
    assert err <= 3 * 2.0 ** -9 + 5e-4
    # O is built to be near zero on those rows, so the relative-RMS part of the parity
    # bound says nothing here; the absolute parts apply to the whole tensor.
    assert np.abs(to64(o) - ow).max() <= 2e-2
    assert np.abs(to64(lse) - lw).max() <= 2e-2
