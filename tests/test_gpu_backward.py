"""GPU parity of the backward pass (ra_bwd) against the float64 oracle.

The oracle differentiates the forward's definition (pinned by finite differences
in the oracle's own tests).  Both sides read the same bf16 (or f32) inputs; the
kernels use the forward's own O and LSE, as a training step would.

Tolerance for bf16 gradients, from the arithmetic.  P and dS enter the tensor-core
products rounded to bf16 (relative error up to 2^-9 each), and the outputs are
rounded to bf16 once more; everything else accumulates in fp32.  Elementwise
relative errors then stay near 2^-9, but the gradients are sums with heavy
cancellation (each row of dS sums to zero).  So the error is measured against
the size of the whole tensor: relative RMS <= 1e-2 (about 5x the 2^-9 rounding
of three bf16 factors), and max-abs <= 2e-2 times the tensor's largest
magnitude.  float32 problems: max-abs 1e-4 times the largest magnitude, since
the sums run over up to a few hundred fp32 terms.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import to64

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

BWD_REL_RMS = 1e-2
BWD_MAX_REL = 2e-2
F32_MAX_REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def _close(got, want, what, rel_rms=BWD_REL_RMS, max_rel=BWD_MAX_REL):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite"
    scale = np.abs(want).max()
    err = np.abs(got - want).max()
    rr = np.sqrt(np.mean((got - want) ** 2)) / max(np.sqrt(np.mean(want ** 2)), 1e-30)
    assert err <= max_rel * scale, f"{what}: max-abs {err:.3e} > {max_rel} x {scale:.3e}"
    assert rr <= rel_rms, f"{what}: rel-RMS {rr:.3e} > {rel_rms}"
    return err / scale, rr


def _run(B, S, Hq, Hkv, n, layout, causal, seed, dtype="bf16", d=128, q_scale=1.0):
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, d, seed=seed, device="cuda", dtype=dtype, q_scale=q_scale)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1000)
    do = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    pos = oracle.layout_positions(layout, S, n)
    pos_t = torch.from_numpy(pos).cuda()
    ql, kl, vl, dol = (t.index_select(2, pos_t).contiguous() for t in (q, k, v, do))
    plan = ra.ra_plan(B, S, Hq, Hkv, d, n, layout, causal, dtype)
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    dq, dk, dv = ra.ra_bwd(plan, ql, kl, vl, o, lse, dol)
    ra.ra_sync_status(plan)
    want = oracle.attention_backward(to64(ql), to64(kl), to64(vl), to64(dol), causal=causal, positions=pos)
    return (dq, dk, dv), want


SHAPES = [
    # B, S, Hq, Hkv, N
    (1, 1024, 4, 2, 2),    # 512 rows per shard
    (1, 900, 4, 2, 3),     # 300 rows per shard: ragged 64- and 128-row tiles
    (2, 640, 2, 2, 4),     # G = 1
    (1, 768, 6, 2, 2),     # G = 3
    (1, 256, 8, 1, 1),     # N = 1, G = 8
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_backward_matches_oracle(shape, layout, causal):
    B, S, Hq, Hkv, n = shape
    if layout == "zigzag" and S % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    got, want = _run(B, S, Hq, Hkv, n, layout, causal, seed=sum(shape) + 5)
    for name, g_, w_ in zip(("dQ", "dK", "dV"), got, want):
        _close(to64(g_), w_, f"{name} {layout} causal={causal} {shape}")


def test_bf16_backward_short_shards_and_large_logits():
    # 40 rows per shard (every tile ragged); Q x4 (peaked probabilities)
    for args in ((1, 320, 2, 1, 8, "zigzag", True, 41, 1.0), (1, 1024, 4, 2, 4, "contiguous", True, 42, 4.0)):
        B, S, Hq, Hkv, n, layout, causal, seed, qs = args
        got, want = _run(B, S, Hq, Hkv, n, layout, causal, seed=seed, q_scale=qs)
        for name, g_, w_ in zip(("dQ", "dK", "dV"), got, want):
            _close(to64(g_), w_, f"{name} {args}")


def test_bf16_backward_deterministic():
    got1, _ = _run(1, 2048, 8, 2, 4, "zigzag", True, seed=51)
    got2, _ = _run(1, 2048, 8, 2, 4, "zigzag", True, seed=51)
    for a, b in zip(got1, got2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_f32_backward_matches_oracle(causal, layout):
    # Module 23's example shape: (2, 4, 96, 32) in float32, 4 devices
    got, want = _run(2, 96, 4, 4, 4, layout, causal, seed=61, dtype="f32", d=32)
    for name, g_, w_ in zip(("dQ", "dK", "dV"), got, want):
        _close(to64(g_), w_, f"f32 {name}", rel_rms=1e-5, max_rel=F32_MAX_REL)


def test_bf16_backward_32k_one_group():
    """Full size: the 32k causal zigzag workload (32 query heads, 8 key/value heads);
    the oracle recomputes one whole group -- key/value head 0 and query heads 0-3 --
    so all 32768 rows of dK and dV and four heads of dQ are compared element by element."""
    wl = workloads.WORKLOADS["causal_32k_n8"]
    q, k, v = workloads.torch_inputs(wl, "cuda")
    layout, n = "zigzag", wl.n_shards
    ql, kl, vl = (ra.ra_layout_perm(t, layout, n) for t in (q, k, v))
    del q, k, v
    g = torch.Generator(device="cuda")
    g.manual_seed(3232)
    dol = torch.randn(ql.shape, generator=g, device="cuda").to(torch.bfloat16)
    plan = ra.ra_plan(wl.batch, wl.seq, wl.heads_q, wl.heads_kv, wl.head_dim, n, layout, True, "bf16")
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    dq, dk, dv = ra.ra_bwd(plan, ql, kl, vl, o, lse, dol)
    ra.ra_sync_status(plan)
    G = wl.heads_q // wl.heads_kv
    pos = oracle.layout_positions(layout, wl.seq, n)
    want = oracle.attention_backward(to64(ql[:, :G]), to64(kl[:, :1]), to64(vl[:, :1]), to64(dol[:, :G]),
                                     causal=True, positions=pos, block=2048)
    for name, g_, w_ in zip(("dQ", "dK", "dV"), (dq[:, :G], dk[:, :1], dv[:, :1]), want):
        err, rr = _close(to64(g_), w_, f"32k {name}")
        print(f"32k {name}: max-abs {err:.2e} of max, rel-RMS {rr:.2e}")


def test_bf16_backward_zigzag_1m_sampled():
    """Full size, the way the benchmark runs it: the 1M-token causal zigzag workload,
    ra_fwd then ra_bwd over the whole problem with the plan's own schedule.  What the
    oracle can afford there:
      * dQ of sampled query rows (a row's dQ needs only its own row of P), for the
        query heads of key/value heads 0 and Hkv-1;
      * dK and dV of the last 32 key positions of those two key/value heads: only
        the last 32 query positions see them, so the oracle sums the parts of those
        rows of the group's four query heads exactly (and checks their dQ too);
      * for every key/value head, the rows of dV add up to the sum of the dO rows of
        its query heads, because each row of P sums to one."""
    wl = workloads.WORKLOADS["zigzag_1m_n8"]
    layout, n, S = "zigzag", wl.n_shards, wl.seq
    G = wl.heads_q // wl.heads_kv
    q, k, v = workloads.torch_inputs(wl, "cuda")
    ql, kl, vl = (ra.ra_layout_perm(t, layout, n) for t in (q, k, v))
    del q, k, v
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)
    dol = torch.randn(ql.shape, generator=g, device="cuda").to(torch.bfloat16)
    plan = ra.ra_plan(wl.batch, S, wl.heads_q, wl.heads_kv, wl.head_dim, n, layout, True, "bf16")
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    dq, dk, dv = ra.ra_bwd(plan, ql, kl, vl, o, lse, dol)
    ra.ra_sync_status(plan)
    del o, lse

    pos = oracle.layout_positions(layout, S, n)
    row_of = np.empty(S, np.int64)
    row_of[pos] = np.arange(S)                       # natural position -> layout row
    nat = torch.from_numpy(row_of).cuda()

    def rows(t, h, xs):                              # rows of head h at natural positions xs
        return to64(t[0, h].index_select(0, torch.from_numpy(row_of[xs]).cuda()))

    picks = np.asarray(workloads.sample_rows(wl, 256), np.int64)
    tail = np.arange(S - 32, S)
    got_dq, want_dq, got_kv, want_kv = [], [], [], []
    for gk in (0, wl.heads_kv - 1):
        kh = to64(kl[0, gk].index_select(0, nat))    # the group's keys and values, natural order
        vh = to64(vl[0, gk].index_select(0, nat))
        dk_tail, dv_tail = np.zeros((32, wl.head_dim)), np.zeros((32, wl.head_dim))
        for h in range(gk * G, (gk + 1) * G):
            dq_t, dk_p, dv_p = oracle.attention_backward_rows(rows(ql, h, tail), rows(dol, h, tail), tail, kh, vh,
                                                              causal=True, key_idx=tail)
            dk_tail += dk_p
            dv_tail += dv_p
            got_dq.append(rows(dq, h, tail))
            want_dq.append(dq_t)
            xs = picks[picks[:, 1] == h, 2]
            for r0 in range(0, len(xs), 16):
                blk = xs[r0:r0 + 16]
                want_dq.append(oracle.attention_backward_rows(rows(ql, h, blk), rows(dol, h, blk), blk, kh, vh,
                                                              causal=True))
                got_dq.append(rows(dq, h, blk))
        got_kv.append((rows(dk, gk, tail), rows(dv, gk, tail)))
        want_kv.append((dk_tail, dv_tail))
        del kh, vh
    err, rr = _close(np.concatenate(got_dq), np.concatenate(want_dq), "1M sampled dQ")
    print(f"1M dQ: {sum(len(x) for x in got_dq)} rows, max-abs {err:.2e} of max, rel-RMS {rr:.2e}")
    for name, i in (("dK", 0), ("dV", 1)):
        err, rr = _close(np.concatenate([x[i] for x in got_kv]), np.concatenate([x[i] for x in want_kv]),
                         f"1M last-32 {name}")
        print(f"1M last 32 keys {name}: max-abs {err:.2e} of max, rel-RMS {rr:.2e}")

    # sum over keys of dV = sum over the group's query rows of dO (rows of P sum to one);
    # rounding P to bf16 moves each row sum by about 2^-9, far inside 1e-2 of the total
    for gk in range(wl.heads_kv):
        got = dv[0, gk].float().cpu().numpy().sum(axis=0, dtype=np.float64)
        want = sum(dol[0, h].float().cpu().numpy().sum(axis=0, dtype=np.float64) for h in range(gk * G, (gk + 1) * G))
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert rel <= 1e-2, f"kv head {gk}: sum of dV rows off by {rel:.3e} of the dO sum"


@pytest.mark.parametrize("s_n", [1, 2, 3])
@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_bf16_backward_shards_of_a_few_rows(s_n, layout):
    # N = 16 shards of 1-3 rows, causal: every streamed 64-row tile is a ragged tail
    if layout == "zigzag" and s_n % 2:
        pytest.skip("zigzag needs 2N | S")
    got, want = _run(1, 16 * s_n, 4, 2, 16, layout, True, seed=80 + s_n)
    for name, g_, w_ in zip(("dQ", "dK", "dV"), got, want):
        _close(to64(g_), w_, f"{name} s_n={s_n} {layout}")


@pytest.mark.parametrize("d", [13, 128])
def test_f32_backward_head_dim_edges(d):
    got, want = _run(1, 96, 4, 2, 4, "striped", True, seed=90 + d, dtype="f32", d=d)
    for name, g_, w_ in zip(("dQ", "dK", "dV"), got, want):
        _close(to64(g_), w_, f"f32 d={d} {name}", rel_rms=1e-5, max_rel=F32_MAX_REL)
