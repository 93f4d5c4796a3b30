"""GPU parity at the full sizes of the benchmark workloads, on sampled rows.

Each workload runs exactly as bench.py runs it (natural-order inputs ->
ra_layout_perm -> ra_fwd over the whole problem -> inverse ra_layout_perm), and
the float64 oracle recomputes sampled rows one by one against every key.  The
4096-token-per-shard 4k workload is also compared element by element on a few
whole heads.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bf16_close, to64
from tests.oracle_pool import attention_rows_parallel

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def _run_workload(wl, layout):
    q, k, v = workloads.torch_inputs(wl, "cuda")
    plan = ra.ra_plan(wl.batch, wl.seq, wl.heads_q, wl.heads_kv, wl.head_dim, wl.n_shards, layout,
                      wl.causal, wl.dtype)
    ql, kl, vl = (ra.ra_layout_perm(t, layout, wl.n_shards) for t in (q, k, v))
    o_l, lse_l = ra.ra_fwd(plan, ql, kl, vl)
    del ql, kl, vl
    o = ra.ra_layout_perm(o_l, layout, wl.n_shards, inverse=True)
    lse = ra.ra_layout_perm(lse_l, layout, wl.n_shards, inverse=True)
    del o_l, lse_l
    ra.ra_sync_status(plan)
    return plan, (q, k, v), (o, lse)


def _check_sampled(wl, qkv, out, picks, what):
    q, k, v = qkv
    o, lse = out
    G = wl.heads_q // wl.heads_kv
    picks = np.asarray(picks, np.int64)
    got_o = np.zeros((len(picks), wl.head_dim))
    got_l = np.zeros(len(picks))
    want_o = np.zeros_like(got_o)
    want_l = np.zeros_like(got_l)
    for b in np.unique(picks[:, 0]):
        for g in range(wl.heads_kv):
            sel = np.nonzero((picks[:, 0] == b) & (picks[:, 1] // G == g))[0]
            if sel.size == 0:
                continue
            hs = torch.from_numpy(picks[sel, 1]).cuda()
            xs = torch.from_numpy(picks[sel, 2]).cuda()
            q_rows = to64(q[int(b)][hs, xs])
            got_o[sel] = to64(o[int(b)][hs, xs])
            got_l[sel] = to64(lse[int(b)][hs, xs])
            kh = k[int(b), g].float().cpu().numpy()
            vh = v[int(b), g].float().cpu().numpy()
            want_o[sel], want_l[sel] = attention_rows_parallel(q_rows, picks[sel, 2], kh, vh, wl.causal)
    err, rr = assert_bf16_close(got_o, want_o, got_l, want_l, what)
    print(f"{what}: {len(picks)} rows, O max-abs {err:.2e}, rel-RMS {rr:.2e}")


@pytest.mark.parametrize("name", ["noncausal_4k_n8", "noncausal_4k_n8_q4"])
def test_noncausal_4k(name):
    wl = workloads.WORKLOADS[name]
    plan, (q, k, v), (o, lse) = _run_workload(wl, "contiguous")
    # two whole heads element by element
    for h in (0, wl.heads_q - 1):
        ow, lw = oracle.full_attention(to64(q[:1, h:h + 1]), to64(k[:1, h:h + 1]), to64(v[:1, h:h + 1]))
        assert_bf16_close(to64(o[:1, h:h + 1]), ow, to64(lse[:1, h:h + 1]), lw, f"{name} head {h}")
    _check_sampled(wl, (q, k, v), (o, lse), workloads.sample_rows(wl, 1024), name)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_causal_32k(layout):
    wl = workloads.WORKLOADS["causal_32k_n8"]
    plan, qkv, out = _run_workload(wl, layout)
    _check_sampled(wl, qkv, out, workloads.sample_rows(wl, 1024), f"causal_32k {layout}")
    full, part, skip = ra.ra_plan_tile_counts(plan)
    want = oracle.tile_counts(layout, wl.seq, wl.n_shards, causal=True)
    assert [full.tolist(), part.tolist(), skip.tolist()] == [x.tolist() for x in want]


def test_striped_131k():
    wl = workloads.WORKLOADS["striped_131k_n32"]
    plan, qkv, out = _run_workload(wl, "striped")
    _check_sampled(wl, qkv, out, workloads.sample_rows(wl, 1024), "striped_131k")


def test_zigzag_1m():
    wl = workloads.WORKLOADS["zigzag_1m_n8"]
    plan, qkv, out = _run_workload(wl, "zigzag")
    _check_sampled(wl, qkv, out, workloads.sample_rows(wl, 4096), "zigzag_1m")
