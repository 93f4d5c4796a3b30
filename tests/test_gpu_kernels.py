"""GPU parity of the HBM kernels and the float32 forward, through the C ABI."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_f32_close, to64, to_layout, to_natural

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


# ----------------------------------------------------------------- layout --

@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("seq,n", [(12, 4), (1000, 4), (4096, 8), (96, 8)])
def test_layout_perm_bitexact(layout, seq, n):
    if layout == "zigzag" and seq % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    g = torch.Generator(device="cuda").manual_seed(seq + n)
    x = torch.randn((2, 3, seq, 128), generator=g, device="cuda").to(torch.bfloat16)
    lse = torch.randn((2, 3, seq), generator=g, device="cuda")
    pos = oracle.layout_positions(layout, seq, n)
    pos_t = torch.from_numpy(pos).cuda()
    y = ra.ra_layout_perm(x, layout, n)
    assert torch.equal(y, x.index_select(2, pos_t))
    back = ra.ra_layout_perm(y, layout, n, inverse=True)
    assert torch.equal(back, x)
    ly = ra.ra_layout_perm(lse, layout, n)
    assert torch.equal(ly, lse.index_select(2, pos_t))
    assert torch.equal(ra.ra_layout_perm(ly, layout, n, inverse=True), lse)
    # fp32 rows of 12 bytes (3 floats) take the 4-byte path
    z = torch.randn((5, seq, 3), generator=g, device="cuda")
    assert torch.equal(ra.ra_layout_perm(z, layout, n, seq_dim=1), z.index_select(1, pos_t))


# ------------------------------------------------------------------ merge --

@pytest.mark.parametrize("n_parts,rows,d", [(8, 1000, 128), (5, 1001, 128), (3, 77, 8), (32, 300, 128), (9, 33, 128),
                                             (1, 5, 13), (1, 64, 128), (40, 100, 128)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_merge_matches_oracle(n_parts, rows, d, out):
    g = torch.Generator(device="cuda").manual_seed(n_parts * 1000 + rows)
    o_parts = torch.randn((n_parts, rows, d), generator=g, device="cuda")
    lse_parts = torch.randn((n_parts, rows), generator=g, device="cuda") * 5
    drop = torch.rand((n_parts, rows), generator=g, device="cuda") < 0.3
    lse_parts[drop] = -float("inf")
    lse_parts[:, 0] = -float("inf")                      # a row with no mass at all
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    o, lse = ra.ra_merge_partials(o_parts, lse_parts, out_dtype=dt)
    torch.cuda.synchronize()
    ow, lw = oracle.merge_partials(to64(o_parts), to64(lse_parts))
    assert_f32_close(to64(lse), lw, "merge LSE", atol=1e-5 * max(1.0, np.abs(lw[np.isfinite(lw)]).max()))
    if out == "f32":
        assert_f32_close(to64(o), ow, "merge O", atol=2e-6 * max(1.0, float(np.abs(ow).max())) * 4)
    else:
        err = np.abs(to64(o) - ow).max()
        assert err <= np.abs(ow).max() * 2 ** -8 + 1e-6
    assert np.all(to64(o)[0] == 0)


# ------------------------------------------------------------- f32 forward --

def _f32_case(q, k, v, n, layout, causal, scale=0.0):
    B, Hq, S, d = q.shape
    plan = ra.ra_plan(B, S, Hq, k.shape[1], d, n, layout, causal, "f32", scale)
    pos = oracle.layout_positions(layout, S, n)
    pos_t = torch.from_numpy(pos).cuda()
    ql, kl, vl = (to_layout(t, pos_t) for t in (q, k, v))
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=causal, scale=scale or None)
    assert_f32_close(to64(to_natural(o, pos_t)), ow, f"O {layout} causal={causal}")
    assert_f32_close(to64(to_natural(lse, pos_t)), lw, f"LSE {layout} causal={causal}")
    return plan, (ql, kl, vl), pos


def test_toy_ring_f32():
    wl = workloads.WORKLOADS["toy_ring_4x3_d8"]
    q, k, v = workloads.torch_inputs(wl, "cuda")
    plan = ra.ra_plan(1, 12, 1, 1, 8, 4, "contiguous", False, "f32")
    o, lse = ra.ra_fwd(plan, q, k, v)
    ra.ra_sync_status(plan)
    Q, K, V = workloads.toy_inputs()
    ring, ring_lse = oracle.ring_sim(Q[None, None], K[None, None], V[None, None], 4)
    assert_f32_close(to64(o), ring, "toy O")
    assert_f32_close(to64(lse), ring_lse, "toy LSE")


@pytest.mark.parametrize("causal", [False, True])
def test_module23_example_f32(causal):
    torch.manual_seed(0)
    q, k, v = (torch.randn(2, 4, 96, 32) for _ in range(3))
    _f32_case(q.cuda(), k.cuda(), v.cuda(), 8, "contiguous", causal)


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_f32_layouts_gqa_partials(layout, causal):
    q, k, v = workloads.small_inputs(2, 120, 6, 2, 40, seed=11, device="cuda", dtype="f32")
    n = 3
    plan, (ql, kl, vl), pos = _f32_case(q, k, v, n, layout, causal, scale=0.2)
    op, lp = ra.ra_fwd(plan, ql, kl, vl, partials=True)
    ra.ra_sync_status(plan)
    owp, lwp = oracle.ring_partials(to64(ql), to64(kl), to64(vl), n, positions=pos, causal=causal, scale=0.2)
    assert_f32_close(to64(op), owp, "partials O")
    assert_f32_close(to64(lp), lwp, "partials LSE")
    om, lm = ra.ra_merge_partials(op, lp)
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    torch.cuda.synchronize()
    assert_f32_close(to64(om), to64(o), "merge vs fused O")
    assert_f32_close(to64(lm), to64(lse), "merge vs fused LSE")


@pytest.mark.parametrize("d", [13, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_head_dim_edges(d, causal):
    # the SIMT fp32 path at its largest head dimension and at one that is not a
    # multiple of 4 (the lanes' column loops end mid-warp), striped with GQA
    q, k, v = workloads.small_inputs(1, 96, 4, 2, d, seed=13 + d, device="cuda", dtype="f32")
    _f32_case(q, k, v, 4, "striped", causal)
