"""GPU parity of the explicit ring driver: per-step launches, the K/V exchange, the merge.

The exchange (``ra_ring_rotate``) must move bytes exactly as the oracle's
``pass_blocks`` does.  A step (``ra_fwd_step``) over the blocks the shards hold
must reproduce the oracle's per-step partial.  It must also reproduce, bit for
bit, entry t of ``ra_fwd``'s partials, which are computed with K/V read in place.
The driver (``ra_ring_fwd``) must reproduce the oracle's attention, with the
rotation on its own stream or on the compute stream.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bf16_close, assert_f32_close, to64

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def _bits(t):
    """The tensor's bytes as an integer numpy array (bf16 -> int16, f32 -> int32)."""
    it = torch.int16 if t.dtype == torch.bfloat16 else torch.int32
    return t.contiguous().view(it).cpu().numpy()


def _from_bits(a, like):
    return torch.from_numpy(np.ascontiguousarray(a)).to(like.device).view(like.dtype)


def _inputs(B, S, Hq, Hkv, n, layout, seed, dtype="bf16", d=128):
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, d, seed=seed, device="cuda", dtype=dtype)
    pos = oracle.layout_positions(layout, S, n)
    pos_t = torch.from_numpy(pos).cuda()
    return tuple(t.index_select(2, pos_t).contiguous() for t in (q, k, v)), pos


ROTATE_CASES = [
    # B, S, Hq, Hkv, N, dtype, d
    (2, 1024, 4, 2, 4, "bf16", 128),
    (1, 900, 4, 2, 3, "bf16", 128),   # shards of 300 rows
    (1, 256, 2, 1, 1, "bf16", 128),   # N = 1: the exchange is a copy
    (1, 96, 1, 1, 8, "f32", 32),
]


@pytest.mark.parametrize("case", ROTATE_CASES)
def test_rotate_bit_exact(case):
    B, S, Hq, Hkv, n, dt, d = case
    (_, k, v), _ = _inputs(B, S, Hq, Hkv, n, "contiguous", seed=11, dtype=dt, d=d)
    plan = ra.ra_plan(B, S, Hq, Hkv, d, n, "contiguous", False, dt)
    kd, vd = ra.ra_ring_rotate(plan, k, v)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kd), oracle.pass_blocks(_bits(k), n))
    assert np.array_equal(_bits(vd), oracle.pass_blocks(_bits(v), n))
    # N exchanges bring every block home
    for _ in range(n - 1):
        kd, vd = ra.ra_ring_rotate(plan, kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd, k) and torch.equal(vd, v)


STEP_CASES = [
    # B, S, Hq, Hkv, N, layout, causal
    (1, 2048, 8, 2, 4, "zigzag", True),
    (1, 900, 4, 2, 3, "contiguous", True),     # ragged shards
    (1, 768, 6, 2, 2, "striped", True),        # G = 3: row tiles paired
    (2, 640, 2, 2, 4, "striped", False),       # G = 1
]


@pytest.mark.parametrize("case", STEP_CASES)
def test_step_equals_partials_and_oracle(case):
    B, S, Hq, Hkv, n, layout, causal = case
    (q, k, v), pos = _inputs(B, S, Hq, Hkv, n, layout, seed=sum(case[:5]))
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, layout, causal, "bf16")
    op_all, lp_all = ra.ra_fwd(plan, q, k, v, partials=True)
    ra.ra_sync_status(plan)
    owp, lwp = oracle.ring_partials(to64(q), to64(k), to64(v), n, positions=pos, causal=causal)
    kb, vb = _bits(k), _bits(v)
    for t in range(n):
        # the blocks the shards hold at step t, built by the oracle's exchange
        kt = _from_bits(oracle.held_blocks(kb, n, t), k)
        vt = _from_bits(oracle.held_blocks(vb, n, t), v)
        o_t, l_t = ra.ra_fwd_step(plan, t, q, kt, vt)
        ra.ra_sync_status(plan)
        assert torch.equal(o_t, op_all[t]), f"step {t}: O differs from ra_fwd partial"
        assert torch.equal(l_t, lp_all[t]), f"step {t}: LSE differs from ra_fwd partial"
        live = np.isfinite(lwp[t])
        assert np.array_equal(np.isneginf(to64(l_t)), ~live), f"step {t}: skipped rows differ"
        if live.any():
            assert_bf16_close(to64(o_t)[live], owp[t][live], to64(l_t)[live], lwp[t][live], f"step {t}")
        assert np.all(to64(o_t)[~live] == 0)


def test_any_ring_order_gives_the_same_answer():
    """Module 23 ("The Math: One Block at a Time"): the fold does not depend on the order
    in which the blocks arrive.  The shards visit their blocks in a shuffled step order,
    one ra_fwd_step per step; merging the partials in that order gives the attention of
    the oracle, and the in-order merge to within one bf16 rounding."""
    B, S, Hq, Hkv, n, layout = 1, 2048, 8, 2, 4, "zigzag"
    (q, k, v), pos = _inputs(B, S, Hq, Hkv, n, layout, seed=77)
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, layout, True, "bf16")
    kb, vb = _bits(k), _bits(v)
    parts = {}
    for t in (2, 0, 3, 1):
        kt = _from_bits(oracle.held_blocks(kb, n, t), k)
        vt = _from_bits(oracle.held_blocks(vb, n, t), v)
        parts[t] = ra.ra_fwd_step(plan, t, q, kt, vt)
    ra.ra_sync_status(plan)
    shuffled = [2, 0, 3, 1]
    o_s, l_s = ra.ra_merge_partials(torch.stack([parts[t][0] for t in shuffled]).contiguous(),
                                    torch.stack([parts[t][1] for t in shuffled]).contiguous(),
                                    out_dtype=torch.bfloat16)
    o_i, l_i = ra.ra_merge_partials(torch.stack([parts[t][0] for t in range(n)]).contiguous(),
                                    torch.stack([parts[t][1] for t in range(n)]).contiguous(),
                                    out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=True, positions=pos)
    assert_bf16_close(to64(o_s), ow, to64(l_s), lw, "shuffled ring order")
    assert_bf16_close(to64(o_i), ow, to64(l_i), lw, "in-order ring")
    # the two merges differ only in the order of fp32 additions (a few fp32 ulps of terms
    # below 8 in magnitude), then each rounds to bf16 (half a step, 2^-8 relative)
    a, b = to64(o_s), to64(o_i)
    assert np.all(np.abs(a - b) <= 2.0 ** -7 * 1.01 * np.maximum(np.abs(a), np.abs(b)) + 4e-6)
    assert np.abs(to64(l_s) - to64(l_i)).max() <= 1e-5


def test_step_toy_ring_f32():
    # the Q&A page's toy ring: 4 devices x 3 tokens, d = 8, one step at a time
    wl = workloads.WORKLOADS["toy_ring_4x3_d8"]
    q, k, v = workloads.torch_inputs(wl, "cuda")
    plan = ra.ra_plan(1, 12, 1, 1, 8, 4, "contiguous", False, "f32")
    Q, K, V = workloads.toy_inputs()
    owp, lwp = oracle.ring_partials(Q[None, None], K[None, None], V[None, None], 4)
    kt, vt = k, v
    for t in range(4):
        o_t, l_t = ra.ra_fwd_step(plan, t, q, kt, vt)
        kt, vt = ra.ra_ring_rotate(plan, kt, vt)
        ra.ra_sync_status(plan)
        assert_f32_close(to64(o_t), owp[t], f"toy step {t} O")
        assert_f32_close(to64(l_t), lwp[t], f"toy step {t} LSE")


DRIVER_CASES = [
    # B, S, Hq, Hkv, N, layout, causal
    (1, 2048, 8, 2, 4, "zigzag", True),
    (1, 2048, 4, 4, 8, "contiguous", True),
    (1, 1536, 4, 2, 3, "striped", False),
    (1, 512, 4, 1, 1, "contiguous", True),     # N = 1: one step, no exchange
]


@pytest.mark.parametrize("case", DRIVER_CASES)
def test_ring_driver_matches_oracle(case):
    B, S, Hq, Hkv, n, layout, causal = case
    (q, k, v), pos = _inputs(B, S, Hq, Hkv, n, layout, seed=7 + n)
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, layout, causal, "bf16")
    o_parts = torch.empty((n, B, Hq, S, 128), dtype=torch.float32, device="cuda")
    lse_parts = torch.empty((n, B, Hq, S), dtype=torch.float32, device="cuda")
    o, lse = ra.ra_ring_fwd(plan, q, k, v, o_parts=o_parts, lse_parts=lse_parts)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(q), to64(k), to64(v), causal=causal, positions=pos)
    assert_bf16_close(to64(o), ow, to64(lse), lw, f"ring driver {case}")
    # the driver's partials are ra_fwd's partials, bit for bit
    op_all, lp_all = ra.ra_fwd(plan, q, k, v, partials=True)
    ra.ra_sync_status(plan)
    assert torch.equal(o_parts, op_all) and torch.equal(lse_parts, lp_all)
    # K and V are left untouched
    (q2, k2, v2), _ = _inputs(B, S, Hq, Hkv, n, layout, seed=7 + n)
    assert torch.equal(k, k2) and torch.equal(v, v2)


def test_ring_driver_same_stream_and_repeat():
    # rotation on the compute stream (no overlap) and on its own stream agree bit
    # for bit; a second call reusing the same scratch gives the same result
    (q, k, v), _ = _inputs(1, 2048, 8, 2, 4, "zigzag", seed=77)
    plan = ra.ra_plan(1, 2048, 8, 2, 128, 4, "zigzag", True, "bf16")
    kb = torch.empty((2,) + tuple(k.shape), dtype=k.dtype, device="cuda")
    vb = torch.empty_like(kb)
    cur = torch.cuda.current_stream()
    o1, l1 = ra.ra_ring_fwd(plan, q, k, v, k_buf=kb, v_buf=vb, comm_stream=cur)
    side = torch.cuda.Stream()
    o2, l2 = ra.ra_ring_fwd(plan, q, k, v, k_buf=kb, v_buf=vb, comm_stream=side)
    o3, l3 = ra.ra_ring_fwd(plan, q, k, v, k_buf=kb, v_buf=vb, comm_stream=side)
    ra.ra_sync_status(plan)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o2, o3) and torch.equal(l2, l3)


def test_ring_driver_f32_toy():
    wl = workloads.WORKLOADS["toy_ring_4x3_d8"]
    q, k, v = workloads.torch_inputs(wl, "cuda")
    plan = ra.ra_plan(1, 12, 1, 1, 8, 4, "contiguous", False, "f32")
    o, lse = ra.ra_ring_fwd(plan, q, k, v)
    ra.ra_sync_status(plan)
    Q, K, V = workloads.toy_inputs()
    ring, ring_lse = oracle.ring_sim(Q[None, None], K[None, None], V[None, None], 4)
    assert_f32_close(to64(o), ring, "toy O")
    assert_f32_close(to64(lse), ring_lse, "toy LSE")


def test_round_synchronised_paths_match_fused():
    # 131072 tokens take the round-synchronised schedule (cooperative launches) in the
    # per-step, gathered and backward kernels too; each must agree with the fused
    # ra_fwd (itself checked against the oracle at this size): the per-step partials
    # bit for bit with ra_fwd's, the driver and the gathered forward within bf16
    # rounding of the merge / visiting order.
    B, S, Hq, Hkv, n, layout = 1, 131072, 4, 2, 8, "zigzag"
    (q, k, v), _ = _inputs(B, S, Hq, Hkv, n, layout, seed=131)
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, layout, True, "bf16")
    o, lse = ra.ra_fwd(plan, q, k, v)
    op, lp = ra.ra_fwd(plan, q, k, v, partials=True)
    o_parts = torch.empty_like(op)
    lse_parts = torch.empty_like(lp)
    o_r, lse_r = ra.ra_ring_fwd(plan, q, k, v, o_parts=o_parts, lse_parts=lse_parts)
    k_all, v_all = ra.ra_allgather_kv(plan, k, v)
    o_g, lse_g = ra.ra_fwd_gathered(plan, q, k_all, v_all)
    ra.ra_sync_status(plan)
    assert torch.equal(o_parts, op) and torch.equal(lse_parts, lp)
    for what, (o_x, l_x) in (("ring driver", (o_r, lse_r)), ("gathered", (o_g, lse_g))):
        assert_bf16_close(to64(o_x), to64(o), to64(l_x), to64(lse), f"{what} vs fused at 131k")
