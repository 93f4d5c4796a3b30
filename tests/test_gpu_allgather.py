"""GPU parity of the all-gather variant (ra_allgather_kv, ra_fwd_gathered).

Every device gathers all K/V blocks (natural order) and attends its own query
shard to them in one step.  The gather must move bytes exactly as the oracle's
to_natural; the forward must reproduce the oracle's attention.
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
    it = torch.int16 if t.dtype == torch.bfloat16 else torch.int32
    return t.contiguous().view(it).cpu().numpy()


SHAPES = [
    # B, S, Hq, Hkv, N
    (1, 1024, 4, 2, 2),
    (1, 900, 4, 2, 3),     # ragged 128-row tiles
    (2, 640, 2, 2, 4),     # G = 1
    (1, 768, 6, 2, 2),     # G = 3
    (1, 256, 8, 1, 1),     # N = 1
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_gathered_forward_matches_oracle(shape, layout, causal):
    B, S, Hq, Hkv, n = shape
    if layout == "zigzag" and S % (2 * n):
        pytest.skip("zigzag needs 2N | S")
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=sum(shape) + 9, device="cuda", dtype="bf16")
    pos = oracle.layout_positions(layout, S, n)
    pt = torch.from_numpy(pos).cuda()
    ql, kl, vl = (t.index_select(2, pt).contiguous() for t in (q, k, v))
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, layout, causal, "bf16")
    k_all, v_all = ra.ra_allgather_kv(plan, kl, vl)
    o, lse = ra.ra_fwd_gathered(plan, ql, k_all, v_all)
    ra.ra_sync_status(plan)
    assert np.array_equal(_bits(k_all), oracle.to_natural(_bits(kl), pos))
    assert np.array_equal(_bits(v_all), oracle.to_natural(_bits(vl), pos))
    ow, lw = oracle.full_attention(to64(ql), to64(kl), to64(vl), causal=causal, positions=pos)
    assert_bf16_close(to64(o), ow, to64(lse), lw, f"gathered {layout} causal={causal} {shape}")


def test_gathered_forward_f32():
    # Module 23's example shape (2, 4, 96, 32), float32, 4 devices, zigzag, causal
    q, k, v = workloads.small_inputs(2, 96, 4, 4, 32, seed=71, device="cuda", dtype="f32")
    pos = oracle.layout_positions("zigzag", 96, 4)
    pt = torch.from_numpy(pos).cuda()
    ql, kl, vl = (t.index_select(2, pt).contiguous() for t in (q, k, v))
    plan = ra.ra_plan(2, 96, 4, 4, 32, 4, "zigzag", True, "f32")
    k_all, v_all = ra.ra_allgather_kv(plan, kl, vl)
    o, lse = ra.ra_fwd_gathered(plan, ql, k_all, v_all)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(ql), to64(kl), to64(vl), causal=True, positions=pos)
    assert_f32_close(to64(o), ow, "gathered f32 O")
    assert_f32_close(to64(lse), lw, "gathered f32 LSE")
