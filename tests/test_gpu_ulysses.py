"""GPU parity of DeepSpeed-Ulysses' exchange (ra_ulysses_a2a) and of the forward
composed from it: exchange Q, K, V to head shards, ordinary attention per device
(one plan: batch N*B, H/N heads, one shard), exchange O and the LSE back.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bf16_close, to64

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


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("n", [2, 4])
def test_exchange_bit_exact(layout, n):
    B, H, S = 2, 8, 512 + 128 * (n == 4)
    x = torch.randn((B, H, S, 128), device="cuda").to(torch.bfloat16)
    lse = torch.randn((B, H, S), device="cuda")
    pos = oracle.layout_positions(layout, S, n)
    y = ra.ra_ulysses_a2a(x, layout, n, 0)
    yl = ra.ra_ulysses_a2a(lse, layout, n, 0)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.ulysses_seq_to_head(_bits(x), pos, n))
    assert np.array_equal(_bits(yl)[..., None], oracle.ulysses_seq_to_head(_bits(lse)[..., None], pos, n))
    back = ra.ra_ulysses_a2a(y, layout, n, 1)
    backl = ra.ra_ulysses_a2a(yl, layout, n, 1)
    torch.cuda.synchronize()
    assert torch.equal(back, x) and torch.equal(backl, lse)


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_ulysses_forward_matches_oracle(layout, causal):
    B, S, Hq, Hkv, n = 1, 1024, 8, 4, 4
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=81, device="cuda", dtype="bf16")
    pos = oracle.layout_positions(layout, S, n)
    pt = torch.from_numpy(pos).cuda()
    ql, kl, vl = (t.index_select(2, pt).contiguous() for t in (q, k, v))
    qh, kh, vh = (ra.ra_ulysses_a2a(t, layout, n, 0) for t in (ql, kl, vl))
    # every device: its H/N heads over all S tokens in natural order -- one plan for all devices
    plan = ra.ra_plan(n * B, S, Hq // n, Hkv // n, 128, 1, "contiguous", causal, "bf16")
    oh, lh = ra.ra_fwd(plan, qh.view(n * B, Hq // n, S, 128), kh.view(n * B, Hkv // n, S, 128),
                       vh.view(n * B, Hkv // n, S, 128))
    o = ra.ra_ulysses_a2a(oh.view(n, B, Hq // n, S, 128), layout, n, 1)
    lse = ra.ra_ulysses_a2a(lh.view(n, B, Hq // n, S), layout, n, 1)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(ql), to64(kl), to64(vl), causal=causal, positions=pos)
    assert_bf16_close(to64(o), ow, to64(lse), lw, f"ulysses {layout} causal={causal}")
