"""Failure detection on the GPU without a fault.

Every mbarrier wait of the tensor-core kernels gives up after about one second,
records a bit in a device status word and lets its kernel return.  ra_wait_selftest
runs that wait routine against a barrier that nothing ever completes; the test
checks the bit it leaves, that it gave up after about its budget, and that the
context still runs the forward correctly afterwards.
"""

import time

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bf16_close, to64

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

STATUS_MMA = 2      # the MMA-side timeout bit of the status word


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def test_bounded_wait_runs_out_and_the_context_survives():
    torch.cuda.synchronize()
    t0 = time.monotonic()
    word = ra.ra_wait_selftest()
    waited = time.monotonic() - t0
    assert word == STATUS_MMA, f"status word {word:#x}"
    assert 0.95 <= waited < 30.0, f"the wait gave up after {waited:.2f} s"
    # the same context: a causal zigzag forward still matches the oracle
    B, S, Hq, Hkv, n = 1, 1024, 4, 2, 4
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=91, device="cuda", dtype="bf16")
    pos = oracle.layout_positions("zigzag", S, n)
    pos_t = torch.from_numpy(pos).cuda()
    ql, kl, vl = (t.index_select(2, pos_t).contiguous() for t in (q, k, v))
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, n, "zigzag", True, "bf16")
    o, lse = ra.ra_fwd(plan, ql, kl, vl)
    ra.ra_sync_status(plan)
    ow, lw = oracle.full_attention(to64(ql), to64(kl), to64(vl), causal=True, positions=pos)
    assert_bf16_close(to64(o), ow, to64(lse), lw, "forward after the wait self-test")
