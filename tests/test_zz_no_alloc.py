"""ra_fwd_static: the bf16 forward for callers that cannot allocate device memory.

Callers that must not call cudaMalloc at run time (code under an allocator or
memory pool it may not bypass, or with a device footprint fixed at load time)
cannot build a plan, because ra_plan allocates the work table and status word.
ra_fwd_static keeps those in the library's static device array instead.  These
tests call it through the C ABI and compare it with the plan-based ra_fwd.

This file is collected last on purpose, so a stop-at-first-failure run has
already run every other test before it.
"""

import ctypes

import numpy as np
import pytest

from tests.gpu_util import assert_bf16_close, to64

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")
from context_ring_attention_gb300 import workloads  # noqa: E402


def _problem(B, S, Hq, Hkv, N, layout, causal):
    return ra._Problem(B, S, Hq, Hkv, 128, N, ra.LAYOUTS[layout], int(causal), 1, 0.0)


def test_fwd_static_rejects_oversize_and_bad_dtype():
    lib = ra.load_library()
    buf = ctypes.create_string_buffer(64 + 16)
    a = (ctypes.addressof(buf) + 15) & ~15
    big = _problem(1, 1 << 22, 32, 8, 8, "zigzag", True)        # 524288 work items > 131072
    assert lib.ra_fwd_static(ctypes.byref(big), a, a, a, a, None, None) == 2
    assert "static maximum" in ra.ra_last_error()
    f32 = ra._Problem(1, 256, 2, 2, 128, 2, 0, 1, 0, 0.0)
    assert lib.ra_fwd_static(ctypes.byref(f32), a, a, a, a, None, None) == 2


@pytest.mark.gpu
def test_fwd_static_matches_fwd_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ra.load_library()
    stream = torch.cuda.current_stream()
    cases = [
        # B, S, Hq, Hkv, N, layout, causal   (second call: other shape, layout and mask;
        # third call: the first problem again)
        (1, 2048, 8, 2, 4, "zigzag", True),
        (2, 900, 4, 4, 3, "contiguous", False),
        (1, 2048, 8, 2, 4, "zigzag", True),
    ]
    bufs = []
    for n, (B, S, Hq, Hkv, N, layout, causal) in enumerate(cases):
        q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=70 + n, device="cuda", dtype="bf16")
        bufs.append(((q, k, v), torch.empty_like(q), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")))
    torch.cuda.synchronize()
    free_after = []
    for n, (B, S, Hq, Hkv, N, layout, causal) in enumerate(cases):
        (q, k, v), o, lse = bufs[n]
        prob = _problem(B, S, Hq, Hkv, N, layout, causal)
        st = lib.ra_fwd_static(ctypes.byref(prob), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, ra.ra_last_error()
        ra.ra_fwd_static_status(stream)   # no device wait gave up
        torch.cuda.synchronize()
        free_after.append(torch.cuda.mem_get_info()[0])
    # the first call on a device may load the library's device code; later calls allocate nothing
    assert free_after[1] == free_after[0] and free_after[2] == free_after[0], free_after
    for (B, S, Hq, Hkv, N, layout, causal), ((q, k, v), o, lse) in zip(cases, bufs):
        plan = ra.ra_plan(B, S, Hq, Hkv, 128, N, layout, causal, "bf16")
        o_ref, lse_ref = ra.ra_fwd(plan, q, k, v)
        ra.ra_sync_status(plan)
        # the same work list in the same order, every row folded by one CTA in a fixed
        # order: bit for bit the plan's result (and within bf16 of the oracle's, which
        # the plan-based parity tests check)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), f"static vs plan {layout}"
        assert_bf16_close(to64(o), to64(o_ref), to64(lse), to64(lse_ref), f"static vs plan {layout}")


@pytest.mark.gpu
def test_fwd_static_round_synchronised():
    # 131072 tokens: large enough for the round-synchronised schedule (cooperative
    # launch); the static path builds the same work list, so it matches ra_fwd bit for bit
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ra.load_library()
    B, S, Hq, Hkv, N, layout = 1, 131072, 4, 2, 8, "zigzag"
    q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=99, device="cuda", dtype="bf16")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    prob = _problem(B, S, Hq, Hkv, N, layout, True)
    stream = torch.cuda.current_stream()
    st = lib.ra_fwd_static(ctypes.byref(prob), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, ra.ra_last_error()
    plan = ra.ra_plan(B, S, Hq, Hkv, 128, N, layout, True, "bf16")
    o2, lse2 = ra.ra_fwd(plan, q, k, v)
    ra.ra_sync_status(plan)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
