"""The binding refuses caller buffers of the wrong shape, dtype or layout before
anything is launched (the C ABI sees only pointers, so it cannot check sizes).

Every wrong buffer here is at least as large as the right one, so that even a
missing check could not make a kernel overrun it.
"""

import pytest

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def test_wrong_output_buffers_are_refused():
    B, S, Hq, Hkv, d, N = 1, 256, 2, 1, 128, 2
    plan = ra.ra_plan(B, S, Hq, Hkv, d, N, "contiguous", True, "bf16")
    bf, f32 = torch.bfloat16, torch.float32
    q = torch.zeros((B, Hq, S, d), dtype=bf, device="cuda")
    k = torch.zeros((B, Hkv, S, d), dtype=bf, device="cuda")
    v = torch.zeros_like(k)
    with pytest.raises(ValueError):
        ra.ra_fwd(plan, q, k, v, o=torch.empty((B, Hq, 2 * S, d), dtype=bf, device="cuda"))
    with pytest.raises(ValueError):
        ra.ra_fwd(plan, q, k, v, lse=torch.empty((B, Hq, S), dtype=torch.float64, device="cuda"))
    with pytest.raises(ValueError):
        ra.ra_fwd(plan, q, k, v, partials=True, o_parts=torch.empty((N + 1, B, Hq, S, d), dtype=f32, device="cuda"))
    with pytest.raises(ValueError):
        ra.ra_fwd_step(plan, 0, q, k, v, lse_part=torch.empty((B, Hq, S, 2), dtype=f32, device="cuda"))
    with pytest.raises(ValueError):
        ra.ra_layout_perm(q, "contiguous", N, out=torch.empty((B, Hq, 2 * S, d), dtype=bf, device="cuda"))
    with pytest.raises(ValueError):
        ra.ra_fwd_gathered(plan, q, k, v, o=torch.empty((B, Hq, S, 2 * d), dtype=bf, device="cuda"))
    o = torch.zeros_like(q)
    lse = torch.zeros((B, Hq, S), dtype=f32, device="cuda")
    with pytest.raises(ValueError):
        ra.ra_bwd(plan, q, k, v, o, lse, o, dq=torch.empty((B, Hq, 2 * S, d), dtype=bf, device="cuda"))
    with pytest.raises(ValueError):
        ra.ra_bwd(plan, q, k, v, o, lse, o,
                  scratch=torch.empty(ra.ra_bwd_scratch_size(plan), dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError):   # n_shards says 2 head shards, x holds 4
        ra.ra_ulysses_a2a(torch.zeros((4, B, 1, S, d), dtype=bf, device="cuda"), "contiguous", N, 1)
    with pytest.raises(ValueError):
        ra.ra_merge_partials(torch.zeros((N, 8, d), dtype=f32, device="cuda"),
                             torch.zeros((N, 9), dtype=f32, device="cuda"))
    torch.cuda.synchronize()


def test_c_abi_rejects_memory_of_the_host():
    # The kernels run on the current device: a host pointer (pinned or pageable)
    # is refused before anything is launched.
    import ctypes
    lib = ra.load_library()
    S, N = 256, 2
    x = torch.zeros((1, 1, S, 128), dtype=torch.bfloat16, device="cuda")
    pinned = torch.zeros((1, 1, S, 128), dtype=torch.bfloat16).pin_memory()
    pageable = ctypes.create_string_buffer(S * 256 + 16)
    host = (ctypes.addressof(pageable) + 15) & ~15
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for src in (pinned.data_ptr(), host):
        assert lib.ra_layout_perm(0, S, N, 0, 1, 256, ctypes.c_void_p(src), ctypes.c_void_p(x.data_ptr()),
                                  stream) == 1
        assert "not device memory" in ra.ra_last_error()
    plan = ra.ra_plan(1, S, 1, 1, 128, N, "contiguous", True, "bf16")
    o = torch.empty_like(x)
    assert lib.ra_fwd(plan.handle, ctypes.c_void_p(pinned.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                      ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(o.data_ptr()), None, None, None,
                      stream) == 1
    with pytest.raises(ValueError):   # the binding refuses a CPU tensor before the C call
        ra.ra_layout_perm(pinned, "contiguous", N)
    torch.cuda.synchronize()


def test_plan_destroy_does_not_wait_for_other_work():
    # Plan A's forwards keep the GPU busy on one stream.  Destroying plan B, whose work
    # has finished, must return while A's kernels still run.  Plan C's kernel is queued
    # behind A's on the same stream: destroying C right away must not wait either, and
    # must not pull C's tables from under its kernel (the frees are queued behind it).
    import time
    B, S, Hq, Hkv, N = 1, 32768, 32, 8, 8
    q = torch.randn((B, Hq, S, 128), device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Hkv, S, 128), device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    o, lse = torch.empty_like(q), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    plan_a = ra.ra_plan(B, S, Hq, Hkv, 128, N, "zigzag", True, "bf16")
    small = (1, 1024, 2, 1, 128, 2, "contiguous", True, "bf16")
    qs = torch.randn((1, 2, 1024, 128), device="cuda").to(torch.bfloat16)
    ks = torch.randn((1, 1, 1024, 128), device="cuda").to(torch.bfloat16)
    plan_b = ra.ra_plan(*small)
    want, want_lse = ra.ra_fwd(plan_b, qs, ks, ks)
    s_a = torch.cuda.Stream()
    torch.cuda.synchronize()
    done_a = torch.cuda.Event()
    for _ in range(40):                      # about 0.2 s of forward work
        ra.ra_fwd(plan_a, q, k, v, o=o, lse=lse, stream=s_a)
    done_a.record(s_a)
    t0 = time.perf_counter()
    plan_b.close()
    dt_b = time.perf_counter() - t0
    plan_c = ra.ra_plan(*small)
    oc = torch.empty_like(qs)
    lc = torch.empty((1, 2, 1024), dtype=torch.float32, device="cuda")
    ra.ra_fwd(plan_c, qs, ks, ks, o=oc, lse=lc, stream=s_a)
    t0 = time.perf_counter()
    plan_c.close()
    dt_c = time.perf_counter() - t0
    assert not done_a.query(), "plan A's work had already ended: the test proves nothing"
    assert dt_b < 0.05 and dt_c < 0.05, f"a destroy waited for the device ({dt_b:.3f} s, {dt_c:.3f} s)"
    torch.cuda.synchronize()
    ra.ra_sync_status(plan_a)
    assert torch.equal(oc, want) and torch.equal(lc, want_lse)
