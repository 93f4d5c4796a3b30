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
