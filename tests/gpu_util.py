"""Helpers shared by the GPU parity tests (comparison metrics, layout shuffles)."""

import numpy as np

# Tolerances of the forward pass against the float64 oracle.
F32_MAX_ABS = 1e-5
BF16_MAX_ABS = 2e-2
BF16_REL_RMS = 5e-3


def to64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_rms(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.sqrt(np.mean(want ** 2))
    return float(np.sqrt(np.mean((got - want) ** 2)) / den) if den > 0 else float(np.abs(got - want).max())


def assert_bf16_close(o_got, o_want, lse_got=None, lse_want=None, what=""):
    o_got = np.asarray(o_got, np.float64)
    o_want = np.asarray(o_want, np.float64)
    assert np.isfinite(o_got).all(), f"{what}: non-finite output"
    err = np.abs(o_got - o_want).max()
    rr = rel_rms(o_got, o_want)
    assert err <= BF16_MAX_ABS, f"{what}: O max-abs {err:.3e} > {BF16_MAX_ABS}"
    assert rr <= BF16_REL_RMS, f"{what}: O rel-RMS {rr:.3e} > {BF16_REL_RMS}"
    if lse_got is not None:
        lg = np.asarray(lse_got, np.float64)
        lw = np.asarray(lse_want, np.float64)
        assert np.array_equal(np.isneginf(lg), np.isneginf(lw)), f"{what}: -inf LSE pattern differs"
        fin = np.isfinite(lw)
        e2 = np.abs(lg[fin] - lw[fin]).max() if fin.any() else 0.0
        r2 = rel_rms(lg[fin], lw[fin]) if fin.any() else 0.0
        assert e2 <= BF16_MAX_ABS, f"{what}: LSE max-abs {e2:.3e}"
        assert r2 <= BF16_REL_RMS, f"{what}: LSE rel-RMS {r2:.3e}"
    return err, rr


def assert_f32_close(got, want, what="", atol=F32_MAX_ABS):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    same_inf = np.isneginf(got) == np.isneginf(want)
    assert same_inf.all(), f"{what}: -inf pattern differs"
    fin = np.isfinite(want)
    err = np.abs(got[fin] - want[fin]).max() if fin.any() else 0.0
    assert err <= atol, f"{what}: max-abs {err:.3e} > {atol}"
    return err


def to_layout(t, pos_t, dim=2):
    """Natural order -> layout order along `dim` (pos_t: torch long tensor of positions)."""
    return t.index_select(dim, pos_t).contiguous()


def to_natural(t, pos_t, dim=2):
    out = t.new_empty(t.shape)
    out.index_copy_(dim, pos_t, t)
    return out
