"""Merging partial attention results (oracle; test infrastructure only).

Module 23 ("The Math: One Block at a Time") states that the online-softmax fold
is order independent, so partial results over disjoint key sets can be combined
after the fact.  Written on (O_t, LSE_t) pairs this is the plain identity

    LSE = ln sum_t e^(LSE_t),     O = sum_t e^(LSE_t - LSE) O_t,

(the same max/sum algebra 3.6's vocabulary-parallel cross entropy applies across
ranks).  Parts with LSE_t = -inf carry no mass and are ignored; if every part is
-inf the row is O = 0, LSE = -inf.
"""

import numpy as np


def merge_partials(o_parts, lse_parts):
    """o_parts: [n, ..., d]; lse_parts: [n, ...].  Returns (O [..., d], LSE [...])."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    top = lse_parts.max(axis=0)
    live = np.isfinite(top)
    ref = np.where(live, top, 0.0)
    w = np.exp(lse_parts - ref[None])                 # 0 for -inf parts
    z = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(live, ref + np.log(z), -np.inf)
        frac = np.where(live[None], w / z[None], 0.0)
    out = (frac[..., None] * o_parts).sum(axis=0)
    return out, lse
