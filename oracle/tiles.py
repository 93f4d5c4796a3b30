"""Causal tile classification counts (oracle; test infrastructure only).

Module 23 ("The Causal Imbalance — and the Striped Fix") counts the causal (q, k)
pairs each device computes.  At tile granularity the same question becomes: for
every pair of a query tile of device p and a key tile of the block it holds at
step t, is the tile

* SKIP    -- no (q, k) pair in it is causal (the block part lies strictly in the
             future of every query of the tile),
* FULL    -- every pair is causal (no mask needed), or
* PARTIAL -- some but not all pairs are causal (masked pair by pair)?

Non-causal attention has only FULL tiles.  Tiles are ``tile`` rows of the shard
in layout order; the last tile of a shard may be shorter.  ``tile_counts`` uses
"no pair allowed  <=>  min key position > max query position" and "all pairs
allowed  <=>  max key position <= min query position", which is the definition
restated (not a property of any layout); ``tile_classes_bruteforce`` checks every
pair and pins it.
"""

import numpy as np

from .layouts import layout_positions

FULL, PARTIAL, SKIP = 0, 1, 2


def _tile_bounds(p_slice, tile):
    n = p_slice.shape[0]
    mins, maxs = [], []
    for i0 in range(0, n, tile):
        blk = p_slice[i0:i0 + tile]
        mins.append(blk.min())
        maxs.append(blk.max())
    return np.array(mins, np.int64), np.array(maxs, np.int64)


def tile_counts(layout, seq, n_shards, causal=True, tile=128):
    """Per-shard counts of FULL, PARTIAL and SKIP tiles over all N ring steps.

    Returns three int64 arrays of length N (one query head, one batch entry).
    """
    pos = layout_positions(layout, seq, n_shards)
    s_n = seq // n_shards
    full = np.zeros(n_shards, np.int64)
    part = np.zeros(n_shards, np.int64)
    skip = np.zeros(n_shards, np.int64)
    bounds = [_tile_bounds(pos[p * s_n:(p + 1) * s_n], tile) for p in range(n_shards)]
    for p in range(n_shards):
        qmin, qmax = bounds[p]
        for t in range(n_shards):
            r = (p - t) % n_shards
            kmin, kmax = bounds[r]
            if not causal:
                full[p] += qmin.size * kmin.size
                continue
            none_ok = kmin[None, :] > qmax[:, None]
            all_ok = kmax[None, :] <= qmin[:, None]
            skip[p] += int(none_ok.sum())
            full[p] += int(all_ok.sum())
            part[p] += int((~none_ok & ~all_ok).sum())
    return full, part, skip


def tile_classes_bruteforce(layout, seq, n_shards, causal=True, tile=128):
    """Same counts, deciding each tile by looking at every (q, k) pair in it."""
    pos = layout_positions(layout, seq, n_shards)
    s_n = seq // n_shards
    out = np.zeros((3, n_shards), np.int64)
    for p in range(n_shards):
        qp = pos[p * s_n:(p + 1) * s_n]
        for t in range(n_shards):
            r = (p - t) % n_shards
            kp = pos[r * s_n:(r + 1) * s_n]
            for i0 in range(0, s_n, tile):
                for j0 in range(0, s_n, tile):
                    ok = (kp[j0:j0 + tile][None, :] <= qp[i0:i0 + tile][:, None]) if causal \
                        else np.ones((len(qp[i0:i0 + tile]), len(kp[j0:j0 + tile])), bool)
                    cls = FULL if ok.all() else (SKIP if not ok.any() else PARTIAL)
                    out[cls, p] += 1
    return out[FULL], out[PARTIAL], out[SKIP]
