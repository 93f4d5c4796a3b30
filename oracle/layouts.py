"""Token-to-device layouts (oracle; test infrastructure only).

A layout says which global token positions device (shard) p owns.  Tensors handed
to the ring are in *layout order*: shard p occupies rows [p*S_N, (p+1)*S_N) and
row p*S_N + i holds the token whose natural position is ``pos[p*S_N + i]``.
"""

import numpy as np

CONTIGUOUS = "contiguous"
STRIPED = "striped"
ZIGZAG = "zigzag"
LAYOUTS = (CONTIGUOUS, STRIPED, ZIGZAG)


def _check(layout, seq, n_shards):
    if layout not in LAYOUTS:
        raise ValueError(f"unknown layout {layout!r}")
    if n_shards < 1 or seq % n_shards:
        # Uneven shards are rejected, never silently handled (Module 23, "Common
        # Pitfalls": uneven shards are rejected rather than silently biased).
        raise ValueError("seq must be a multiple of n_shards")
    if layout == ZIGZAG and seq % (2 * n_shards):
        raise ValueError("zigzag needs seq to be a multiple of 2*n_shards")


def layout_positions(layout, seq, n_shards):
    """Natural position of every layout-ordered row, as int64 of length ``seq``.

    * contiguous -- device p holds the p-th contiguous block of S/N positions
      (Q&A page, "The ring", step 1 "Split"; 3.6, "Sequence & Context
      Parallelism": GPU 0 owns tokens 0..s/c-1, GPU 1 the next chunk, ...).
    * striped -- device p holds positions p, p+N, p+2N, ... (Module 23, "The
      Causal Imbalance — and the Striped Fix").
    * zigzag -- the pages only say "the same idea, paired up block-by-block".
      Reading used here: cut the sequence into 2N equal chunks; device p holds
      chunk p followed by chunk 2N-1-p (an early chunk paired with a late one).
    """
    _check(layout, seq, n_shards)
    s_n = seq // n_shards
    pos = np.empty(seq, dtype=np.int64)
    local = np.arange(s_n, dtype=np.int64)
    for p in range(n_shards):
        rows = slice(p * s_n, (p + 1) * s_n)
        if layout == CONTIGUOUS:
            pos[rows] = p * s_n + local
        elif layout == STRIPED:
            pos[rows] = local * n_shards + p
        else:
            c = seq // (2 * n_shards)
            first = p * c + local[:c]
            second = (2 * n_shards - 1 - p) * c + local[: s_n - c]
            pos[rows] = np.concatenate([first, second])
    return pos


def causal_pair_counts(n_shards, block_size, layout):
    """Causal (q, k) pairs each device computes, counted pair by pair.

    A pair is causal when the key's position is not after the query's (the
    diagonal is kept: the reference mask of "Exact by Construction" only blanks
    keys strictly after the query).  Returns a dict with ``work`` (per device),
    ``imbalance`` (max/min) and ``total`` — the quantities printed in Module 23,
    "The Causal Imbalance — and the Striped Fix".
    """
    seq = n_shards * block_size
    pos = layout_positions(layout, seq, n_shards)
    all_keys = np.arange(seq, dtype=np.int64)
    work = []
    for p in range(n_shards):
        q = pos[p * block_size:(p + 1) * block_size]
        allowed = all_keys[None, :] <= q[:, None]
        work.append(int(allowed.sum()))
    return {"work": work, "imbalance": max(work) / min(work), "total": sum(work)}


def to_natural(x, positions):
    """Rows in layout order -> natural order along axis -2: out[..., pos[j], :] = x[..., j, :].

    What the all-gather variant of context parallelism hands every device: the K/V
    blocks of all shards, each row at its token position.
    """
    x = np.asarray(x)
    pos = np.asarray(positions, np.int64)
    out = np.empty_like(x)
    out[..., pos, :] = x
    return out
