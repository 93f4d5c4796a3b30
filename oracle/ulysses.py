"""DeepSpeed-Ulysses' exchange (oracle; test infrastructure only).

The Q&A page ("Explain ring attention ...", section "Related approaches") names
DeepSpeed-Ulysses as the alternative that splits by attention heads with an
all-to-all instead of a ring.  Reading: N devices each start with their shard of
the sequence (S/N tokens, in the layout's order) for all H heads; the all-to-all
hands device p' every token, in natural order, of heads p'*H/N .. (p'+1)*H/N - 1;
each device then runs ordinary attention over the whole sequence for its heads, and
a second all-to-all returns the outputs to the sequence shards.

Device buffers are packed side by side:
  sequence-sharded  [N, B, H, S/N, ...]   (device p: rows i of its shard)
  head-sharded      [N, B, H/N, S, ...]   (device p': natural positions s)
"""

import numpy as np


def ulysses_seq_to_head(x, positions, n_shards):
    """[N, B, H, S/N, ...] sequence shards -> [N, B, H/N, S, ...] head shards."""
    x = np.asarray(x)
    N, B, H, s_n = x.shape[:4]
    if N != n_shards or H % N:
        raise ValueError("need N shards and H divisible by N")
    hl = H // N
    pos = np.asarray(positions, np.int64)
    out = np.empty((N, B, hl, N * s_n) + x.shape[4:], dtype=x.dtype)
    for p in range(N):                       # sending device
        for i in range(s_n):                 # its local row i holds token pos[p*s_n + i]
            s = pos[p * s_n + i]
            for q in range(N):               # receiving device: heads q*hl .. q*hl + hl - 1
                out[q, :, :, s] = x[p, :, q * hl:(q + 1) * hl, i]
    return out


def ulysses_head_to_seq(y, positions, n_shards):
    """[N, B, H/N, S, ...] head shards -> [N, B, H, S/N, ...] sequence shards."""
    y = np.asarray(y)
    N, B, hl, S = y.shape[:4]
    if N != n_shards or S % N:
        raise ValueError("need N shards and S divisible by N")
    s_n = S // N
    pos = np.asarray(positions, np.int64)
    out = np.empty((N, B, hl * N, s_n) + y.shape[4:], dtype=y.dtype)
    for p in range(N):
        for i in range(s_n):
            s = pos[p * s_n + i]
            for q in range(N):
                out[p, :, q * hl:(q + 1) * hl, i] = y[q, :, :, s]
    return out
