"""DeepSpeed-Ulysses' exchange (oracle; test infrastructure only).

The Q&A page ("Explain ring attention ...", section "Related approaches") names
DeepSpeed-Ulysses as the alternative that splits by attention heads with an
all-to-all instead of a ring.  Reading: N devices each start with their shard of
the sequence (S/N tokens, in the layout's order) for all H heads; the all-to-all
hands device p' every token, in natural order, of heads p'*H/N .. (p'+1)*H/N - 1;
each device then runs ordinary attention over the whole sequence for its heads, and
a second all-to-all returns the outputs to the sequence shards.

Packing (as the library's tensors):
  sequence-sharded  [B, H, S, ...] in layout order: device p holds rows
                    [p*S/N, (p+1)*S/N) of every (batch, head)
  head-sharded      [N, B, H/N, S, ...]: device p' holds heads p'*H/N.. by position
"""

import numpy as np


def ulysses_seq_to_head(x, positions, n_shards):
    """[B, H, S, ...] layout-ordered sequence shards -> [N, B, H/N, S, ...] head shards."""
    x = np.asarray(x)
    B, H, S = x.shape[:3]
    N = n_shards
    if H % N or S % N:
        raise ValueError("need H and S divisible by N")
    hl, s_n = H // N, S // N
    pos = np.asarray(positions, np.int64)
    out = np.empty((N, B, hl, S) + x.shape[3:], dtype=x.dtype)
    for p in range(N):                       # sending device
        for i in range(s_n):                 # its local row i holds token pos[p*s_n + i]
            s = pos[p * s_n + i]
            for q in range(N):               # receiving device: heads q*hl .. q*hl + hl - 1
                out[q, :, :, s] = x[:, q * hl:(q + 1) * hl, p * s_n + i]
    return out


def ulysses_head_to_seq(y, positions, n_shards):
    """[N, B, H/N, S, ...] head shards -> [B, H, S, ...] layout-ordered sequence shards."""
    y = np.asarray(y)
    N, B, hl, S = y.shape[:4]
    if N != n_shards or S % N:
        raise ValueError("need N shards and S divisible by N")
    s_n = S // N
    pos = np.asarray(positions, np.int64)
    out = np.empty((B, hl * N, S) + y.shape[4:], dtype=y.dtype)
    for p in range(N):
        for i in range(s_n):
            s = pos[p * s_n + i]
            for q in range(N):
                out[:, q * hl:(q + 1) * hl, p * s_n + i] = y[q, :, :, s]
    return out
