"""The ring itself, simulated device by device (oracle; test infrastructure only).

Follows the method as the pages state it:

* Q, K and V are split along the sequence into N shards; device p keeps its
  query block and starts out holding its own K/V block (Q&A page, "The ring",
  steps 1-4; Module 23, "Sequence Parallelism: Ring Attention").
* At every one of N steps each device folds the K/V block it holds into three
  running quantities per query row -- the max logit m, the denominator l and the
  unnormalised output o -- with the update of Module 23, "The Math: One Block at
  a Time":  m <- max(m, max_j s_j);  l <- l e^(m_old - m) + sum_j e^(s_j - m);
  o <- o e^(m_old - m) + sum_j e^(s_j - m) v_j.
* Then every device passes its block to the next device and receives one from
  the previous device (device i -> i+1: 3.6, "Ring Attention"; the Q&A page
  rotates its list of blocks the same way).  So at step t device p holds the
  block that started on device (p - t) mod N.
* At the end out = o / l.
* Causal: a block strictly in the future of all of a device's queries is skipped,
  any other block is masked key by key by global position (Module 23, "Exact by
  Construction": "skips any K/V block strictly in the future ... and masks the
  diagonal block").

Reading for the case the pages leave open: when every score seen so far is
masked, m stays -inf; the correction factor and the new probabilities are then
taken as 0 instead of the NaN that -inf - (-inf) would give.
"""

import numpy as np


def _scale(d, scale):
    return 1.0 / np.sqrt(d) if not scale else float(scale)


def _absorb(state, q_blk, k_blk, v_blk, allowed, sc):
    """Fold one K/V block into (m, l, o) of one device's query rows."""
    m_old, l_old, o_old = state
    s = (q_blk @ k_blk.T) * sc
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    m_new = np.maximum(m_old, s.max(axis=1))
    ref = np.where(np.isneginf(m_new), 0.0, m_new)      # no -inf - -inf
    corr = np.exp(m_old - ref)                           # e^(m_old - m_new)
    p = np.exp(s - ref[:, None])                         # e^(s_j - m_new)
    l_new = l_old * corr + p.sum(axis=1)
    o_new = o_old * corr[:, None] + p @ v_blk
    return m_new, l_new, o_new


def ring_sim(q, k, v, n_shards, positions=None, causal=False, scale=None):
    """Simulate the N-device ring on layout-ordered tensors.

    q: [B, Hq, S, d]; k, v: [B, Hkv, S, d], rows in layout order (shard p owns rows
    [p*S/N, (p+1)*S/N)).  positions: natural position of every row (needed for the
    causal mask; default 0..S-1, i.e. the contiguous layout).
    Returns O [B, Hq, S, d] and LSE [B, Hq, S] (float64) in layout order, with
    LSE = m + ln(l) on the scaled scores.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, S, d = q.shape
    group = Hq // k.shape[1]
    if S % n_shards:
        raise ValueError("seq must be a multiple of n_shards")
    s_n = S // n_shards
    sc = _scale(d, scale)
    pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)
    out = np.zeros_like(q)
    lse = np.full((B, Hq, S), -np.inf)
    shard = [slice(p * s_n, (p + 1) * s_n) for p in range(n_shards)]
    for b in range(B):
        for h in range(Hq):
            g = h // group
            queries = [q[b, h, sl] for sl in shard]
            qpos = [pos[sl] for sl in shard]
            # The block each device holds; device p starts with its own.
            held = [(k[b, g, sl], v[b, g, sl], pos[sl]) for sl in shard]
            state = [(np.full(s_n, -np.inf), np.zeros(s_n), np.zeros((s_n, d)))
                     for _ in range(n_shards)]
            for _step in range(n_shards):
                for dev in range(n_shards):
                    k_blk, v_blk, kpos = held[dev]
                    allowed = None
                    if causal:
                        allowed = kpos[None, :] <= qpos[dev][:, None]
                        if not allowed.any():
                            continue          # block strictly in the future: skipped
                    state[dev] = _absorb(state[dev], queries[dev], k_blk, v_blk, allowed, sc)
                # Pass K/V on: device dev now holds what device dev-1 held.
                held = [held[(dev - 1) % n_shards] for dev in range(n_shards)]
            for dev in range(n_shards):
                m, l, o = state[dev]
                with np.errstate(divide="ignore", invalid="ignore"):
                    out[b, h, shard[dev]] = np.where(l[:, None] > 0, o / l[:, None], 0.0)
                    lse[b, h, shard[dev]] = np.where(l > 0, m + np.log(l), -np.inf)
    return out, lse


def ring_partials(q, k, v, n_shards, positions=None, causal=False, scale=None):
    """Per-step partial results of the ring, one (O_t, LSE_t) per step t.

    Partial t of a row on device p is attention of that row over the block the
    device holds at step t -- the block that started on device (p - t) mod N --
    alone: O_t normalised by its own denominator, LSE_t = m_t + ln(l_t).  A
    skipped block (causal, strictly in the future) gives O_t = 0, LSE_t = -inf.
    Returns O_parts [N, B, Hq, S, d] and LSE_parts [N, B, Hq, S] in layout order.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, S, d = q.shape
    group = Hq // k.shape[1]
    s_n = S // n_shards
    sc = _scale(d, scale)
    pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)
    o_parts = np.zeros((n_shards, B, Hq, S, d))
    lse_parts = np.full((n_shards, B, Hq, S), -np.inf)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for p in range(n_shards):
                rows = slice(p * s_n, (p + 1) * s_n)
                for t in range(n_shards):
                    r = (p - t) % n_shards
                    cols = slice(r * s_n, (r + 1) * s_n)
                    allowed = None
                    if causal:
                        allowed = pos[cols][None, :] <= pos[rows][:, None]
                        if not allowed.any():
                            continue
                    fresh = (np.full(s_n, -np.inf), np.zeros(s_n), np.zeros((s_n, d)))
                    m, l, o = _absorb(fresh, q[b, h, rows], k[b, g, cols], v[b, g, cols], allowed, sc)
                    with np.errstate(divide="ignore", invalid="ignore"):
                        o_parts[t, b, h, rows] = np.where(l[:, None] > 0, o / l[:, None], 0.0)
                        lse_parts[t, b, h, rows] = np.where(l > 0, m + np.log(l), -np.inf)
    return o_parts, lse_parts


def pass_blocks(x, n_shards):
    """One exchange of the ring: every device hands the block it holds to the next.

    x: [..., S, d] in layout order (shard p owns rows [p*S/N, (p+1)*S/N)).  Returns a
    new array in which shard p's rows hold what shard p-1 (mod N) held -- device
    i -> i+1 (3.6, "Ring Attention"; the Q&A page, "The ring", rotates its block
    list the same way).
    """
    x = np.asarray(x)
    S = x.shape[-2]
    if S % n_shards:
        raise ValueError("seq must be a multiple of n_shards")
    s_n = S // n_shards
    blocks = [x[..., p * s_n:(p + 1) * s_n, :] for p in range(n_shards)]
    received = [blocks[(p - 1) % n_shards] for p in range(n_shards)]
    return np.concatenate(received, axis=-2)


def held_blocks(x, n_shards, step):
    """What every device holds at ring step ``step``: ``step`` exchanges of ``pass_blocks``."""
    x = np.asarray(x)
    for _ in range(step):
        x = pass_blocks(x, n_shards)
    return x
