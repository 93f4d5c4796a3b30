"""Gradients of ring attention (oracle; test infrastructure only).

The pages present ring attention as a way to train on long sequences (Module 23,
"Sequence Parallelism: Ring Attention"; 3.6, "Ring Attention": every layer's
activations are kept for the backward pass), but they print no backward pass.
So the oracle is the derivative of the forward's own definition,
O = softmax(scale * Q K^T + M) V with M = -inf on masked pairs, written out:

    P  = softmax(S),            S = scale * Q K^T + M
    dV = P^T dO
    dP = dO V^T
    dS = P * (dP - D),          D_i = sum_j P_ij dP_ij = sum_c dO_ic O_ic
    dQ = scale * dS K
    dK = scale * dS^T Q

With grouped query heads, a key/value head's dK and dV are sums over the query
heads that read it.  Everything is float64 numpy.

``ring_backward`` computes the same gradients the way the ring does: every
device p recomputes P for each block it meets from the forward's LSE
(P = exp(S - LSE)); its dQ accumulates locally, and each block's dK, dV
accumulators travel around the ring with the block and are home again after N
steps.
"""

import numpy as np


def _scale(d, scale):
    return 1.0 / np.sqrt(d) if not scale else float(scale)


def _mask(pos_q, pos_k, causal):
    if not causal:
        return None
    return pos_k[None, :] <= pos_q[:, None]


def attention_backward_rows(q_rows, do_rows, q_pos, k, v, k_pos=None, causal=False, scale=None, key_idx=None):
    """The gradient terms owed to a set of query rows of one (batch, query head).

    q_rows, do_rows: [n, d], the rows and their upstream gradients; q_pos: [n]
    their positions.  k, v: [S, d], every key and value of the head's key/value
    head, at positions ``k_pos`` (default 0..S-1).  A query row's dQ depends only
    on its own row of P, so it comes out whole.  dK and dV are sums over query
    rows: for the key rows ``key_idx`` (optional), the part these query rows add,
    scale * dS[:, j]^T q_rows and P[:, j]^T do_rows (``key_idx`` may be a slice).
    The parts of every query row that sees a key add up to that key's gradient.
    Returns dq [n, d], and with ``key_idx`` also dk_part and dv_part [len(key_idx), d].
    """
    q_rows, do_rows = (np.asarray(t, dtype=np.float64) for t in (q_rows, do_rows))
    k, v = np.asarray(k, dtype=np.float64), np.asarray(v, dtype=np.float64)
    sc = _scale(q_rows.shape[1], scale)
    kp = np.arange(k.shape[0], dtype=np.int64) if k_pos is None else np.asarray(k_pos, np.int64)
    s = sc * (q_rows @ k.T)
    allowed = _mask(np.asarray(q_pos, np.int64), kp, causal)
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    s_max = s.max(axis=1, keepdims=True)
    e = np.exp(s - s_max)
    p = e / e.sum(axis=1, keepdims=True)
    o = p @ v
    dp = do_rows @ v.T
    delta = (do_rows * o).sum(axis=1, keepdims=True)
    ds = p * (dp - delta)
    dq = sc * (ds @ k)
    if key_idx is None:
        return dq
    if not isinstance(key_idx, slice):
        key_idx = np.asarray(key_idx, np.int64)
    return dq, sc * (ds[:, key_idx].T @ q_rows), p[:, key_idx].T @ do_rows


def attention_backward(q, k, v, do, causal=False, positions=None, scale=None, block=None):
    """dQ, dK, dV of O = attention(q, k, v) for the upstream gradient dO.

    q, do: [B, Hq, S, d]; k, v: [B, Hkv, S, d]; rows in any order when
    ``positions`` gives each row's natural position (default 0..S-1).
    ``block``: take the query rows that many at a time (each row's softmax is its
    own; dK and dV add the blocks' contributions), so long sequences fit in memory.
    Returns (dq [B, Hq, S, d], dk [B, Hkv, S, d], dv [B, Hkv, S, d]) in float64.
    """
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, Hq, S, d = q.shape
    group = Hq // k.shape[1]
    pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)
    every_key = slice(None)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    step = S if block is None else int(block)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for r0 in range(0, S, step):
                rows = slice(r0, min(S, r0 + step))
                dq[b, h, rows], dk_part, dv_part = attention_backward_rows(
                    q[b, h, rows], do[b, h, rows], pos[rows], k[b, g], v[b, g], k_pos=pos, causal=causal,
                    scale=scale, key_idx=every_key)
                dk[b, g] += dk_part
                dv[b, g] += dv_part
    return dq, dk, dv


def ring_backward(q, k, v, do, o, lse, n_shards, positions=None, causal=False, scale=None):
    """The same gradients computed device by device around the ring.

    Inputs in layout order (shard p owns rows [p*S/N, (p+1)*S/N)); ``o`` and
    ``lse`` are the forward's output and log-sum-exp.  Device p meets, at step
    t, the block that started on device (p - t) mod N (the forward's rotation),
    recomputes its probabilities as exp(scale * q k - LSE), adds dS K to its own
    dQ, and adds P^T dO and dS^T Q to the dK, dV accumulators that travel with
    the block.  After N steps every accumulator is back on its block's device.
    """
    q, k, v, do, o = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do, o))
    lse = np.asarray(lse, dtype=np.float64)
    B, Hq, S, d = q.shape
    group = Hq // k.shape[1]
    N = n_shards
    s_n = S // N
    sc = _scale(d, scale)
    pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)
    rows = [slice(p * s_n, (p + 1) * s_n) for p in range(N)]
    delta = (do * o).sum(axis=-1)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            # block r with its travelling accumulators, held by device p at step t
            held = [(r, np.zeros((s_n, d)), np.zeros((s_n, d))) for r in range(N)]
            for _step in range(N):
                for p in range(N):
                    r, dk_acc, dv_acc = held[p]
                    qp, kr = rows[p], rows[r]
                    allowed = _mask(pos[qp], pos[kr], causal)
                    if allowed is not None and not allowed.any():
                        continue              # block strictly in the future: skipped
                    s = sc * (q[b, h, qp] @ k[b, g, kr].T)
                    p_blk = np.exp(s - lse[b, h, qp][:, None])
                    if allowed is not None:
                        p_blk = np.where(allowed, p_blk, 0.0)
                    dp = do[b, h, qp] @ v[b, g, kr].T
                    ds = p_blk * (dp - delta[b, h, qp][:, None])
                    dq[b, h, qp] += sc * (ds @ k[b, g, kr])
                    dk_acc += sc * (ds.T @ q[b, h, qp])
                    dv_acc += p_blk.T @ do[b, h, qp]
                # pass each block, with its accumulators, to the next device
                held = [held[(p - 1) % N] for p in range(N)]
            for r, dk_acc, dv_acc in held:     # home again: held[r] carries block r
                dk[b, g, rows[r]] += dk_acc
                dv[b, g, rows[r]] += dv_acc
    return dq, dk, dv
