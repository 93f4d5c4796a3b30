"""Plain softmax attention in float64 (oracle; test infrastructure only).

This is the quantity the ring reaches exactly: Module 23, "Exact by Construction"
compares the ring against ``softmax(q k^T * scale) v`` computed on one device,
and the Q&A page's simulation ("The ring") checks its result against the same
expression.  Scores are ``s_ij = q_i . k_j / sqrt(d)`` ("The Math: One Block at a
Time").  The causal variant blanks keys strictly after the query (the
``triu(..., diagonal=1)`` mask of "Exact by Construction"), so the diagonal is
kept.

Conventions fixed here because the pages do not state them:
* LSE is the natural-log log-sum-exp of the scaled, masked scores of a row.
* GQA: query head h reads key/value head h // (Hq/Hkv).
* A row with no allowed key (not reachable in causal self-attention) gives
  O = 0 and LSE = -inf.
"""

import numpy as np


def _scale(d, scale):
    return 1.0 / np.sqrt(d) if not scale else float(scale)


def full_attention(q, k, v, causal=False, scale=None, positions=None, row_block=1024):
    """O and LSE of ordinary softmax attention.

    q: [B, Hq, S, d]; k, v: [B, Hkv, S, d] (any float dtype; computed in float64).
    positions: natural position of each of the S rows (default 0..S-1); the causal
    mask compares positions, so layout-ordered inputs may be passed with their
    layout's positions.
    Returns O [B, Hq, S, d] float64 and LSE [B, Hq, S] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    sc = _scale(d, scale)
    pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)
    out = np.zeros((B, Hq, S, d), dtype=np.float64)
    lse = np.full((B, Hq, S), -np.inf, dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kh = k[b, h // group]
            vh = v[b, h // group]
            for r0 in range(0, S, row_block):
                r1 = min(S, r0 + row_block)
                s = (q[b, h, r0:r1] @ kh.T) * sc
                if causal:
                    s = np.where(pos[None, :] <= pos[r0:r1, None], s, -np.inf)
                row_max = s.max(axis=1)
                live = np.isfinite(row_max)
                shift = np.where(live, row_max, 0.0)
                e = np.exp(s - shift[:, None])
                z = e.sum(axis=1)
                with np.errstate(divide="ignore", invalid="ignore"):
                    probs = np.where(live[:, None], e / z[:, None], 0.0)
                    lse[b, h, r0:r1] = np.where(live, shift + np.log(z), -np.inf)
                out[b, h, r0:r1] = probs @ vh
    return out, lse


def full_attention_rows(q, k, v, picks, causal=False, scale=None, positions=None, chunk=64):
    """O and LSE for selected rows only, each computed against all S keys.

    picks: iterable of (b, h, row) with row an index into the S axis.
    Returns O [n, d] and LSE [n] in float64, in the order of ``picks``.
    Rows sharing a (b, kv-head) are batched so the keys are converted once.
    """
    picks = [tuple(int(x) for x in t) for t in picks]
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    sc = _scale(d, scale)
    pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)
    out = np.zeros((len(picks), d), dtype=np.float64)
    lse = np.full(len(picks), -np.inf, dtype=np.float64)
    by_kv = {}
    for n, (b, h, r) in enumerate(picks):
        by_kv.setdefault((b, h // group), []).append(n)
    for (b, g), idxs in by_kv.items():
        kh = np.asarray(k[b, g], dtype=np.float64)
        vh = np.asarray(v[b, g], dtype=np.float64)
        for c0 in range(0, len(idxs), chunk):
            sel = idxs[c0:c0 + chunk]
            qs = np.stack([np.asarray(q[b, picks[n][1], picks[n][2]], dtype=np.float64) for n in sel])
            s = (qs @ kh.T) * sc
            if causal:
                qp = np.array([pos[picks[n][2]] for n in sel], dtype=np.int64)
                s = np.where(pos[None, :] <= qp[:, None], s, -np.inf)
            row_max = s.max(axis=1)
            live = np.isfinite(row_max)
            shift = np.where(live, row_max, 0.0)
            e = np.exp(s - shift[:, None])
            z = e.sum(axis=1)
            with np.errstate(divide="ignore", invalid="ignore"):
                probs = np.where(live[:, None], e / z[:, None], 0.0)
                lse[sel] = np.where(live, shift + np.log(z), -np.inf)
            out[sel] = probs @ vh
    return out, lse


def attention_rows(q_rows, k_head, v_head, q_positions=None, k_positions=None, causal=False,
                   scale=None, chunk=64):
    """O and LSE of individual query rows against one key/value head.

    q_rows: [n, d]; k_head, v_head: [S, d]; positions are natural token positions
    (needed when causal).  The plain definition again, one row block at a time so
    that million-key heads fit in memory.  When the keys are given in natural
    order (k_positions None) a causal row block only reads keys up to its largest
    position: later keys are masked and carry no weight.
    Returns O [n, d], LSE [n] in float64.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    n, d = q_rows.shape
    sc = _scale(d, scale)
    out = np.zeros((n, d))
    lse = np.full(n, -np.inf)
    natural_keys = k_positions is None
    order = np.arange(n)
    if causal:
        qp = np.asarray(q_positions, np.int64)
        kp = np.arange(k_head.shape[0], dtype=np.int64) if natural_keys else np.asarray(k_positions, np.int64)
        order = np.argsort(qp, kind="stable")
    for c0 in range(0, n, chunk):
        rows = order[c0:c0 + chunk]
        limit = k_head.shape[0]
        if causal and natural_keys:
            limit = int(qp[rows].max()) + 1
        kh = np.asarray(k_head[:limit], dtype=np.float64)
        vh = np.asarray(v_head[:limit], dtype=np.float64)
        s = (q_rows[rows] @ kh.T) * sc
        if causal:
            s = np.where(kp[None, :limit] <= qp[rows, None], s, -np.inf)
        row_max = s.max(axis=1)
        live = np.isfinite(row_max)
        shift = np.where(live, row_max, 0.0)
        e = np.exp(s - shift[:, None])
        z = e.sum(axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            probs = np.where(live[:, None], e / z[:, None], 0.0)
            lse[rows] = np.where(live, shift + np.log(z), -np.inf)
        out[rows] = probs @ vh
    return out, lse
