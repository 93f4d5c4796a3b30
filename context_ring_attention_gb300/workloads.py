"""Synthetic workloads of the ring-attention forward and their seeded inputs.

This module holds configuration data and random-number draws only; it performs
none of the method's arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it.

Inputs are drawn in NATURAL token order; callers move them into a ring layout
with ``ra_layout_perm`` (device) or index by the layout positions (host).
"""

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seq: int
    heads_q: int
    heads_kv: int
    head_dim: int
    n_shards: int
    layouts: tuple            # layouts the workload is run under
    causal: bool
    dtype: str                # "f32" or "bf16"
    seed_base: int            # Q/K/V seeds are seed_base + 0/1/2
    q_scale: float = 1.0      # Q multiplied after the draw (exact in bf16 for powers of 2)
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def s_n(self):
        return self.seq // self.n_shards

    def flops(self):
        """Algorithmic FLOPs: 4*d per allowed (q, k) pair (two matmuls), per (batch, query head)."""
        pairs = self.seq * (self.seq + 1) // 2 if self.causal else self.seq * self.seq
        return 4 * self.head_dim * pairs * self.batch * self.heads_q


WORKLOADS = {
    # The Q&A page's 4-device toy ring ("The ring"): inputs from numpy default_rng(1).
    "toy_ring_4x3_d8": Workload("toy_ring_4x3_d8", 1, 12, 1, 1, 8, 4, ("contiguous",), False, "f32", 1,
                                note="Q, K, V = three rng.normal((12, 8)) draws of default_rng(1)"),
    "noncausal_4k_n8": Workload("noncausal_4k_n8", 2, 4096, 32, 32, 128, 8, ("contiguous",), False, "bf16", 2000),
    "noncausal_4k_n8_q4": Workload("noncausal_4k_n8_q4", 2, 4096, 32, 32, 128, 8, ("contiguous",), False, "bf16",
                                   2000, q_scale=4.0, note="Q x4 stresses running-max rescaling"),
    "causal_32k_n8": Workload("causal_32k_n8", 1, 32768, 32, 8, 128, 8, ("contiguous", "zigzag"), True, "bf16", 3000),
    "striped_131k_n32": Workload("striped_131k_n32", 1, 131072, 32, 8, 128, 32, ("striped",), True, "bf16", 4000),
    "zigzag_1m_n8": Workload("zigzag_1m_n8", 1, 1048576, 32, 8, 128, 8, ("zigzag",), True, "bf16", 5000),
}


def toy_inputs():
    """The toy ring's Q, K, V as float64 [12, 8] arrays, drawn exactly as the page does."""
    rng = np.random.default_rng(1)
    return tuple(rng.normal(size=(12, 8)) for _ in range(3))


def torch_inputs(wl, device, chunk_rows=1 << 22):
    """Natural-order q [B,Hq,S,d], k, v [B,Hkv,S,d] as torch tensors of the workload dtype.

    bf16: iid N(0,1) drawn in float32 by a torch.Generator on `device` seeded
    seed_base+{0,1,2}, then rounded to bf16 (RNE); drawn in row chunks so the
    float32 staging stays small.  f32 toy: the page's numpy draws.
    """
    import torch
    if wl.dtype == "f32" and wl.name == "toy_ring_4x3_d8":
        q, k, v = toy_inputs()
        as_t = lambda a: torch.tensor(a, dtype=torch.float32, device=device).reshape(1, 1, 12, 8).contiguous()
        return as_t(q), as_t(k), as_t(v)
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    out = []
    for n, heads in enumerate((wl.heads_q, wl.heads_kv, wl.heads_kv)):
        g = torch.Generator(device=device)
        g.manual_seed(wl.seed_base + n)
        t = torch.empty((wl.batch, heads, wl.seq, wl.head_dim), dtype=dt, device=device)
        flat = t.view(-1, wl.head_dim)
        for r0 in range(0, flat.shape[0], chunk_rows):
            r1 = min(flat.shape[0], r0 + chunk_rows)
            x = torch.randn((r1 - r0, wl.head_dim), generator=g, device=device, dtype=torch.float32)
            if n == 0 and wl.q_scale != 1.0:
                x.mul_(wl.q_scale)
            flat[r0:r1].copy_(x)
        out.append(t)
    return tuple(out)


def small_inputs(batch, seq, heads_q, heads_kv, head_dim, seed, device, dtype, q_scale=1.0):
    """Seeded iid N(0,1) tensors for parity tests of arbitrary small shapes."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    q = (torch.randn((batch, heads_q, seq, head_dim), generator=g, device=device) * q_scale).to(dt)
    k = torch.randn((batch, heads_kv, seq, head_dim), generator=g, device=device).to(dt)
    v = torch.randn((batch, heads_kv, seq, head_dim), generator=g, device=device).to(dt)
    return q.contiguous(), k.contiguous(), v.contiguous()


def sample_rows(wl, n_rows=4096, seed=7, heads=None):
    """(b, h, natural position) picks: forced edge rows plus uniform draws without replacement.

    Forced: positions 0, 1, S-1 and the first/last position of every zigzag chunk
    (2N chunks) or of every striped/contiguous shard's first and last rows, for
    heads 0 and Hq-1.  They count within n_rows.
    """
    S, N = wl.seq, wl.n_shards
    heads = wl.heads_q if heads is None else heads
    forced_pos = {0, 1, S - 1}
    c = S // (2 * N)
    for j in range(2 * N):
        forced_pos.update({j * c, j * c + c - 1})
    for p in range(N):
        forced_pos.update({p, S - N + p, p * (S // N), (p + 1) * (S // N) - 1})
    picks = [(0, h, x) for x in sorted(forced_pos) for h in (0, heads - 1)]
    picks = list(dict.fromkeys(picks))
    rng = np.random.default_rng(seed)
    total = wl.batch * heads * S
    taken = set(picks)
    while len(picks) < n_rows:
        for f in rng.integers(0, total, size=2 * (n_rows - len(picks)) + 16):
            b, rem = divmod(int(f), heads * S)
            h, x = divmod(rem, S)
            if (b, h, x) not in taken:
                taken.add((b, h, x))
                picks.append((b, h, x))
                if len(picks) == n_rows:
                    break
    return picks[:n_rows]
