"""Shapes that stress the kernels' index arithmetic, run through every bf16 and f32 path.

``run_cases()`` uses whichever library the binding loads.  The debug-bounds GPU
test runs it once in a child process with RA_LIBRARY_VARIANT=debug (libra_debug.so,
whose kernels check their tensor-memory, shared-memory and global indices and
report a failed check as RA_ERR_BOUNDS through the status word) and once in its own
process with libra.so, and requires both to pass every status check and to produce
the same bits.  Run as ``python -m tests.bounds_cases OUT.npz`` for the child.
"""

import sys

import numpy as np

# B, S, Hq, Hkv, N, layout, causal: ragged tiles, shards shorter than one tile,
# odd and unit GQA groups, a single shard, every layout.
FWD_SHAPES = [
    (1, 1024, 4, 2, 2, "zigzag", True),
    (1, 900, 4, 2, 3, "striped", True),
    (1, 900, 4, 2, 3, "contiguous", False),
    (2, 640, 2, 2, 4, "contiguous", True),
    (1, 768, 6, 2, 2, "zigzag", True),
    (1, 256, 8, 1, 1, "contiguous", True),
    (1, 320, 2, 1, 8, "zigzag", True),
    (1, 320, 2, 2, 8, "striped", False),
    (1, 16, 4, 2, 16, "contiguous", True),
    (1, 32, 4, 2, 16, "zigzag", True),
    (1, 48, 4, 2, 16, "striped", False),
]
BWD_SHAPES = [
    (1, 900, 4, 2, 3, "striped", True),
    (1, 320, 2, 1, 8, "zigzag", True),
    (2, 640, 2, 2, 4, "contiguous", False),
    (1, 768, 6, 2, 2, "zigzag", True),
    (1, 48, 4, 2, 16, "striped", True),
]


def run_cases():
    """Every case's outputs as float32 numpy arrays, keyed by case name."""
    import torch

    import context_ring_attention_gb300 as ra
    from context_ring_attention_gb300 import workloads

    out = {}
    dev = "cuda"

    def keep(name, *tensors):
        for n, t in enumerate(tensors):
            out[f"{name}/{n}"] = t.float().cpu().numpy()

    for n_case, (B, S, Hq, Hkv, N, layout, causal) in enumerate(FWD_SHAPES):
        q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=700 + n_case, device=dev, dtype="bf16")
        plan = ra.ra_plan(B, S, Hq, Hkv, 128, N, layout, causal, "bf16")
        name = f"fwd{n_case}"
        keep(name, *ra.ra_fwd(plan, q, k, v))
        ra.ra_sync_status(plan)
        op, lp = ra.ra_fwd(plan, q, k, v, partials=True)
        ra.ra_sync_status(plan)
        keep(name + "_merged", *ra.ra_merge_partials(op, lp, out_dtype=torch.bfloat16))
        keep(name + "_ring", *ra.ra_ring_fwd(plan, q, k, v))
        ra.ra_sync_status(plan)
        k_all, v_all = ra.ra_allgather_kv(plan, k, v)
        keep(name + "_gathered", *ra.ra_fwd_gathered(plan, q, k_all, v_all))
        ra.ra_sync_status(plan)
        keep(name + "_static", *ra.ra_fwd_static(B, S, Hq, Hkv, N, layout, causal, q, k, v))
        ra.ra_fwd_static_status()
        ra.ra_plan_destroy(plan)

    for n_case, (B, S, Hq, Hkv, N, layout, causal) in enumerate(BWD_SHAPES):
        q, k, v = workloads.small_inputs(B, S, Hq, Hkv, 128, seed=800 + n_case, device=dev, dtype="bf16")
        g = torch.Generator(device=dev)
        g.manual_seed(900 + n_case)
        do = torch.randn(q.shape, generator=g, device=dev).to(torch.bfloat16)
        plan = ra.ra_plan(B, S, Hq, Hkv, 128, N, layout, causal, "bf16")
        o, lse = ra.ra_fwd(plan, q, k, v)
        keep(f"bwd{n_case}", *ra.ra_bwd(plan, q, k, v, o, lse, do))
        ra.ra_sync_status(plan)
        ra.ra_plan_destroy(plan)

    # f32 (CUDA cores), d = 32: forward, partials and backward
    q, k, v = workloads.small_inputs(2, 96, 4, 4, 32, seed=950, device=dev, dtype="f32")
    do = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(951), device=dev)
    plan = ra.ra_plan(2, 96, 4, 4, 32, 4, "zigzag", True, "f32")
    o, lse = ra.ra_fwd(plan, q, k, v)
    keep("f32_fwd", o, lse)
    op, lp = ra.ra_fwd(plan, q, k, v, partials=True)
    keep("f32_parts", op, lp)
    keep("f32_bwd", *ra.ra_bwd(plan, q, k, v, o, lse, do))
    ra.ra_sync_status(plan)
    ra.ra_plan_destroy(plan)
    torch.cuda.synchronize()
    return out


if __name__ == "__main__":
    np.savez(sys.argv[1], **run_cases())
