"""Benchmark of the ring-attention forward on GB300 (one JSON line on stdout).

A step is one pass of the whole path over one batch of synthetic input that is
already resident in HBM: natural-order Q, K, V are moved into the ring layout
(ra_layout_perm), the ring forward runs (ra_fwd, fused O and LSE), and O and
LSE are moved back to natural order.  Default workload: causal zigzag, 1,048,576
tokens in 8 shards, batch 1, 32 query / 8 key-value heads, d = 128, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload on the host cores (the only other place this script runs the oracle).
Under torchrun each rank runs an independent replica (no data-path collective);
rank 0 prints max-over-ranks timing.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attention fwd TFLOP/s (bf16, 1 GB300) and % of dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, dist_mod, device):
    """Element-wise maximum of per-rank values over all ranks (the values themselves
    without a process group): the job is as slow as its slowest replica."""
    if dist_mod is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return t.tolist()


def job_rate(world, flops_per_rank, ms):
    """Whole-job TFLOP/s of `world` replicas that each do flops_per_rank in ms (weak scaling)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# Dense bf16 tensor-core rate of one SM per clock: a 128 x 256 x 16 MMA (1,048,576
# FLOP) issues every 128 cycles.  152 SMs at 2070 MHz give 2577 TFLOP/s; a stand-alone
# MMA issue loop measured 2430 TFLOP/s (0.94 of it) at that clock.
TC_FLOP_PER_CLK_SM = 8192


def clock_peak(sms, sm_mhz):
    """The tensor pipe's issue-rate peak (TFLOP/s) at the SM clock the kernel ran at."""
    if not sm_mhz:
        return None
    return sms * TC_FLOP_PER_CLK_SM * float(sm_mhz) * 1e6 / 1e12


# The exponential unit: 32 ex2.approx per clock per SM (measured on a GB300 with 256
# threads per SM on independent chains: 31.3; the packed bf16x2 and f16x2 forms give
# the same element rate).  The forward takes one exponential per credited (q, k) pair,
# i.e. per 4*d = 512 algorithmic FLOPs at d = 128.
EX2_PER_CLK_SM = 32


def exp_rate(flops, head_dim, seconds, sms, sm_mhz):
    """Exponentials per second of the credited pairs against the unit's rate at the clock."""
    achieved = flops / (4 * head_dim) / seconds
    peak = sms * EX2_PER_CLK_SM * float(sm_mhz) * 1e6 if sm_mhz else None
    return {"achieved_per_s": achieved, "peak_per_s": peak, "frac": achieved / peak if peak else None,
            "note": (f"one exp per credited (q, k) pair (4 x d FLOPs); peak {sms} SMs x {EX2_PER_CLK_SM} ex2 per SM "
                     "clock x the median SM clock; masked pairs inside partial tiles also take an exp, uncredited")}


# A (batch, key/value head) unit of the end-to-end pipeline needs this many FLOPs
# (about 0.1 s of forward) before a step is split into such units.
E2E_UNIT_FLOPS = 2e14


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle --

def blas_threads():
    """Threads of the BLAS numpy calls (None when it cannot be asked)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            libs = sorted({ln.split()[-1] for ln in f if "blas" in ln.lower() and ".so" in ln})
    except OSError:
        return None
    for lib in libs:
        try:
            h = ctypes.CDLL(lib)
        except OSError:
            continue
        for name in ("openblas_get_num_threads", "scipy_openblas_get_num_threads64_",
                     "openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            fn = getattr(h, name, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


def ring_sim_timings():
    """The ring simulation oracle (the Q&A page's N-round loop) timed on the two small
    workloads: the toy ring in full, and one (batch, head) of the 4k non-causal ring
    (extrapolated to its 64 heads)."""
    import oracle
    from context_ring_attention_gb300 import workloads
    out = {}
    toy = workloads.WORKLOADS["toy_ring_4x3_d8"]
    q, k, v = (a.reshape(1, 1, 12, 8) for a in workloads.toy_inputs())
    reps = 200
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.ring_sim(q, k, v, toy.n_shards)
    dt = (time.perf_counter() - t0) / reps
    out[toy.name] = {"seconds": dt, "TFLOP/s": toy.flops() / dt / 1e12, "sample": "whole problem"}
    wl = workloads.WORKLOADS["noncausal_4k_n8"]
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((1, 1, wl.seq, wl.head_dim)) for _ in range(3))
    t0 = time.perf_counter()
    oracle.ring_sim(q, k, v, wl.n_shards)
    dt = time.perf_counter() - t0
    per_head = wl.flops() / (wl.batch * wl.heads_q)
    out[wl.name] = {"seconds": dt, "TFLOP/s": per_head / dt / 1e12,
                    "sample": f"one (batch, head) of {wl.batch * wl.heads_q}, N(0,1) float64",
                    "extrapolated_full_s": dt * wl.batch * wl.heads_q}
    return out


def cpu_baseline_record(wl, rows, seed=11, with_ring_sim=True):
    """The cpu_baseline object: the oracle's rate on a bounded sample, the threads it
    ran on, and the whole workload's time extrapolated from that rate."""
    v_cpu, dt, _, desc = cpu_oracle_sample(wl, rows=rows, seed=seed)
    rec = {"value": v_cpu, "unit": "TFLOP/s", "cores": os.cpu_count(), "blas_threads": blas_threads(),
           "kind": "oracle", "sample": desc, "seconds": dt,
           "extrapolated_full_s": wl.flops() / (v_cpu * 1e12),
           "extrapolated_note": "whole workload at the sample's rate (extrapolated, not run)"}
    if with_ring_sim:
        rec["ring_sim"] = ring_sim_timings()
    return rec


def cpu_oracle_sample(wl, rows=192, seed=11):
    """Time the float64 oracle on `rows` causal query rows of one key/value head.

    Inputs are host-drawn N(0,1) of the workload's shape (one kv head, rows of its
    query heads at uniformly drawn positions); returns (TFLOP/s, seconds, flops, desc).
    """
    import oracle
    rng = np.random.default_rng(seed)
    S, d = wl.seq, wl.head_dim
    k = rng.standard_normal((S, d))
    v = rng.standard_normal((S, d))
    pos_all = oracle.layout_positions(wl.layouts[0], S, wl.n_shards)
    qpos = np.sort(rng.choice(S, size=rows, replace=False))
    q = rng.standard_normal((rows, d))
    t0 = time.perf_counter()
    oracle.attention_rows(q, k[pos_all], v[pos_all], q_positions=qpos, k_positions=pos_all,
                          causal=wl.causal)
    dt = time.perf_counter() - t0
    keys = (qpos + 1) if wl.causal else np.full(rows, S)
    flops = 4.0 * d * float(keys.sum())
    desc = (f"{rows} query rows (uniform positions, seed {seed}) of one head against all {S} keys "
            f"of the {wl.name} workload, float64 numpy oracle")
    return flops / dt / 1e12, dt, flops, desc


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    times, tf = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        v, dt, flops, desc = cpu_oracle_sample(wl, rows=args.ref_rows, seed=100 + i)
        if i >= args.warmup:
            times.append(dt)
            tf.append(v)
    value = statistics.median(tf)
    cores = os.cpu_count()
    full_s = wl.flops() / (value * 1e12)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "blas_threads": blas_threads(),
                         "kind": "oracle", "sample": desc, "extrapolated_full_s": full_s,
                         "extrapolated_note": "whole workload at the sample's rate (extrapolated, not run)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(wl):
    return {"workload": wl.name, "batch": wl.batch, "seq": wl.seq, "heads_q": wl.heads_q,
            "heads_kv": wl.heads_kv, "head_dim": wl.head_dim, "n_shards": wl.n_shards,
            "layout": wl.layouts[0], "causal": wl.causal,
            "l2": "inputs larger than L2 (no flush needed)"}


# ------------------------------------------------------------- GPU (ours) --

def run_ours(args, wl):
    import torch
    import context_ring_attention_gb300 as ra
    from context_ring_attention_gb300 import workloads

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    dev = torch.device("cuda", local)
    layout = wl.layouts[0]
    N = wl.n_shards
    plan = ra.ra_plan(wl.batch, wl.seq, wl.heads_q, wl.heads_kv, wl.head_dim, N, layout, wl.causal, wl.dtype)
    q, k, v = workloads.torch_inputs(wl, dev)
    ql, kl, vl = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    o_l = torch.empty_like(q)
    lse_l = torch.empty((wl.batch, wl.heads_q, wl.seq), dtype=torch.float32, device=dev)
    o_n = torch.empty_like(q)
    lse_n = torch.empty_like(lse_l)
    stream = torch.cuda.current_stream()
    launches_per_step = 6
    if args.path == "ring":
        # explicit ring driver: scratch for two receive buffers and the N partials
        kbuf = torch.empty((2,) + tuple(k.shape), dtype=k.dtype, device=dev)
        vbuf = torch.empty_like(kbuf)
        o_parts = torch.empty((N,) + tuple(q.shape), dtype=torch.float32, device=dev)
        lse_parts = torch.empty((N,) + tuple(lse_l.shape), dtype=torch.float32, device=dev)
        comm = torch.cuda.Stream(device=dev)
        launches_per_step = 5 + N + 1   # permutes, one forward launch per ring step, the merge
    if args.path == "allgather":
        k_all, v_all = torch.empty_like(k), torch.empty_like(v)
        launches_per_step = 5 + 2 + 1   # permutes, the K and V gathers, the forward
    if args.path == "ulysses":
        Hl, Hkl = wl.heads_q // N, wl.heads_kv // N
        uplan = ra.ra_plan(N * wl.batch, wl.seq, Hl, Hkl, wl.head_dim, 1, "contiguous", wl.causal, wl.dtype)
        qh = torch.empty((N, wl.batch, Hl, wl.seq, wl.head_dim), dtype=q.dtype, device=dev)
        kh = torch.empty((N, wl.batch, Hkl, wl.seq, wl.head_dim), dtype=q.dtype, device=dev)
        vh, oh = torch.empty_like(kh), torch.empty_like(qh)
        lh = torch.empty((N, wl.batch, Hl, wl.seq), dtype=torch.float32, device=dev)
        launches_per_step = 5 + 3 + 1 + 2   # permutes, 3 exchanges, the forward, 2 exchanges back

    def forward(qx, kx, vx):
        if args.path == "ring":
            ra.ra_ring_fwd(plan, qx, kx, vx, o=o_l, lse=lse_l, k_buf=kbuf, v_buf=vbuf, o_parts=o_parts,
                           lse_parts=lse_parts, comm_stream=comm)
        elif args.path == "allgather":
            ra.ra_allgather_kv(plan, kx, vx, k_all, v_all)
            ra.ra_fwd_gathered(plan, qx, k_all, v_all, o=o_l, lse=lse_l)
        elif args.path == "ulysses":
            for src, dst in ((qx, qh), (kx, kh), (vx, vh)):
                ra.ra_ulysses_a2a(src, layout, N, 0, out=dst)
            B_ = N * wl.batch
            ra.ra_fwd(uplan, qh.view(B_, Hl, wl.seq, -1), kh.view(B_, Hkl, wl.seq, -1), vh.view(B_, Hkl, wl.seq, -1),
                      o=oh.view(B_, Hl, wl.seq, -1), lse=lh.view(B_, Hl, wl.seq))
            ra.ra_ulysses_a2a(oh, layout, N, 1, out=o_l)
            ra.ra_ulysses_a2a(lh, layout, N, 1, out=lse_l)
        else:
            ra.ra_fwd(plan, qx, kx, vx, o=o_l, lse=lse_l)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ra.ra_layout_perm(q, layout, N, out=ql)
        ra.ra_layout_perm(k, layout, N, out=kl)
        ra.ra_layout_perm(v, layout, N, out=vl)
        if ev is not None:
            ev[1].record(stream)
        forward(ql, kl, vl)
        if ev is not None:
            ev[2].record(stream)
        ra.ra_layout_perm(o_l, layout, N, inverse=True, out=o_n)
        ra.ra_layout_perm(lse_l, layout, N, inverse=True, out=lse_n)
        if ev is not None:
            ev[3].record(stream)

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    ra.ra_sync_status(plan)

    fwd_ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(fwd_ev[i])
        end.record(stream)
        barrier()
    ra.ra_sync_status(plan)
    total_ms = start.elapsed_time(end)
    fwd_ms = [e[1].elapsed_time(e[2]) for e in fwd_ev]
    perm_in_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in fwd_ev)
    perm_out_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in fwd_ev)
    total_ms, fwd_max = max_over_ranks([total_ms, max(fwd_ms)], pg, dev)
    ms_per_step = total_ms / args.steps
    flops = wl.flops()
    value = job_rate(world, flops, ms_per_step)

    # End to end through host buffers: every step copies its natural-order Q/K/V in
    # from pinned host memory and its O/LSE back out.  Steps are pipelined the way a
    # serving loop runs: step i+1's inputs travel (H2D stream) while step i computes,
    # and step i's outputs travel back (D2H stream) while step i+1 computes.  When one
    # (batch, key/value head) with its query heads is enough work to fill the GPU on
    # its own (the 1M-token workload), a step also runs in such units: unit j's inputs
    # arrive while unit j-1 computes and its outputs leave while unit j+1 computes, so
    # that only the first unit's inputs and the last unit's outputs wait on the host link.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        ho = torch.empty(o_n.shape, dtype=o_n.dtype, pin_memory=True)
        hl = torch.empty(lse_n.shape, dtype=lse_n.dtype, pin_memory=True)
        bufs = [(q, k, v, o_n, lse_n),
                (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o_n),
                 torch.empty_like(lse_n))]
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        G = wl.heads_q // wl.heads_kv
        if args.path == "fused" and wl.flops() / (wl.batch * wl.heads_kv) >= E2E_UNIT_FLOPS:
            uplan = ra.ra_plan(1, wl.seq, G, 1, wl.head_dim, N, layout, wl.causal, wl.dtype)
            units = [(b, g) for b in range(wl.batch) for g in range(wl.heads_kv)]
        else:
            uplan, units = None, [None]
        U = len(units)

        def qs(t, u):      # unit u's part of a [B, Hq, ...] tensor (a contiguous view)
            return t if u is None else t[u[0]:u[0] + 1, u[1] * G:(u[1] + 1) * G]

        def ks(t, u):      # ... of a [B, Hkv, ...] tensor
            return t if u is None else t[u[0]:u[0] + 1, u[1]:u[1] + 1]

        def unit_forward(u):
            if u is None:
                forward(ql, kl, vl)
            else:
                ra.ra_fwd(uplan, qs(ql, u), ks(kl, u), ks(vl, u), o=qs(o_l, u), lse=qs(lse_l, u))

        evs = lambda: [[torch.cuda.Event() for _ in range(U)] for _ in range(2)]
        h2d_done, in_free, comp_done, d2h_done = evs(), evs(), evs(), evs()

        def h2d(slot, j):
            u = units[j]
            bq, bk, bv = bufs[slot][:3]
            qs(bq, u).copy_(qs(hq, u), non_blocking=True)
            ks(bk, u).copy_(ks(hk, u), non_blocking=True)
            ks(bv, u).copy_(ks(hv, u), non_blocking=True)
            h2d_done[slot][j].record(h2d_s)

        def run_pipeline(n, ev=None):
            with torch.cuda.stream(h2d_s):
                for j in range(U):
                    h2d(0, j)
            for i in range(n):
                b = i % 2
                bq, bk, bv, bo, bl = bufs[b]
                for j, u in enumerate(units):
                    stream.wait_event(h2d_done[b][j])     # this unit's inputs have arrived
                    if ev is not None and j == 0:
                        ev[i][0].record(stream)
                    ra.ra_layout_perm(qs(bq, u), layout, N, out=qs(ql, u))
                    ra.ra_layout_perm(ks(bk, u), layout, N, out=ks(kl, u))
                    ra.ra_layout_perm(ks(bv, u), layout, N, out=ks(vl, u))
                    in_free[b][j].record(stream)
                    if ev is not None:
                        ev[i][1 + 2 * j].record(stream)
                    unit_forward(u)
                    if ev is not None:
                        ev[i][2 + 2 * j].record(stream)
                    if i >= 2:
                        stream.wait_event(d2h_done[b][j])  # step i-2's outputs have left this slot
                    ra.ra_layout_perm(qs(o_l, u), layout, N, inverse=True, out=qs(bo, u))
                    ra.ra_layout_perm(qs(lse_l, u), layout, N, inverse=True, out=qs(bl, u))
                    comp_done[b][j].record(stream)
                    if i + 1 < n:
                        with torch.cuda.stream(h2d_s):
                            if i >= 1:
                                h2d_s.wait_event(in_free[1 - b][j])  # step i-1 has read these inputs
                            h2d(1 - b, j)
                    with torch.cuda.stream(d2h_s):
                        d2h_s.wait_event(comp_done[b][j])
                        qs(ho, u).copy_(qs(bo, u), non_blocking=True)
                        qs(hl, u).copy_(qs(bl, u), non_blocking=True)
                        d2h_done[b][j].record(d2h_s)
                if ev is not None:
                    ev[i][-1].record(stream)
            stream.wait_stream(h2d_s)
            stream.wait_stream(d2h_s)

        run_pipeline(2)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 + 2 * U)] for _ in range(args.steps)]
        with ClockSampler(local) as e_clk:
            e0.record(stream)
            run_pipeline(args.steps, e_ev)
            e1.record(stream)
            barrier()
        e_ms = max_over_ranks([e0.elapsed_time(e1) / args.steps], pg, dev)[0]
        # where the end-to-end time goes, on this rank
        e_parts = {
            "units_per_step": U,
            "first_input_wait_ms": e0.elapsed_time(e_ev[0][0]),
            "step_ms": statistics.mean(x[0].elapsed_time(x[-1]) for x in e_ev),
            "fwd_ms": statistics.mean(sum(x[1 + 2 * j].elapsed_time(x[2 + 2 * j]) for j in range(U))
                                      for x in e_ev),
            "last_output_wait_ms": e_ev[-1][-1].elapsed_time(e1),
        }
        h2d_bytes = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h_bytes = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        e2e = {"value": job_rate(world, flops, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "breakdown": e_parts, "clocks": e_clk.summary(),
               "note": ("pinned host buffers, two device slots; H2D of step i+1 and D2H of step i-1 overlap "
                        "step i" + ("; each step runs as one ra_fwd per (batch, key/value head) with its "
                                    "query heads, whose copies overlap the neighbouring units" if U > 1 else ""))}
        ra.ra_sync_status(plan)
        if uplan is not None:
            ra.ra_sync_status(uplan)

    kernels = None
    if not args.no_kernels:
        bytes_in = 2 * sum(t.numel() * t.element_size() for t in (q, k, v))
        bytes_out = 2 * (o_n.numel() * o_n.element_size() + lse_n.numel() * lse_n.element_size())
        kernels = {
            "layout_perm_in": {"ms": perm_in_ms, "bytes": bytes_in, "GB/s": bytes_in / perm_in_ms / 1e6},
            "layout_perm_out": {"ms": perm_out_ms, "bytes": bytes_out, "GB/s": bytes_out / perm_out_ms / 1e6},
            "merge": merge_bandwidth(ra, torch, dev, stream),
        }

    backward = None
    if not args.no_bwd:
        backward = backward_report(ra, torch, plan, (ql, kl, vl), (o_l, lse_l), stream, flops, pg)

    ulysses = None
    if args.path == "ulysses":
        ulysses = ulysses_report(ra, torch, layout, N, (ql, kl, vl), (o_l, lse_l), (qh, kh, vh, oh, lh), stream)

    ring = None
    if args.path == "ring":
        ring = ring_driver_report(ra, torch, plan, N, (ql, kl, vl), (o_l, lse_l), (kbuf, vbuf),
                                  (o_parts, lse_parts), stream, statistics.mean(fwd_ms), flops)

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0

    peaks, src = load_peaks()
    fwd_mean = statistics.mean(fwd_ms)
    achieved = flops / (fwd_mean * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    clocks = clk.summary()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    at_clock = clock_peak(sms, clocks.get("sm_mhz"))
    traffic = measured_traffic(wl.name)
    full, part, skip = ra.ra_plan_tile_counts(plan)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(wl),
        "roofline": {"bound": "tensor", "kernel": "fwd_bf16_kernel", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{src} bf16_tflops_sustained",
                     "frac_of_burst": achieved / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                     "frac_at_clock": achieved / at_clock if at_clock else None,
                     "peak_at_clock": at_clock,
                     "peak_at_clock_note": (f"{sms} SMs x {TC_FLOP_PER_CLK_SM} dense bf16 FLOP per SM clock x the "
                                            "median SM clock sampled during the timed steps"),
                     "fwd_ms_mean": fwd_mean, "fwd_ms_median": statistics.median(fwd_ms),
                     "fwd_ms_all": fwd_ms,
                     "exp_rate": exp_rate(flops, wl.head_dim, fwd_mean * 1e-3, sms, clocks.get("sm_mhz"))},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "tile_counts": {"full": full.tolist(), "partial": part.tolist(), "skip": skip.tolist(),
                        "granularity": "128x128 per (batch, query head)"},
        "algorithmic_flops_per_step": flops,
        "kernels": kernels,
    }
    if backward is not None:
        peak_s = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        backward["frac_of_sustained"] = backward["TFLOP/s"] / peak_s
        line["backward"] = backward
    if ulysses is not None:
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        ulysses["in_frac_of_hbm"] = ulysses["exchange_in_GB/s"] / hbm
        ulysses["out_frac_of_hbm"] = ulysses["exchange_out_GB/s"] / hbm
        line["ulysses"] = ulysses
    if args.path == "ulysses":
        line["config"]["path"] = "ulysses: all-to-all to head shards, one-shard attention per device, all-to-all back"
        line["roofline"]["kernel"] = "fwd_bf16_kernel (one shard, batch N*B, H/N heads) + 5 exchanges"
        line["roofline"]["traffic"] = None
    if args.path == "allgather":
        line["config"]["path"] = "all-gather variant: K/V gathered into natural order, one step over all keys"
        line["roofline"]["kernel"] = "fwd_bf16_kernel (gathered K/V) + 2 gathers"
        line["roofline"]["traffic"] = None
    if ring is not None:
        line["ring_driver"] = ring
        line["config"]["path"] = "ring driver: per-step launches, K/V exchange on a second stream, merge"
        line["roofline"]["kernel"] = "fwd_bf16_kernel (one launch per ring step) + merge_kernel"
        line["roofline"]["traffic"] = None
    if kernels is not None:
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        for kv in kernels.values():
            kv["frac_of_hbm"] = kv["GB/s"] / hbm
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_record(wl, args.ref_rows)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


FWD_SOURCES = ("fwd_bf16_sm103.cu", "sm100_ptx.cuh", "ra_internal.h")


def fwd_source_digest():
    """sha256 over the forward kernel's sources (file name + bytes, in a fixed order)."""
    import hashlib
    h = hashlib.sha256()
    for name in FWD_SOURCES:
        h.update(name.encode())
        with open(os.path.join(ROOT, "context_ring_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload):
    """DRAM bytes per forward launch from the committed ncu summary of this workload.

    The summary carries `traffic_bytes_per_launch:` and `fwd_source_sha256:` lines; the
    figure is reported only while the kernel's sources still hash to the captured digest.
    """
    path = os.path.join(ROOT, "profiles", f"fwd_bf16_traffic_{workload}.md")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for ln in f:
            key, sep, val = ln.strip().strip("`").partition(":")
            if sep:
                rec[key.strip()] = val.strip()
    try:
        if rec.get("fwd_source_sha256") != fwd_source_digest():
            return None
        return int(rec["traffic_bytes_per_launch"])
    except (KeyError, ValueError, OSError):
        return None


def backward_report(ra, torch, plan, qkv, out, stream, flops, pg):
    """dQ, dK, dV of the timed forward's output for a random upstream gradient.

    One untimed call, then one timed call (CUDA events around ra_bwd: the
    preparation kernel and both tensor-core passes).  FLOPs are counted the usual
    way for attention gradients, 2.5x the forward's (five matrix products per
    (q, k) pair against two); the kernels execute 3.5x (scores and dP are
    recomputed in both passes).
    """
    ql, kl, vl = qkv
    o_l, lse_l = out
    g = torch.Generator(device=ql.device)
    g.manual_seed(4242)
    dout = torch.randn(ql.shape, generator=g, device=ql.device).to(ql.dtype)
    dq, dk, dv = torch.empty_like(ql), torch.empty_like(kl), torch.empty_like(vl)
    scratch = torch.empty(ra.ra_bwd_scratch_size(plan) // 4, dtype=torch.float32, device=ql.device)
    ra.ra_bwd(plan, ql, kl, vl, o_l, lse_l, dout, dq, dk, dv, scratch)
    ra.ra_sync_status(plan)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    a.record(stream)
    ra.ra_bwd(plan, ql, kl, vl, o_l, lse_l, dout, dq, dk, dv, scratch)
    b.record(stream)
    torch.cuda.synchronize()
    ra.ra_sync_status(plan)
    ms = max_over_ranks([a.elapsed_time(b)], pg, ql.device)[0]
    del dout, dq, dk, dv, scratch
    world = dist_env()[0]
    return {"ms": ms, "TFLOP/s": job_rate(world, 2.5 * flops, ms),
            "executed_TFLOP/s": job_rate(world, 3.5 * flops, ms),
            "flops_convention": "2.5x forward (dV, dP, dQ, dK and the recomputed scores)",
            "launches": 3}


def ulysses_report(ra, torch, layout, N, seq_side, out_side, head_side, stream, reps=3):
    """Bandwidth of Ulysses' exchanges: Q, K, V to head shards, then O and the LSE back."""
    ql, kl, vl = seq_side
    o_l, lse_l = out_side
    qh, kh, vh, oh, lh = head_side

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def ex_in():
        for src, dst in ((ql, qh), (kl, kh), (vl, vh)):
            ra.ra_ulysses_a2a(src, layout, N, 0, out=dst)

    def ex_out():
        ra.ra_ulysses_a2a(oh, layout, N, 1, out=o_l)
        ra.ra_ulysses_a2a(lh, layout, N, 1, out=lse_l)

    t_in, t_out = timed(ex_in), timed(ex_out)
    b_in = 2 * sum(t.numel() * t.element_size() for t in (ql, kl, vl))
    b_out = 2 * (o_l.numel() * o_l.element_size() + lse_l.numel() * lse_l.element_size())
    return {"exchange_in_ms": t_in, "exchange_in_GB/s": b_in / t_in / 1e6,
            "exchange_out_ms": t_out, "exchange_out_GB/s": b_out / t_out / 1e6}


def ring_driver_report(ra, torch, plan, N, qkv, out, bufs, parts, stream, driver_ms, flops):
    """Where the explicit ring driver's time goes: its pieces timed one by one.

    steps_only: the N per-step launches back to back (K/V read from one buffer;
    the data does not change the work).  rotations_only: the N-1 exchanges back to
    back.  merge_only: the final merge.  With the exchange hidden behind compute the
    driver takes about steps_only + merge_only.
    """
    ql, kl, vl = qkv
    o_l, lse_l = out
    kbuf, vbuf = bufs
    o_parts, lse_parts = parts

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def steps():
        for t in range(N):
            ra.ra_fwd_step(plan, t, ql, kl, vl, o_part=o_parts[t], lse_part=lse_parts[t])

    def rotations():
        src_k, src_v = kl, vl
        for t in range(N - 1):
            ra.ra_ring_rotate(plan, src_k, src_v, kbuf[t % 2], vbuf[t % 2])
            src_k, src_v = kbuf[t % 2], vbuf[t % 2]

    def merge():
        ra.ra_merge_partials(o_parts, lse_parts, o=o_l, lse=lse_l)

    steps_ms, rot_ms, merge_ms = timed(steps), timed(rotations), timed(merge)
    fused_ms = timed(lambda: ra.ra_fwd(plan, ql, kl, vl, o=o_l, lse=lse_l))
    ra.ra_sync_status(plan)
    rot_bytes = 2 * (N - 1) * 2 * kl.numel() * kl.element_size()   # K and V, read + write
    serial = steps_ms + rot_ms + merge_ms
    return {
        "driver_ms": driver_ms, "driver_TFLOP/s": flops / (driver_ms * 1e-3) / 1e12,
        "steps_only_ms": steps_ms, "rotations_only_ms": rot_ms, "merge_only_ms": merge_ms,
        "rotation_GB/s": rot_bytes / rot_ms / 1e6 if rot_ms > 0 else None,
        "serial_sum_ms": serial,
        "rotation_hidden_frac": (serial - driver_ms) / rot_ms if rot_ms > 0 else None,
        "fused_ra_fwd_ms": fused_ms,
    }


def merge_bandwidth(ra, torch, dev, stream, n_parts=8, rows=1 << 20, d=128, reps=5):
    """ra_merge_partials on 8 synthetic float32 parts of 1M rows x 128 -> bf16 (HBM-bound)."""
    g = torch.Generator(device=dev).manual_seed(77)
    o_parts = torch.randn((n_parts, rows, d), generator=g, device=dev)
    lse_parts = torch.randn((n_parts, rows), generator=g, device=dev)
    o = torch.empty((rows, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    for _ in range(3):
        ra.ra_merge_partials(o_parts, lse_parts, o=o, lse=lse)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        ra.ra_merge_partials(o_parts, lse_parts, o=o, lse=lse)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    nbytes = n_parts * rows * (4 * d + 4) + rows * (2 * d + 4)
    return {"ms": ms, "bytes": nbytes, "GB/s": nbytes / ms / 1e6,
            "shape": f"{n_parts} parts x {rows} rows x {d} f32 -> bf16 (working set > L2)"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="zigzag_1m_n8")
    ap.add_argument("--layout", default=None, help="override the workload's layout")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernels", action="store_true", help="skip the permute/merge bandwidth lines")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--path", default="fused", choices=["fused", "ring", "allgather", "ulysses"],
                    help="fused: one ra_fwd launch per step; ring: the explicit ring driver "
                         "(per-step launches, K/V exchange on a second stream, merge); allgather: "
                         "K/V gathered into natural order, then one step over all keys; ulysses: all-to-all to head "
                         "shards, one-shard attention per device, all-to-all back")
    args = ap.parse_args()
    from context_ring_attention_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    if args.layout:
        import dataclasses
        wl = dataclasses.replace(wl, layouts=(args.layout,))
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
