"""The bench's multi-process logic on CPU ranks (gloo, world size 2).

On GPUs the bench runs one replica per GPU (the path needs no collective: one GPU
plays all N ring devices), times every rank, and reports the job's rate from the
slowest rank.  Here two gloo ranks check that logic: the rank environment, the
element-wise maximum over ranks, the whole-job rate, and that only rank 0 runs the
reference arm.
"""

import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    # rank r "measured" 10 + r ms for the step and 5 - r ms for the kernel
    step_ms, kern_ms = bench.max_over_ranks([10.0 + r, 5.0 - r], dist, "cpu")
    dist.barrier()
    rate = bench.job_rate(w, 2e12, step_ms)
    # the reference arm runs on rank 0 only; other ranks return 0 without work
    class A:
        warmup, steps, ref_rows = 0, 0, 1
    ref = bench.run_reference(A, None) if r != 0 else None
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"w": w, "r": r, "local": local, "step": step_ms, "kern": kern_ms, "rate": rate, "ref": ref}, f)
    dist.destroy_process_group()


def test_two_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert (g["w"], g["r"], g["local"]) == (2, r, r)
        assert g["step"] == 11.0 and g["kern"] == 5.0        # the slowest rank's times
        assert abs(g["rate"] - 2 * 2e12 / 11e-3 / 1e12) < 1e-9
    assert got[1]["ref"] == 0


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks([3, 4], None, "cpu") == [3.0, 4.0]
    assert bench.job_rate(1, 1e12, 1000.0) == pytest.approx(1.0)
