"""The multi-process side of bench.py on CPU: two gloo ranks (world size 2).
Each GPU runs its own replica of the chain (no collective on the data path),
so what crosses ranks is the timing: the step time is the slowest rank's,
every rank gets it, and the whole-job throughput counts every replica.  The
reference arm runs on rank 0 only; other ranks exit 0 without output."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank step times 1.5 ms and 3.0 ms: both ranks see the slower one
        ms = bench.max_over_ranks(1.5 * (rank + 1), world)
        value = bench.job_gbps(world, 3_000_000, ms)
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.reference_arm(SimpleNamespace(steps=1, warmup=0)) if rank != 0 else None
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value, "ref_rc": rc, "ref_out": buf.getvalue()}, f)


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == pytest.approx(3.0)
        # 2 replicas x 3 MB per step in 3 ms = 2 GB/s for the whole job
        assert r["value"] == pytest.approx(2.0)
    assert res[1]["ref_rc"] == 0 and res[1]["ref_out"] == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_gbps(1, 1_000_000, 1.0) == pytest.approx(1.0)
