"""The benchmark's N > 1 path on CPU: world size 2 over gloo (127.0.0.1).

Under torchrun every rank runs an independent replica of the workload (the
(sequence, head) units need no exchange), so the only collectives are the
barrier and the max over ranks of the timed interval; the whole-job value is
every rank's tokens over the slowest rank's time.  The reference arm prints
on rank 0 only.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        # each rank timed its own replica; rank 1 was slower
        ms = 10.0 + 5.0 * rank
        dist.barrier()
        mx = bench.max_over_ranks(ms, world, device="cpu")
        value = bench.aggregate_value(tokens_per_step_per_rank=1000, steps=4, world=world, max_ms=mx)
        with open(f"{result_path}.{rank}", "w") as f:
            json.dump({"max_ms": mx, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_over_gloo(tmp_path):
    world, port = 2, _free_port()
    out = str(tmp_path / "res")
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    res = [json.load(open(f"{out}.{r}")) for r in range(world)]
    for r in res:
        assert r["max_ms"] == 15.0                         # the slowest rank's time, on every rank
        assert r["value"] == pytest.approx(1000 * 4 * 2 / 0.015)   # all ranks' tokens / slowest time


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.aggregate_value(1000, 4, 1, 10.0) == pytest.approx(400_000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "fp32_n1024"])
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""                            # other ranks exit without work
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
