"""Host logic of `bench.py --gpus N` (replicas only: one process per GPU and
no data-path collective), run as two gloo ranks on the CPU: the barrier, the
max over ranks that sets the timed duration, the whole-job rate, and the
reference arm printing from rank 0 alone."""
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ranks = bench.Ranks(dist, "cpu")
        ranks.barrier()
        # each rank "took" a different time; the job took the longest
        t = ranks.max(1.0 + 0.25 * rank)
        rate = bench.whole_job_rate(1000.0, world, t)
        ranks.barrier()
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, rate in res:
        assert t == pytest.approx(1.25)            # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 / 1.25)


def test_single_process_ranks_are_identity():
    r = bench.Ranks(None)
    r.barrier()
    assert r.max(3.5) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_prints_from_rank_zero_only(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"])
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the reference arm names the GPU arm's metric and workload
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["config"] == bench.headline_config(line["n_gpus"])


def test_q6k_cpu_baseline_times_the_oracle():
    r = bench.run_cpu_q6k(0.2)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] >= 1
    assert "Q6_K GEMV 4096x4096" in r["sample"]


def test_q4_0_cpu_baseline_times_the_oracle():
    r = bench.run_cpu_q4_0(0.1)
    assert r["kind"] == "oracle" and r["cores"] == 1 and r["us_per_gemv"] > 0
    assert "Q4_0 GEMV 512x1024" in r["sample"]
