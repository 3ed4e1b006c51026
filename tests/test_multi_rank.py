"""The benchmark's multi-GPU path is replicas: each rank runs its own sequences, and the
job's time is the slowest rank's. Its host logic runs here as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    assert bench.dist_info() == (ws, rank, rank)
    ms = 10.0 + 3.0 * rank                      # rank 1 is the slower replica
    t = bench.max_over_ranks(ms, ws, device="cpu")
    out.put((rank, t, bench.job_rate(ws, 1, 100, t / 1e3)))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, t, rate in res:
        assert t == 13.0                          # both ranks see the slowest rank's time
        assert rate == pytest.approx(2 * 100 / 0.013)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1"])
    bench.main()
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_contract_line_on_the_tiny_workload(monkeypatch, capsys):
    import json
    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                                     "--warmup", "1"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["unit"] == "steps/s"
