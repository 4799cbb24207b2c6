"""The replica path of bench.py under several ranks, on the CPU with gloo:
the timing taken is each value's maximum over the ranks and the job's rate
counts every rank's units.  Ranks are separate processes (spawn)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], world)
        out[rank] = got
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_whole_job_rate(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == [10.0 + world - 1, 5.0]
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_rate(96, world, 0.5) == 96 * world / 0.5


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched as the driver launches multi-GPU
    runs (torchrun, 127.0.0.1): rank 0 prints one JSON line, rank 1 exits 0."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_cpu_baseline_falls_back_to_one_process(monkeypatch):
    """When the oracle's process pool cannot start, the CPU baseline times one
    process and reports one core instead of failing the benchmark."""
    import bench
    monkeypatch.setattr(bench, "_spawn_oracle_pool", lambda workers: None)
    r = bench.cpu_baseline(seconds=0.0)
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0
    assert "one process" in r["sample"]
