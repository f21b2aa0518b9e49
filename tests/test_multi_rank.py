"""The N > 1 path of bench.py on CPU: two ranks over gloo (no GPU).

bench.py runs one replica per GPU with a host-side gloo group used only for the
barrier around the timed region and the max-over-ranks of the timed duration;
the reference arm prints from rank 0 alone.  Both are exercised here with
world size 2, the rendezvous on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, local, ws, dist = bench._dist()
    try:
        bench._barrier(dist)
        got = bench._max_over_ranks(10.0 * (rank + 1), dist)  # each rank's "duration"
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"rank": r, "local": local, "ws": ws, "max": got}, f)
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1] and all(x["ws"] == 2 for x in res)
    assert all(x["max"] == 20.0 for x in res)  # every rank sees the slowest rank's time
    del torch


def test_reference_arm_prints_once_from_rank_zero():
    pytest.importorskip("torch")
    env = dict(os.environ, OMP_NUM_THREADS="1")
    for attempt in range(3):
        # the port is free when chosen but is bound again only by the launcher: another process may take
        # it in between, so a rendezvous that fails on its address is retried on a new port
        port = _free_port()
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
               "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
               "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "tiny", "--cpu-rows", "2000",
               "--cpu-trees", "1"]
        p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
        if p.returncode == 0 or not any(m in p.stderr for m in ("EADDRINUSE", "Address already in use",
                                                                 "DistNetworkError")):
            break
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(ln) for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
