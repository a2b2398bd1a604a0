"""Multi-process host logic on CPU, world size 2 over gloo (127.0.0.1):
  - the bench's barrier and max-over-ranks reduction of the timed region (every rank
    reports the slowest rank's time, which the whole-job value divides by);
  - the reference arm launched the way the driver launches N > 1 runs (torchrun): rank 0
    alone runs and prints one JSON line, the other rank exits 0 without work.
The GPU arm of N > 1 runs independent replicas with no data-path collective, so these
are the only multi-rank steps it takes."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_env()[:2] == (ws, rank)
        bench.barrier(ws)
        slowest = bench.barrier_max(10.0 * (rank + 1), ws, "cpu")
        bench.barrier(ws)
        with open(os.path.join(out, f"rank{rank}"), "w") as f:
            f.write(repr(slowest))
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_two_gloo_ranks(tmp_path):
    mp.start_processes(_rank, args=(2, free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    assert [float((tmp_path / f"rank{r}").read_text()) for r in range(2)] == [20.0, 20.0]


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--config", "0", "--steps", "2", "--warmup", "3",
           "--ref-seconds", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
