"""The multi-process host logic of bench.py on the CPU (gloo, world size 2):
the barrier and the max over ranks that the timing takes, and the reference
arm under torchrun, where rank 0 alone runs and prints one JSON line and the
other rank exits 0 without work.  The GPU path itself runs replicas only (one
process per GPU, no collective on the data path), so these are its only
cross-process steps."""
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


def _worker(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(world)
    try:
        assert d.world == world and d.rank == rank
        d.barrier()
        m = d.max(float(10 * rank + 1))
        d.barrier()
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(repr(m))
    finally:
        d.close()


def test_barrier_and_max_over_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"r{r}.txt").read_text()) == 11.0


def test_reference_arm_two_ranks_prints_once():
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--cpu-rows", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2
    assert res["value"] > 0 and res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"]["h2d_bytes_per_step"] == 0
