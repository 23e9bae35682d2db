"""The bench's whole-job reduction over ranks, run as two gloo ranks on the
CPU: the time is the slowest rank's, the bytes are summed."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, nb = bench.reduce_over_ranks(dist, 10.0 + 5.0 * rank, 1000 * (rank + 1))
        out[rank] = torch.tensor([ms, nb], dtype=torch.float64)
    finally:
        dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    world = 2
    out = torch.zeros((world, 2), dtype=torch.float64).share_memory_()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        assert out[r, 0].item() == 15.0          # max over ranks
        assert out[r, 1].item() == 3000.0        # sum over ranks


def test_reduce_single_rank():
    assert bench.reduce_over_ranks(None, 7.5, 42) == (7.5, 42.0)


def test_reference_arm_line_keys():
    """`bench.py --impl reference` (the oracle timed on the host cores)
    prints one JSON line with the contract's keys, the reference arm's
    extras, and no GPU in the loop."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] >= 3
    assert d["config"]["workload"] == "moe_decode_b1"
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
