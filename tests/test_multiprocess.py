"""The N > 1 host logic of bench.py on CPU with the gloo backend, two ranks.

The path shards into independent chains, so N GPUs run N replicas with no
collective on the data path; what needs checking is the launch contract:
rendezvous, the barrier around the timed region, the max-over-ranks time and
that only rank 0 prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    import torch.distributed as dist
    args = argparse.Namespace(impl="reference")
    got_ws, got_rank, _ = bench.dist_setup(args)
    assert dist.get_backend() == "gloo"
    bench.barrier(got_ws)
    # each rank's time differs; every rank must see the maximum
    m = bench.max_over_ranks(1.5 + got_rank, got_ws)
    with open(os.path.join(out_dir, f"rank{got_rank}.json"), "w") as f:
        json.dump({"ws": got_ws, "rank": got_rank, "max": m}, f)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo(tmp_path):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, free_port(), str(tmp_path)), nprocs=ws, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["ws"] == ws and r["max"] == 2.5 for r in res)


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched like the driver's N > 1 runs: rank 0 alone runs the oracle
    and prints one JSON line; the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "gdn_fp32_t1024_h2_d64_r4"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
