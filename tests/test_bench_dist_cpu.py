"""bench.py's multi-process host logic on CPU ranks (gloo): the timing is the
maximum over ranks, and under torchrun only rank 0 of the reference arm
prints its line (the path is replicas only: no data-path collective)."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE="2")
    sys.path.insert(0, ROOT)
    import torch
    import bench
    dist, r, ws = bench.dist_setup()
    assert (r, ws) == (rank, 2) and dist is not None
    got = bench.max_over_ranks(dist, 1.5 + 10.0 * rank, torch.device("cpu"))
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump(dict(rank=rank, max=got), f)
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    mp.spawn(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert [x["max"] for x in res] == [11.5, 11.5]


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-rows", "64"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
