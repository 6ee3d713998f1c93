"""The multi-rank benchmark path on the CPU (gloo, world size 2).

The block shards by tokens with no exchange on the data path ("replicas only"): every rank
runs its own batch; the only collectives are the timing barrier and the max-over-ranks of
the elapsed time.  Run here with the reference arm (the CPU oracle), which uses the same
launch, rank handling and reduction as the GPU arm."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench.dist_init()
    assert (ws, r) == (2, rank) and dist.get_backend() == "gloo"
    bench.barrier(ws)
    out[rank] = bench.allreduce_max(1.5 + rank, ws)
    dist.destroy_process_group()


def test_allreduce_max_over_two_gloo_ranks():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_replicas_take_disjoint_token_rows():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    w = workloads.Workload("rep", T=5, D=128, L=128, E=4, I=128, k=2)
    long_batch = workloads.x_tensor(w.with_tokens(10))
    assert torch.equal(bench.replica_x(w, 0), long_batch[:5])
    assert torch.equal(bench.replica_x(w, 1), long_batch[5:])


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny_fp32", "--steps", "2",
           "--warmup", "1", "--cpu-tokens", "8"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout            # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
