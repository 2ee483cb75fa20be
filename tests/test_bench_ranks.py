"""bench.py's multi-rank host path on CPU: two ranks under torchrun with the
gloo backend (the reference arm runs the oracle on host cores only). Rank 0
prints exactly one JSON line; the other rank exits 0 without output."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_two_ranks_gloo():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29517", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--ref-step-seconds", "0.3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    # rank-dependent timings; every rank must get the element-wise maximum
    vals = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]
    got = bench.max_over_ranks(vals, dist, "cpu")
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_two_ranks_gloo():
    # the repo arm's reduction of step times (the all-reduce MAX that makes
    # the slowest rank decide the timing), on two CPU ranks with gloo
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=5) for _ in range(2))
    assert results[0] == results[1] == [2.0, 10.0, 1.0]


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 1.5]) == [3.0, 1.5]


def test_reference_and_headline_share_the_config():
    sys.path.insert(0, ROOT)
    import bench
    from pass_attention_gb300 import workloads
    cfg = bench.headline_config(workloads.SOFTMAX_32K)
    src = open(os.path.join(ROOT, "bench.py")).read()
    # both JSON lines take their config from the same function
    assert src.count('"config": headline_config(w)') == 2
    assert cfg["rows"] == 32768 and cfg["cols"] == 8192
