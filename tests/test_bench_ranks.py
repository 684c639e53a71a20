"""CPU checks of bench.py's multi-rank plumbing (no GPU): two gloo ranks on
127.0.0.1 set up through the same torchrun environment the driver uses.  The
forward pass runs one replica per rank (no data-path collective), so what a
rank shares is the barrier around the timed region and the maximum of the
elapsed times; the reference arm runs on rank 0 alone."""

import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    world, r, local = bench.dist_setup()
    bench.barrier(world)
    # each rank's "elapsed time"; every rank must get the largest
    got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    backend = dist.get_backend()
    bench.barrier(world)
    dist.destroy_process_group()
    out.put((rank, world, r, local, got, backend))


def test_two_gloo_ranks_share_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 0, 0, 15.0, "gloo"), (1, 2, 1, 1, 15.0, "gloo")]


def test_reference_arm_under_torchrun_prints_from_rank_zero_only():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--workload", "n129_d32_f16_causal", "--steps", "2", "--warmup", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["config"]["parallelism"] == "replicas x2" and d["scaling"] == "weak"
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
