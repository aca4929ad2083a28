"""The multi-rank plumbing of bench.py on CPU (gloo, world size 2, 127.0.0.1): the path
shards with no data exchange, so N GPUs run N replicas; what the ranks share is the
barrier around the timed region and the max over ranks of the time, from which the
whole-job value is all ranks' bytes over the slowest rank's time."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(None)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # rank k "took" (k + 1) ms for its bytes: the job's time is the slowest rank's
    ms = bench.max_over_ranks(float(rank + 1), w)
    step_bytes = 1000.0
    value = w * step_bytes / (ms * 1e-3)
    out[rank] = (ms, value)
    bench.barrier(w)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 2 * 1000.0 / 2e-3)


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """--impl reference launched as the driver launches N > 1: rank 0 alone times the oracle
    and prints one JSON line; the other rank exits 0 without work."""
    import oracle
    oracle.build()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
