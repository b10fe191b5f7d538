"""The N>1 bench path on the host: world-size-2 gloo ranks, no GPU.

Each rank runs an independent replica (the layer has no cross-GPU exchange);
bench.py only needs a barrier and the max of the ranks' times, and the
reference arm runs on rank 0 alone.
"""
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


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.world_barrier(world)
    slowest = bench.world_max(10.0 * (rank + 1), world, "cpu")
    q.put((rank, slowest, bench.job_tokens_per_s(1000, world, 4, slowest)))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree on the slowest time; throughput counts both ranks' tokens
    assert [o[1] for o in out] == [20.0, 20.0]
    assert out[0][2] == pytest.approx(1000 * 2 * 4 / 0.020)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 1:
        assert lines == []
    else:
        line = json.loads(lines[-1])
        assert line["impl"] == "reference" and line["value"] > 0
        assert line["cpu_baseline"]["kind"] == "oracle"
        assert line["e2e"]["h2d_bytes_per_step"] == 0
