"""The benchmark's multi-rank plumbing on the host: two gloo ranks on CPU.

The path shards into independent replicas (one process per GPU, no data-path
collective); what the ranks share is the barrier around the timed region and
the reductions that turn per-rank numbers into the whole-job figure: the
slowest rank's time and the bytes all ranks moved.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_CODE = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
world, rank, local = bench.dist_env()
d = bench.init_dist(world)
bench.barrier(d)
out = {
    "rank": rank, "world": world, "backend": d.get_backend(),
    "max": bench.allmax(d, 1.0 + rank),
    "sum": bench.allsum(d, 10.0 * (rank + 1)),
    # rank r moved (r + 1) GB in (100 + 50 r) ms: 3 GB over the slowest 150 ms
    "rate": bench.aggregate_rate(d, 1e9 * (rank + 1), 100.0 + 50.0 * rank),
}
bench.barrier(d)
print(json.dumps(out))
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return env


def test_two_gloo_ranks_reduce_like_the_benchmark():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_CODE, ROOT], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in (0, 1)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2 and o["backend"] == "gloo"
        assert o["max"] == 2.0
        assert o["sum"] == 30.0
        rate, t_max = o["rate"]
        assert t_max == 150.0
        assert abs(rate - 3.0 / 0.150) < 1e-9  # GB/s over all ranks


def test_reference_arm_only_rank0_reports():
    # rank 1 of a two-rank launch exits at once without work or output
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=_env(1, 2, _free_port()), capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
