"""The N > 1 path of bench.py on the host, with world size 2 over gloo (no GPU).

bench.py runs one rank per GPU. Each rank times its own batch (weak scaling, no
collective in the data path); the ranks meet only at the timing barrier and in the
max-over-ranks / sum-over-ranks reduction of the result. These tests run those parts
as two CPU processes: the reduction and barrier directly, and the reference arm end to
end under torchrun, where rank 0 alone times the oracle and prints one JSON line.
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r took 1.5 + r ms for 10 + r units of work
        t, v = bench.reduce_max_sum(world, 1.5 + rank, 10.0 + rank, "cpu")
        out.put((rank, t, v))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_reduce_takes_the_slowest_rank_and_all_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(world))
    # every rank sees the same result: the max time and the summed work
    assert got == [(0, 2.5, 21.0), (1, 2.5, 21.0)]


def test_single_rank_reduce_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_sum(1, 3.0, 7.0, "cpu") == (3.0, 7.0)


def test_reference_arm_under_torchrun_two_ranks():
    """torchrun with two ranks: rank 0 prints one JSON line for the reference arm and the
    other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "qwen3-4b"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2
    assert res["value"] > 0 and res["steps"] == 1 and res["warmup"] == 0
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["value"] == res["value"]
    assert res["e2e"] == {"value": res["value"], "unit": res["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
