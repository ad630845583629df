"""Multi-rank host logic of the benchmark (replica ranks, weak scaling) on CPU
with the gloo backend, world size 2."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r+1) * 10 ms for its K steps: the job is timed by the slowest
    t = bench.reduce_max_over_ranks((rank + 1) * 10.0, dist, "cpu")
    v = bench.job_gbps(302_000_000, world, t / 1e3 / 5)
    dist.barrier()
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == 20.0
        assert v == pytest.approx(2 * 302_000_000 / (20.0 / 1e3 / 5) / 1e9)


def test_single_rank_identity():
    import bench
    assert bench.reduce_max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_gbps(1_000_000_000, 1, 0.5) == 2.0


def test_bench_launches_its_own_ranks_for_gpus_n():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (here in the
    host-only --dry mode, gloo): one line from rank 0 with n_gpus = 2 and the
    slowest rank's time."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR",
                                                             "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry", "--steps", "3"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["dry_run"] is True and d["measured"] is False
    assert d["max_rank_ms_per_step"] == 2.0 and d["steps"] == 3


def test_bench_refuses_a_world_size_other_than_gpus():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry"], cwd=root, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "--gpus 2" in r.stderr
