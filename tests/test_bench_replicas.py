"""Host logic of the multi-replica bench (N > 1), on CPU with gloo.

The decode has no exchange step, so N GPUs run N independent replicas; the
bench's only cross-rank logic is the max-over-ranks time and the whole-job
rate.  Two gloo ranks check exactly that."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_max(1.0 + rank * 0.5)  # rank 1 is the slow one
    rate = bench.aggregate_rate(1000.0, world, t)
    w, r, _ = bench.dist_env()
    q.put((rank, t, rate, w, r))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_rate():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, rate, w, r in res:
        assert t == pytest.approx(1.5)          # max over ranks
        assert rate == pytest.approx(2 * 1000.0 / 1.5)
        assert (w, r) == (2, rank)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.25) == 3.25
    assert bench.aggregate_rate(10.0, 1, 2.0) == 5.0


def test_gpus_2_starts_two_ranks_on_cpu():
    """bench.py --gpus 2 outside torchrun starts two ranks itself; with
    --launch-check they only run the cross-rank reduction over gloo."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--launch-check"], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
    d = json.loads(line)["launch_check"]
    assert d["gpus"] == 2 and d["world"] == 2
    assert sorted(x["rank"] for x in d["ranks"]) == [0, 1]
    for x in d["ranks"]:
        assert x["max_s"] == pytest.approx(1.5)
        assert x["rate"] == pytest.approx(2 * 1000.0 / 1.5)


def test_gpus_mismatch_is_refused():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--launch-check"], capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
