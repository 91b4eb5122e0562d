"""Multi-process path of bench.py on CPU: with N replicas (one process per
GPU, no data exchange), every rank times its own layer and the job's time is
the slowest rank's, reduced over gloo.  Run here with world size 2."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup(None)
    elapsed_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    slowest = bench.reduce_max(elapsed_ms, w)
    bench.barrier(w)
    tokens_per_rank, steps = 16384, 4
    value = w * tokens_per_rank * steps / (slowest / 1e3)
    q.put((r, local, w, slowest, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[2] == 2 for o in out)
    assert all(o[3] == 20.0 for o in out)                    # max over ranks
    assert all(o[4] == pytest.approx(2 * 16384 * 4 / 0.020) for o in out)


def _ref_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import contextlib
    import io
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main_args(["--impl", "reference", "--config", "0", "--steps", "1",
                              "--warmup", "0", "--ref-tokens", "8"])
    q.put((rank, rc, buf.getvalue()))


def test_reference_arm_prints_on_rank_0_only():
    """bench.py --impl reference under two ranks: rank 0 times the oracle and
    prints one JSON line; rank 1 exits 0 without work."""
    import json
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rc0, text0), (r1, rc1, text1) = out
    assert rc0 == 0 and rc1 == 0 and text1 == ""
    lines = [ln for ln in text0.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
