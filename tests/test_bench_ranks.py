"""bench.py's multi-rank logic on CPU: two gloo ranks exchange their timings
(max over ranks), the whole-job value counts every rank's weights, and the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r = bench.Ranks(backend_gpu=False)
    try:
        mx = r.max(1.5 if rank == 0 else 2.5)     # the slower rank sets the job time
        sm = r.sum(float(rank + 1))
        r.barrier()
        value = bench.job_value(weights_per_rank=1000, world=r.world, max_seconds=mx, steps=4)
        q.put((rank, r.world, mx, sm, value))
    finally:
        r.close()


def test_two_gloo_ranks_agree_on_max_time_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, world, mx, sm, value in got:
        assert world == 2
        assert mx == 2.5 and sm == 3.0
        assert value == pytest.approx(1000 * 2 * 4 / 2.5)


def _reference_rank(rank, port, q):
    os.environ.update({"WORLD_SIZE": "2", "RANK": str(rank), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import contextlib
    import io
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        if rank != 0:
            bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1",
                                                  "--warmup", "0"]))
    q.put((rank, buf.getvalue()))


def test_reference_arm_other_ranks_do_no_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_reference_rank, args=(1, _free_port(), q))
    p.start()
    p.join(timeout=60)
    assert p.exitcode == 0
    rank, out = q.get(timeout=10)
    assert rank == 1 and out == ""
