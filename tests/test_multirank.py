"""The benchmark's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

The path partitions into independent (group, KV head) units with no exchange step,
so ranks only differ in their chunk (seed) and meet only to take the slowest
rank's time.  These tests run that host logic without a GPU.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from sparse_selected_cell_gb300 import gen
        t = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")     # rank r "took" 10 + 5r ms
        w = gen.make(bench.CONFIG_ID, seed=bench.rank_seed(rank), n_q=64)
        digest = int(np.bitwise_xor.reduce(w.sel[:, :16].ravel().astype(np.int64)) + 1000 * int(w.sel_count.sum()))
        out.put((rank, t, bench.rank_seed(rank), w.sel.shape, digest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_chunks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, s0, sh0, d0), (r1, t1, s1, sh1, d1) = res
    assert (r0, r1) == (0, 1)
    assert t0 == t1 == 15.0                  # both ranks see the max over ranks
    assert s0 != s1 and sh0 == sh1           # independent chunks of one shape
    assert d0 != d1


def test_single_process_is_identity_and_job_value():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    # 2 ranks x 393,216 rows x 10 steps in 20 ms (slowest rank)
    assert bench.job_rows_per_s(2, 393216, 10, 20.0) == pytest.approx(2 * 393216 * 10 / 0.02)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(steps=1, warmup=3, gpus=2))()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
