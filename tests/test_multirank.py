"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas only, no
data-path collective; the one collective is the max over ranks of the
timings)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w, lr = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    # rank r "measured" steps of (r + 1) ms: the job time is the slowest rank's
    got = bench.max_over_ranks([float(r + 1)] * 5, "cpu", w)
    thr = bench.replica_throughput(got, w)
    # each replica draws its own inputs (seed = rank)
    from workloads import make_inputs, small_config
    inp = make_inputs(small_config("c0", vocab=64), seed=r)
    dist.destroy_process_group()
    q.put((r, w, lr, got, thr, float(inp["q_bits"][0, 0, 0])))


def test_two_rank_max_over_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert [x[2] for x in res] == [0, 1]
    assert all(x[3] == pytest.approx(2.0) for x in res)       # max over ranks
    assert all(x[4] == pytest.approx(1000.0) for x in res)    # 2 replicas / 2 ms
    assert res[0][5] != res[1][5]                             # independent replica inputs


def test_single_rank_statistics():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    xs = [5.0, 1.0, 2.0, 3.0, 4.0, 100.0]
    assert bench.max_over_ranks(xs, "cpu", 1) == pytest.approx(3.5)  # median: one outlier moves it not
    assert bench.max_over_ranks(xs, "cpu", 1, "mean") == pytest.approx(115.0 / 6)
    st = bench.step_stats(list(range(1, 12)))
    assert (st["p10"], st["median"], st["p90"]) == (2, 6, 10)
    assert bench.replica_throughput(2.0, 1) == pytest.approx(500.0)
