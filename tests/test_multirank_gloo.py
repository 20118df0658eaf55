"""Multi-rank host logic on CPU (gloo, world size 2): the whole-job aggregation used by
bench.py under torchrun, and the data-parallel split of the core (every (b, q, m) output
is independent, so query shards computed separately reproduce the unsharded result with
no exchange on the data path; the gather below exists only to check that)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        import workloads
        # 1) aggregation: slowest rank's time, samples summed over ranks
        value, t_max = bench.aggregate(1.0 + rank, 1000 * (rank + 1), 10, world)
        # 2) query-sharded oracle forward equals the unsharded one
        inp = workloads.random_problem(2, [(9, 7), (4, 3)], B=2, Nq=41, M=3, D=8, P=4,
                                       seed=3)
        a, b = workloads.shard_range(41, rank, world)
        part = oracle.forward(2, inp["value"], inp["spatial_shapes"],
                              inp["level_start_index"], inp["sampling_locations"][:, a:b],
                              inp["attention_weights"][:, a:b])
        parts = [None] * world
        dist.all_gather_object(parts, (a, b, part))
        if rank == 0:
            full = oracle.forward(2, inp["value"], inp["spatial_shapes"],
                                  inp["level_start_index"], inp["sampling_locations"],
                                  inp["attention_weights"])
            glued = np.concatenate([p[2] for p in sorted(parts, key=lambda t: t[0])], axis=1)
            q.put(("ok", value, t_max, bool(np.array_equal(glued, full))))
    except Exception as e:  # report to the parent instead of hanging the test
        q.put(("error", repr(e)))
        raise
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("gloo worker hung")
    res = q.get(timeout=10)
    assert res[0] == "ok", res
    _, value, t_max, equal = res
    assert t_max == 2.0
    assert value == pytest.approx((1000 + 2000) * 10 / 2.0)
    assert equal
    assert all(p.exitcode == 0 for p in procs)
