"""Multi-rank host logic of bench.py on CPU: two gloo ranks as replicas.

The decode / store / append path shards by sequence with no data exchange; ranks only meet at
barriers and in the max-over-ranks reduction of the timed total.  These tests run that plumbing
with world size 2 on the gloo backend (no GPU): each rank builds its own seeded workload, the
slowest rank's time is what every rank reports, and the whole-job value counts every rank's bytes.
"""
import argparse
import hashlib
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_worker(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    from workloads import config_case

    r, w, local = bench.dist_setup(argparse.Namespace(impl="reference"))   # gloo
    assert (r, w, local) == (rank, world, rank)
    case = config_case(1, seed=bench.rank_seed(1, r))
    digest = hashlib.sha256(case.q.tobytes() + case.k_pool.tobytes()).hexdigest()
    digests = [None] * w
    dist.all_gather_object(digests, digest)
    local_ms = 10.0 + 5.0 * r                      # rank 1 is the slower one
    total = bench.max_over_ranks(local_ms, w)
    bench.barrier(w)
    value = bench.whole_job_value(w, 1_000_000, 4, total)
    out_q.put((r, digests, total, value))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_replicas():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    (_, dig0, tot0, val0), (_, dig1, tot1, val1) = results
    # every rank sees the same gathered digests, and the two replicas drew different inputs
    assert dig0 == dig1 and dig0[0] != dig0[1]
    # the reported time is the slowest rank's, on every rank
    assert tot0 == tot1 == 15.0
    # whole-job value: 2 ranks x 1 MB x 4 steps over 15 ms
    assert val0 == val1 == pytest.approx(2 * 1e6 * 4 / 15e-3 / 1e9)


def test_rank_seeds_distinct():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.rank_seed(2, 0) is None                # rank 0: the named configuration
    seeds = {bench.rank_seed(k, r) for k in range(1, 6) for r in range(1, 9)}
    assert len(seeds) == 5 * 8                          # no two (config, rank) pairs collide
