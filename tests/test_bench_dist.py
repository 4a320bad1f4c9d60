"""Multi-process (world size 2, gloo, CPU) check of bench.py's replica logic: each rank
reads its rank from the environment, draws its own batch (distinct seed, weak
scaling), and the reported time is the maximum over ranks.  The data path has no
collective; only the timing reduction crosses ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    from paged_kv_decode_12_gb300 import workloads as wl

    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w, init_method=f"tcp://127.0.0.1:{port}")
    elapsed = 10.0 + 5.0 * r                       # rank 1 is the slow one
    m = bench.reduce_max(elapsed, w)
    seed = bench.replica_seed(12, r)
    lens = wl.make_workload("b64", seed).seq_lens
    results[r] = (r, w, local, m, seed, int(lens.sum()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
    assert all(p.exitcode == 0 for p in procs)
    r0, r1 = results[0], results[1]
    assert (r0[0], r0[1], r1[0], r1[1]) == (0, 2, 1, 2)
    assert r0[3] == r1[3] == 15.0                   # max over ranks, seen by both
    assert r0[4] != r1[4] and r0[5] != r1[5]        # independent replicas draw different batches
