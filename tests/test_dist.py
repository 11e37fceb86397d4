"""Multi-rank host logic on CPU with gloo, world_size 2: the job's step time is
the max over ranks, per-rank batches are distinct, the value counts every
rank's units."""
import os

import pytest
import torch.multiprocessing as mp


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_attention_indexer_idx_gb300 import dist as D
    ms = D.job_step_ms(1.0 + rank * 2.5)
    q.put((rank, ms, D.rank_seed(3, rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert all(p.exitcode == 0 for p in procs)
    assert [r[1] for r in res] == [3.5, 3.5]
    assert res[0][2] != res[1][2]


def test_single_process_and_value():
    from sparse_attention_indexer_idx_gb300 import dist as D
    assert D.job_step_ms(2.0) == 2.0
    assert D.job_value(1000, 2.0, 4) == pytest.approx(2e6)
