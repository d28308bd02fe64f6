"""Host-side logic of the N-GPU benchmark on CPU: two gloo ranks each take
their own shard of chains (no collective on the data path), the shards
together equal the single-process workload, and the step time is the maximum
over ranks."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

import bench
import spec_inputs as si

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, per_rank, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = si.C3_T1.scaled(batch=per_rank * world, vocab=1024)
    b0, nb = bench.shard_range(rank, world, per_rank)
    b = si.generate(w, b0, nb, nthreads=1)
    elapsed = torch.tensor([10.0 * (rank + 1)])            # a stand-in per-rank step time
    dist.all_reduce(elapsed, op=dist.ReduceOp.MAX)
    dist.barrier()
    q.put((rank, b0, nb, b.target.copy(), b.tokens.copy(), b.uniforms.copy(), float(elapsed.item())))
    dist.destroy_process_group()


def test_two_rank_sharding_gloo():
    world, per_rank = 2, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, per_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    whole = si.generate(si.C3_T1.scaled(batch=per_rank * world, vocab=1024), nthreads=1)
    assert [r[1] for r in res] == [0, per_rank] and all(r[2] == per_rank for r in res)
    assert np.array_equal(np.concatenate([r[3] for r in res]), whole.target)
    assert np.array_equal(np.concatenate([r[4] for r in res]), whole.tokens)
    assert np.array_equal(np.concatenate([r[5] for r in res]), whole.uniforms)
    assert all(r[6] == 10.0 * world for r in res)          # max over ranks
