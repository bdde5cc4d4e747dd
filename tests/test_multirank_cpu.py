"""World-size-2 gloo checks on the CPU of the host logic the multi-GPU bench runs: the
max-over-ranks timing reduction, and the amax agreement a sharded quantize needs (each rank
quantizes its row shard with the all-reduced amax; the shards equal the unsharded result)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle as O
        from mxfp8_precision_numerics_gb300 import inputs as I
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank], "cpu")
        x = I.normal_with_outliers(64, 128, seed=3)
        shard = I.bf16_bits(x)[rank * 32:(rank + 1) * 32]
        local = torch.tensor([float(np.abs(x.float().numpy()[rank * 32:(rank + 1) * 32]).max())])
        dist.all_reduce(local, op=dist.ReduceOp.MAX)
        c, s, _, d = O.quantize_1d(np.ascontiguousarray(shard), amax=float(local.item()))
        q.put((rank, got, c, s, d))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_timing_and_amax_agreement():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=120) for _ in range(2)], key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == [2.0, 5.0] and res[1][1] == [2.0, 5.0]
    import oracle as O
    from mxfp8_precision_numerics_gb300 import inputs as I
    c, s, _, d = O.quantize_1d(I.bf16_bits(I.normal_with_outliers(64, 128, seed=3)))
    assert np.array_equal(np.concatenate([res[0][2], res[1][2]]), c)
    assert np.array_equal(np.concatenate([res[0][3], res[1][3]]), s)
    assert res[0][4] == res[1][4] == d
