"""World-size-2 gloo test of the benchmark's multi-rank host logic (CPU only):
rendezvous, barrier, the max-over-ranks step time and per-rank request shards
(weak scaling, no collective on the data path)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import bench
    from speculative_decoding_verification_37_gb300 import workloads as W
    r, w, _ = bench.dist_setup()
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + r, w)
    spec = W.ChainSpec("shard", B=3, gamma=2, V=64, dtype="f32", target_sigma=1.0,
                       temperature=1.0, draft_sigma=0.5)
    shard = W.make_chain(spec, seed=r)               # each rank's own batch, as bench.py does
    q.put((r, w, t, shard.target[0, :4].tolist(), shard.draft_tokens.tolist()))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_gloo_sharding_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[2] == pytest.approx(2.5) for x in res)     # the slowest rank's time
    assert res[0][3] != res[1][3]                            # distinct shards
    assert np.asarray(res[0][4]).shape == (3, 2)
