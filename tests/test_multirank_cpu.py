"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the
max-over-ranks timing reduction, per-rank independent workloads (weak
scaling by batch), and the reference arm running on rank 0 only."""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from gated_delta_rule_chunkwise_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(10.0 * rank + 0.5, world, "cpu")
        w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=8, H=1, seed=bench.rank_seed(rank))
        digest = float(np.sum(w.q.astype(np.float64)))
        # reference arm: only rank 0 does any work
        import argparse
        rc = None
        if rank != 0:
            rc = bench.run_reference(argparse.Namespace(workload="gdn_bf16_b4_t2048_h16_d128", steps=1,
                                                        warmup=3, gpus=world))
        q.put((rank, got, digest, rc))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, d0, _), (r1, m1, d1, rc1) = res
    assert m0 == m1 == 10.5                # max over ranks, seen by every rank
    assert d0 != d1                        # independent sequences per rank
    assert rc1 == 0                        # non-zero ranks skip the reference arm
