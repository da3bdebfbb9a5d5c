"""Multi-rank host logic on CPU (gloo, world_size 2): the weak-scaling
aggregation bench.py uses (max over ranks, whole-job tokens/s), and the
independence of ranks' work -- each rank's (sequence, head) chains computed
alone equal the same chains of a single full run (oracle on the CPU)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from gated_deltanet_chunked_gdn_gb300 import inputs as I
    from oracle import oracle
    # rank r took (1 + r) seconds for 3 steps of 1000 tokens
    value, t = bench.aggregate(1.0 + rank, 1000, 3, world)
    # independent batch per rank (seed differs per rank, as in bench.py)
    w = I.WORKLOADS[2].with_(B=2, T=40, Hqk=1, Hv=2, K=8, V=8, seed=2 + rank, dtype="f32")
    x = I.make_inputs(w, "cpu")
    o, ht = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"])
    gathered = [None] * world
    dist.all_gather_object(gathered, (value, t, o.sum(), ht.sum()))
    if rank == 0:
        out.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_weak_scaling_aggregation_and_rank_independence():
    pytest.importorskip("torch.distributed")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world = 2
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = q.get(timeout=240)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # every rank sees the max elapsed (2 s) and the whole-job value 2*1000*3/2
    for value, t, _, _ in res:
        assert t == 2.0 and value == pytest.approx(3000.0)
    # each rank's batch equals a single-process run of the same seed
    import sys
    sys.path.insert(0, ROOT)
    from gated_deltanet_chunked_gdn_gb300 import inputs as I
    from oracle import oracle
    for r in range(world):
        w = I.WORKLOADS[2].with_(B=2, T=40, Hqk=1, Hv=2, K=8, V=8, seed=2 + r, dtype="f32")
        x = I.make_inputs(w, "cpu")
        o, ht = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"])
        assert np.isclose(res[r][2], o.sum()) and np.isclose(res[r][3], ht.sum())
