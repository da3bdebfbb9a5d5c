"""Multi-rank host logic on CPU (gloo, world_size 2).

* The weak-scaling aggregation bench.py uses (max over ranks, whole-job
  tokens/s).
* One call split over the ranks (gated_deltanet_chunked_gdn_gb300.partition):
  by qk-head groups (each rank its qk heads, their value heads and the matching
  h0 / ht slices) and by whole sequences of a packed batch (cut at cu_seqlens
  boundaries, with empty and sub-chunk sequences).  Each rank runs its slice
  through the fp64 oracle on the CPU, the slices are gathered and put back
  together, and the result must equal a single-process oracle run of the whole
  problem element by element (the chains are independent, so exactly).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(ROOT)

PACKED_LENS = [70, 0, 5, 130, 1, 300, 64, 17]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problems():
    from gated_deltanet_chunked_gdn_gb300 import inputs as I
    heads = I.make_inputs(I.WORKLOADS[1].with_(T=90, Hqk=4, Hv=8, K=16, V=8, dtype="f32"), "cpu")
    heads["h0"] = torch.randn(1, 8, 16, 8, generator=torch.Generator().manual_seed(5)) * 0.1
    packed = I.make_inputs(I.WORKLOADS[3].with_(Hqk=1, Hv=2, K=8, V=8, dtype="f32"), "cpu", lengths=PACKED_LENS)
    return heads, packed


def _run(oracle, x):
    return oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                            cu_seqlens=x["cu_seqlens"])


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from gated_deltanet_chunked_gdn_gb300 import partition as P
    from oracle import oracle
    # rank r took (1 + r) seconds for 3 steps of 1000 tokens
    value, t = bench.aggregate(1.0 + rank, 1000, 3, world)
    heads, packed = _problems()
    hp = P.head_part(4, 8, world, rank)
    o_h, ht_h = _run(oracle, P.slice_heads(heads, hp))
    sp = P.seq_part(world, rank, 1, packed["q"].shape[1], packed["cu_seqlens"].tolist())
    o_s, ht_s = _run(oracle, P.slice_sequences(packed, sp))
    gathered = [None] * world
    dist.all_gather_object(gathered, (value, t, hp, (o_h, ht_h), sp, (o_s, ht_s)))
    if rank == 0:
        out.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_split_one_call_over_two_ranks_equals_the_whole():
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
    for value, t, *_ in res:
        assert t == 2.0 and value == pytest.approx(3000.0)

    import sys
    sys.path.insert(0, ROOT)
    from gated_deltanet_chunked_gdn_gb300 import partition as P
    from oracle import oracle
    heads, packed = _problems()
    t = lambda pair: tuple(torch.from_numpy(a) for a in pair)

    # head split: each rank owns qk heads and their value heads, nobody is left out
    parts = [r[2] for r in res]
    assert [(p.hq0, p.hq1, p.hv0, p.hv1) for p in parts] == [(0, 2, 0, 4), (2, 4, 4, 8)]
    o, ht = P.assemble_heads(parts, [t(r[3]) for r in res])
    o_ref, ht_ref = _run(oracle, heads)
    assert np.array_equal(o.numpy(), o_ref) and np.array_equal(ht.numpy(), ht_ref)

    # sequence split: whole sequences, token counts as even as they allow
    parts = [r[4] for r in res]
    assert parts[0].n0 == 0 and parts[-1].n1 == len(PACKED_LENS) and parts[0].n1 == parts[1].n0
    assert parts[0].t1 == sum(PACKED_LENS[:parts[0].n1])
    o, ht = P.assemble_sequences(parts, [t(r[5]) for r in res], packed=True)
    o_ref, ht_ref = _run(oracle, packed)
    assert np.array_equal(o.numpy(), o_ref) and np.array_equal(ht.numpy(), ht_ref)


def test_partition_bookkeeping():
    import sys
    sys.path.insert(0, ROOT)
    from gated_deltanet_chunked_gdn_gb300 import partition as P
    # every qk head and value head owned exactly once, value heads follow their qk head
    for Hqk, Hv, world in [(8, 32, 3), (16, 32, 4), (3, 3, 2), (1, 4, 2)]:
        parts = [P.head_part(Hqk, Hv, world, r) for r in range(world)]
        assert parts[0].hq0 == 0 and parts[-1].hq1 == Hqk
        for a, b in zip(parts, parts[1:]):
            assert a.hq1 == b.hq0 and a.hv1 == b.hv0
        for p in parts:
            assert p.hv0 == p.hq0 * (Hv // Hqk) and p.hv1 == p.hq1 * (Hv // Hqk)
    # whole sequences, in order, covering every token; balanced within one sequence's length
    cu = [0]
    for L in [5, 0, 900, 3, 3, 400, 0, 77, 1000]:
        cu.append(cu[-1] + L)
    for world in (2, 3, 4):
        parts = [P.seq_part(world, r, 1, cu[-1], cu) for r in range(world)]
        assert parts[0].n0 == 0 and parts[-1].n1 == len(cu) - 1
        for a, b in zip(parts, parts[1:]):
            assert a.n1 == b.n0 and a.t1 == b.t0
        longest = max(b - a for a, b in zip(cu, cu[1:]))
        for p in parts:
            assert abs((p.t1 - p.t0) - cu[-1] / world) <= longest
    # fixed-length batches split by rows
    assert [(p.n0, p.n1) for p in (P.seq_part(2, r, 5, 64) for r in range(2))] == [(0, 2), (2, 5)]
    with pytest.raises(ValueError):
        P.seq_part(2, 0, 1, 10, [0, 5, 3, 10])
