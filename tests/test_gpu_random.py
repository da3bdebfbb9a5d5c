"""Randomised GPU parity sweep: seeded draws of batch shape, GQA ratio, head
dims, chunk length, packed lengths (empty, sub-chunk and multi-chunk
sequences), initial state, gate recipe and execution path, each checked
against the fp64 oracle (the token recurrence) on o and ht at the accuracy
targets (1e-4 relative Frobenius for fp32 inputs, 5e-3 for bf16).  The fixed parity cases pin each path at chosen shapes; this
sweep covers the combinations between them."""
import numpy as np
import pytest
import torch

from conftest import rel_fro
from gated_deltanet_chunked_gdn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 5e-3}
NDRAWS = 64


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    binding.load()
    return binding


def draw(i):
    """Draw i: a workload, its packed lengths (or None) and the forced path."""
    r = np.random.default_rng(7000 + i)
    dtype = "bf16" if r.random() < 0.8 else "f32"
    K = int(r.choice([128, 256] if dtype == "bf16" else [64, 128]))
    V = int(r.choice([128, 256])) if (dtype == "bf16" and K == 256) else (128 if dtype == "bf16" else int(r.choice([64, 128])))
    if dtype == "bf16" and K == 128 and r.random() < 0.2:
        V = 256
    Hqk = int(r.choice([1, 2]))
    Hv = Hqk * int(r.choice([1, 2, 4]))
    C = int(r.choice([64, 128]))
    gate = "softplus_exp" if r.random() < 0.7 else "logsigmoid4"
    h0 = bool(r.random() < 0.6)
    lens = None
    if r.random() < 0.5:
        n = int(r.integers(1, 9))
        lens = [int(x) for x in r.integers(0, 300, size=n)]
        if r.random() < 0.5:
            lens[int(r.integers(0, n))] = int(r.integers(300, 700))
        w = I.Workload("random", 1, 0, Hqk, Hv, K, V, C, dtype, gate, h0, 100 + i, varlen_n=n)
    else:
        w = I.Workload("random", int(r.integers(1, 4)), int(r.integers(1, 400)), Hqk, Hv, K, V, C, dtype, gate,
                       h0, 100 + i)
    paths = ["auto", "staged"]
    if dtype == "bf16" and K in (128, 256) and V in (128, 256):
        paths.append("fused1")
        if K == 128 and V == 128:
            paths += ["fused", "cp"]
    return w, lens, paths[int(r.integers(0, len(paths)))]


@pytest.mark.parametrize("i", range(NDRAWS))
def test_random_draw_against_oracle(gdn, oracle_mod, i):
    w, lens, path = draw(i)
    x = I.make_inputs(w, "cuda", lengths=lens)
    o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], C=w.C, path=path)
    torch.cuda.synchronize()
    cpu = lambda t: None if t is None else t.cpu()
    o_ref, ht_ref = oracle_mod.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), cpu(x["beta"]),
                                         x["scale"], h0=cpu(x["h0"]), cu_seqlens=cpu(x["cu_seqlens"]))
    o_got, ht_got = o.float().cpu().numpy(), ht.cpu().numpy()
    assert np.all(np.isfinite(o_got)) and np.all(np.isfinite(ht_got))
    tol = TOL[w.dtype]
    if o_ref.size:
        assert rel_fro(o_got, o_ref) <= tol, (w, lens, path, rel_fro(o_got, o_ref))
    assert rel_fro(ht_got, ht_ref) <= tol, (w, lens, path, rel_fro(ht_got, ht_ref))


def draw_cp(i):
    """Draw i of the chunk-parallel sweep: sequences long enough to be cut
    into several segments, packed or of equal length."""
    r = np.random.default_rng(9100 + i)
    Hqk = int(r.choice([1, 2]))
    Hv = Hqk * int(r.choice([1, 2, 4]))
    h0 = bool(r.random() < 0.6)
    C = int(r.choice([64, 128]))
    if r.random() < 0.5:
        n = int(r.integers(1, 5))
        lens = [int(x) for x in r.integers(0, 5000, size=n)]
        w = I.Workload("random_cp", 1, 0, Hqk, Hv, 128, 128, C, "bf16", "softplus_exp", h0, 300 + i, varlen_n=n)
        return w, lens
    w = I.Workload("random_cp", int(r.integers(1, 3)), int(r.integers(500, 5000)), Hqk, Hv, 128, 128, C, "bf16",
                   "softplus_exp", h0, 300 + i)
    return w, None


@pytest.mark.parametrize("i", range(16))
def test_random_chunk_parallel_against_oracle(gdn, oracle_mod, i):
    w, lens = draw_cp(i)
    x = I.make_inputs(w, "cuda", lengths=lens)
    o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], C=w.C, path="cp")
    torch.cuda.synchronize()
    cpu = lambda t: None if t is None else t.cpu()
    o_ref, ht_ref = oracle_mod.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), cpu(x["beta"]),
                                         x["scale"], h0=cpu(x["h0"]), cu_seqlens=cpu(x["cu_seqlens"]))
    o_got, ht_got = o.float().cpu().numpy(), ht.cpu().numpy()
    if o_ref.size:
        assert rel_fro(o_got, o_ref) <= TOL["bf16"], (w, lens, rel_fro(o_got, o_ref))
    assert rel_fro(ht_got, ht_ref) <= TOL["bf16"], (w, lens, rel_fro(ht_got, ht_ref))
