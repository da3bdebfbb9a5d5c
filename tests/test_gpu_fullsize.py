"""Parity at the five workloads' full sizes (GPU).

Each workload runs whole on the GPU through the C ABI in the path the
library selects for it (the configuration bench.py times for the
16 x 8192 batch); then a few sampled (sequence, value head) chains are
recomputed one by one by the fp64 oracle and compared on their o rows and
final state.  Inputs come from the seeded recipe, drawn on the device.
"""
import numpy as np
import pytest
import torch

from conftest import rel_fro
from gated_deltanet_chunked_gdn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 5e-3}


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    binding.load()
    return binding


def check_chains(gdn, oracle_mod, w, chains, lengths=None, nthreads=0):
    x = I.make_inputs(w, "cuda", lengths=lengths)
    o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], C=w.C)
    torch.cuda.synchronize()
    G = w.Hv // w.Hqk
    cu = x["cu_seqlens"].cpu().tolist() if x["cu_seqlens"] is not None else None
    for n, h in chains:
        if cu is None:
            b, sl = n, slice(0, w.T)
        else:
            b, sl = 0, slice(cu[n], cu[n + 1])
        hq = h // G
        sub = lambda t, hh: t[b:b + 1, sl, hh:hh + 1].contiguous().cpu()
        h0 = x["h0"][n:n + 1, h:h + 1].cpu() if x["h0"] is not None else None
        o_ref, ht_ref = oracle_mod.recurrent(sub(x["q"], hq), sub(x["k"], hq), sub(x["v"], h), sub(x["g"], h),
                                             sub(x["beta"], h), x["scale"], h0=h0, nthreads=nthreads)
        o_got = o[b:b + 1, sl, h:h + 1].float().cpu().numpy()
        ht_got = ht[n:n + 1, h:h + 1].cpu().numpy()
        tol = TOL[w.dtype]
        assert np.all(np.isfinite(o_got)) and np.all(np.isfinite(ht_got))
        if o_ref.size:
            assert rel_fro(o_got, o_ref) <= tol, (n, h, rel_fro(o_got, o_ref))
        assert rel_fro(ht_got, ht_ref) <= tol, (n, h, rel_fro(ht_got, ht_ref))


def test_full_tiny_fp32(gdn, oracle_mod):
    w = I.WORKLOADS[0]
    check_chains(gdn, oracle_mod, w, [(0, 0), (0, 1)])


def test_full_gqa_prefill(gdn, oracle_mod):
    w = I.WORKLOADS[1]
    check_chains(gdn, oracle_mod, w, [(0, 0), (0, 17), (0, 31)])


@pytest.mark.parametrize("H", [32, 16, 48, 64])
def test_full_batched_16x8192(gdn, oracle_mod, H):
    w = I.WORKLOADS[2].with_(Hqk=H, Hv=H)
    # (0, 1) and (15, H - 1) straddle a window boundary of the fused schedule
    chains = [(0, 0), (0, 1), (7, H // 2 - 1), (15, H - 1)] if H == 32 else [(15, H - 1)]
    check_chains(gdn, oracle_mod, w, chains)


def test_full_varlen_64(gdn, oracle_mod):
    w = I.WORKLOADS[3]
    lens = I.varlen_lengths(w.varlen_n, w.seed, w.varlen_max)
    longest = int(np.argmax(lens))
    shortest = int(np.argmin(lens))
    mid = sorted(range(len(lens)), key=lambda i: lens[i])[len(lens) // 2]
    check_chains(gdn, oracle_mod, w, [(longest, 0), (shortest, 31), (mid, 5), (len(lens) - 1, 16)], lengths=lens)


def test_full_long_d256(gdn, oracle_mod):
    w = I.WORKLOADS[4]
    x = I.make_inputs(w.with_(B=1, T=64), "cuda")
    assert gdn.gdn_resolve_path(gdn.problem_of(x["q"], x["v"], w.C)) == "fused1"
    # chains of every qk group's first and last value head and of every
    # sequence; the fused schedule cuts some of them between two CTAs
    check_chains(gdn, oracle_mod, w, [(0, 0), (1, 7), (2, 20), (3, 31)], nthreads=4)


@pytest.mark.parametrize("path", ["auto", "fused", "fused1"])
def test_packed_long_and_short_sequences(gdn, oracle_mod, path):
    """A packed batch whose two 12 K-token sequences bound the step, mixed with
    short, sub-chunk and empty sequences: AUTO takes the one-CTA-per-SM kernel
    for it; both fused kernels are checked on the long and a few short chains."""
    w = I.WORKLOADS[3].with_(Hqk=4, Hv=8)
    lens = [12288, 5, 0, 700, 12001, 63, 1, 2000, 0, 130]
    x = I.make_inputs(w, "cuda", lengths=lens)
    p = gdn.problem_of(x["q"], x["v"], w.C, x["cu_seqlens"])
    if path == "auto":
        assert gdn.gdn_resolve_path(p) == "fused1"
    o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], C=w.C, path=path)
    torch.cuda.synchronize()
    cu = x["cu_seqlens"].cpu().tolist()
    G = w.Hv // w.Hqk
    for n, h in [(0, 0), (4, 7), (1, 3), (2, 5), (5, 2), (6, 1), (9, 6)]:
        sl = slice(cu[n], cu[n + 1])
        sub = lambda t, hh: t[:, sl, hh:hh + 1].contiguous().cpu()
        o_ref, ht_ref = oracle_mod.recurrent(sub(x["q"], h // G), sub(x["k"], h // G), sub(x["v"], h), sub(x["g"], h),
                                             sub(x["beta"], h), x["scale"], h0=x["h0"][n:n + 1, h:h + 1].cpu())
        o_got = o[:, sl, h:h + 1].float().cpu().numpy()
        ht_got = ht[n:n + 1, h:h + 1].cpu().numpy()
        assert np.all(np.isfinite(o_got)) and np.all(np.isfinite(ht_got))
        if o_ref.size:
            assert rel_fro(o_got, o_ref) <= TOL["bf16"], (n, h, rel_fro(o_got, o_ref))
        assert rel_fro(ht_got, ht_ref) <= TOL["bf16"], (n, h, rel_fro(ht_got, ht_ref))
