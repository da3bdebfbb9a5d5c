"""GPU parity of the chunk-parallel path (sequences cut into segments that run
on separate SMs; segment transitions chained by an fp32 combine step) against
the fp64 oracle, through the C ABI.  Same bar as the other bf16 paths:
relative Frobenius error of o and ht at most 5e-3."""
import numpy as np
import pytest
import torch

from conftest import rel_fro
from gated_deltanet_chunked_gdn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 5e-3


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    binding.load()
    return binding


def run_cp(gdn, w, lens=None, device_inputs=False):
    x = I.make_inputs(w, "cpu", lengths=lens)
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    p = gdn.problem_of(d["q"], d["v"], w.C, d["cu_seqlens"])
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(p, "cp"), dtype=torch.uint8, device="cuda")
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                              cu_seqlens=d["cu_seqlens"], C=w.C, path="cp", workspace=ws)
    assert gdn.gdn_get_device_status(p, "cp", ws) == gdn.DEV_OK
    return x, d, o.float().cpu().numpy(), ht.cpu().numpy()


CASES = {
    "gqa_prefill_1x4096": (I.WORKLOADS[1], None),
    "fixed_B2_ragged_h0": (I.WORKLOADS[2].with_(B=2, T=1000, Hqk=2, Hv=4, C=64), None),
    "varlen_short_empty": (I.WORKLOADS[3].with_(Hqk=1, Hv=2), [5, 64, 200, 1, 0, 129, 63, 700, 2048]),
    "single_chain_long": (I.WORKLOADS[2].with_(B=1, T=3000, Hqk=1, Hv=1, C=128), None),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_cp_parity(gdn, oracle_mod, name):
    w, lens = CASES[name]
    x, _, o, ht = run_cp(gdn, w, lens)
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                         cu_seqlens=x["cu_seqlens"])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(ht))
    assert rel_fro(o, o_ref) <= TOL, rel_fro(o, o_ref)
    assert rel_fro(ht, ht_ref) <= TOL, rel_fro(ht, ht_ref)


def test_auto_takes_cp_for_few_long_chains(gdn):
    w = I.WORKLOADS[1]   # 1 x 4096 tokens, 32 value heads: 32 chains
    x = I.make_inputs(w, "cuda")
    assert gdn.gdn_resolve_path(gdn.problem_of(x["q"], x["v"], w.C)) == "cp"
    w = I.WORKLOADS[2]   # 16 x 8192, 32 heads: 512 chains
    x = I.make_inputs(w.with_(B=16, T=64), "cuda")
    assert gdn.gdn_resolve_path(gdn.problem_of(x["q"], x["v"], w.C)) == "fused"


def test_cp_matches_fused(gdn):
    """The chunk-parallel and serial fused paths agree with each other."""
    w = I.WORKLOADS[2].with_(B=2, T=2500, Hqk=2, Hv=2, C=64)
    x = I.make_inputs(w, "cuda")
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"])
    oc, hc = gdn.gdn_chunk_fwd(*args, h0=x["h0"], C=64, path="cp")
    of, hf = gdn.gdn_chunk_fwd(*args, h0=x["h0"], C=64, path="fused")
    torch.cuda.synchronize()
    assert rel_fro(oc.float().cpu().numpy(), of.float().cpu().numpy()) < TOL
    assert rel_fro(hc.cpu().numpy(), hf.cpu().numpy()) < TOL


def test_cp_without_final_state_and_h0(gdn, oracle_mod):
    w = I.WORKLOADS[1].with_(T=1500, Hqk=2, Hv=4)
    x = I.make_inputs(w, "cpu")
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], C=64, path="cp",
                              output_final_state=False)
    assert ht is None
    o_ref, _ = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"])
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL


def test_cp_malformed_cu_seqlens(gdn):
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    x = I.make_inputs(w, "cuda", lengths=[10, 20, 30])
    bad = torch.tensor([0, 10, 70, 60], dtype=torch.int32, device="cuda")
    p = gdn.problem_of(x["q"], x["v"], 64, bad)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(p, "cp"), dtype=torch.uint8, device="cuda")
    o = torch.full_like(x["v"], 7.0)
    gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], cu_seqlens=bad, C=64, path="cp",
                      o=o, workspace=ws)
    assert gdn.gdn_get_device_status(p, "cp", ws) == gdn.DEV_BAD_CU_SEQLENS
    assert torch.all(o == 7.0)   # nothing written
