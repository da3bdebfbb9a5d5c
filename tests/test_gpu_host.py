"""The forward pass on host tensors (gdn_chunk_fwd_host, through the C ABI):
the batch streamed through the GPU in sub-batches of whole sequences gives
exactly the device-buffer forward's result on the fused path (each chain's
arithmetic does not depend on which other chains share its launch), and the
oracle's within the bf16 bar on AUTO."""
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


def host_inputs(x, pin=True):
    h = {}
    for k_ in ("q", "k", "v", "g", "beta", "h0", "cu_seqlens"):
        t = x[k_]
        h[k_] = None if t is None else (t.cpu().pin_memory() if pin else t.cpu().contiguous())
    return h


def device_reference(gdn, x, C, path, output_final_state=True):
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                              cu_seqlens=d["cu_seqlens"], C=C, path=path, output_final_state=output_final_state)
    torch.cuda.synchronize()
    return o.cpu(), (ht.cpu() if ht is not None else None)


CASES = {
    "fixed_B6_ragged_gqa": (I.WORKLOADS[2].with_(B=6, T=300, Hqk=2, Hv=4, C=64), None),
    "varlen_short_and_empty": (I.WORKLOADS[3].with_(Hqk=1, Hv=2), [5, 64, 200, 1, 0, 129, 63, 65]),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("nsplit", [1, 3, 8])
def test_host_matches_device_fused(gdn, name, nsplit):
    w, lens = CASES[name]
    x = I.make_inputs(w, "cpu", lengths=lens)
    o_ref, ht_ref = device_reference(gdn, x, w.C, "fused")
    h = host_inputs(x)
    o, ht = gdn.gdn_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], x["scale"], h0=h["h0"],
                                   cu_seqlens=h["cu_seqlens"], C=w.C, path="fused", nsplit=nsplit)
    assert torch.equal(o, o_ref)
    assert torch.equal(ht, ht_ref)


def test_host_auto_against_oracle(gdn, oracle_mod):
    w = I.WORKLOADS[3].with_(Hqk=2, Hv=4)
    lens = [700, 3, 0, 2100, 64, 129]
    x = I.make_inputs(w, "cpu", lengths=lens)
    h = host_inputs(x)
    ws = torch.empty(gdn.gdn_chunk_fwd_host_workspace_size(gdn.problem_of(h["q"], h["v"], w.C, h["cu_seqlens"]),
                                                           h["cu_seqlens"], 3), dtype=torch.uint8, device="cuda")
    o, ht = gdn.gdn_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], x["scale"], h0=h["h0"],
                                   cu_seqlens=h["cu_seqlens"], C=w.C, nsplit=3, workspace=ws)
    assert gdn.gdn_chunk_fwd_host_get_device_status(ws) == gdn.DEV_OK
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                         cu_seqlens=x["cu_seqlens"])
    assert rel_fro(o.float().numpy(), o_ref) <= TOL
    assert rel_fro(ht.numpy(), ht_ref) <= TOL


def test_host_pageable_no_h0_no_final_state(gdn):
    w = I.WORKLOADS[1].with_(T=400, Hqk=2, Hv=4)
    x = I.make_inputs(w, "cpu")
    assert x["h0"] is None
    o_ref, _ = device_reference(gdn, x, w.C, "fused", output_final_state=False)
    h = host_inputs(x, pin=False)
    o, ht = gdn.gdn_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], x["scale"], C=w.C, path="fused",
                                   nsplit=2, output_final_state=False)
    assert ht is None
    assert torch.equal(o, o_ref)


def test_host_rejects_malformed_offsets(gdn):
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    x = I.make_inputs(w, "cpu", lengths=[10, 20, 30])
    h = host_inputs(x)
    bad = torch.tensor([0, 25, 20, 60], dtype=torch.int32)
    with pytest.raises(gdn.GDNError):
        gdn.gdn_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], x["scale"], h0=h["h0"], cu_seqlens=bad,
                               C=64, nsplit=2)
