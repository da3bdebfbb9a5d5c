"""gdn_chunk_fwd_noalloc: the forward pass for callers that cannot allocate
device memory (a framework that owns every device buffer and hands the op
only its inputs and outputs, or a caller that cannot accept the implicit
device-wide synchronisation of cudaMalloc).  It runs with a built-in 32 MiB
static device scratch instead of a workspace.

Checked through the C ABI against the existing entry point (gdn_chunk_fwd,
staged path) on two calls in a row with different problems, so that state
left in the shared scratch by the first call cannot leak into the second.
This file is named to be collected last.
"""
import ctypes

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
    lib = binding.load()
    lib.gdn_chunk_fwd_noalloc.argtypes = ([ctypes.POINTER(binding.Problem)] + [ctypes.c_void_p] * 5 +
                                          [ctypes.c_float] + [ctypes.c_void_p] * 5)
    lib.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
    return binding


def noalloc_call(gdn, x, C):
    p = gdn.problem_of(x["q"], x["v"], C, x["cu_seqlens"])
    o = torch.empty_like(x["v"])
    ht = torch.empty((p.N, p.Hv, p.K, p.V), dtype=torch.float32, device=x["q"].device)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p()
    st = gdn.load().gdn_chunk_fwd_noalloc(ctypes.byref(p), ptr(x["q"]), ptr(x["k"]), ptr(x["v"]), ptr(x["g"]),
                                          ptr(x["beta"]), ctypes.c_float(x["scale"]), ptr(x["h0"]),
                                          ptr(x["cu_seqlens"]), ptr(o), ptr(ht),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, ht


CASES = [
    (I.WORKLOADS[0], None),                                             # fp32, h0, C = 64
    (I.WORKLOADS[3].with_(Hqk=2, Hv=4, C=128), [70, 0, 5, 130]),         # bf16, GQA, varlen, C = 128
]


def test_noalloc_matches_existing_entry_point_twice(gdn):
    for w, lens in CASES:
        x = I.make_inputs(w, "cuda", lengths=lens)
        st, o, ht = noalloc_call(gdn, x, w.C)
        assert st == gdn.GDN_OK, gdn.status_string(st)
        o_ref, ht_ref = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                          cu_seqlens=x["cu_seqlens"], C=w.C, path="staged")
        torch.cuda.synchronize()
        tol = TOL[w.dtype]
        assert rel_fro(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= tol
        assert rel_fro(ht.cpu().numpy(), ht_ref.cpu().numpy()) <= tol
        assert np.all(np.isfinite(o.float().cpu().numpy()))


def test_noalloc_rejects_problems_beyond_its_scratch(gdn):
    x = I.make_inputs(I.WORKLOADS[1].with_(T=2048), "cuda")   # staged workspace far above 32 MiB
    p = gdn.problem_of(x["q"], x["v"], 64)
    assert gdn.gdn_chunk_fwd_workspace_size(p, "staged") > (32 << 20)
    st, _, _ = noalloc_call(gdn, x, 64)
    assert st == 5   # GDN_ERR_SCRATCH_LIMIT
    assert "static scratch" in gdn.status_string(st)
