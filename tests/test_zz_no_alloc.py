"""gdn_chunk_fwd_noalloc: the forward pass for callers that cannot allocate
device memory (a framework that owns every device buffer and hands the op
only its inputs and outputs, or a caller that cannot accept the implicit
device-wide synchronisation of cudaMalloc).  It runs with a built-in 32 MiB
static device scratch instead of a workspace: the fused kernels when their
workspace fits (AUTO's choice, the two-CTA kernel in place of the
chunk-parallel path), else the staged path.

Checked through the C ABI against the existing entry point (gdn_chunk_fwd on
the same path: the same kernels, so the results must be equal bit for bit) on
calls in a row with different problems and paths -- the window schedule with
its hand-over states, a packed batch, an fp32 problem on the staged path, and
the packed batch again -- so that data left in the shared scratch by one call
cannot leak into the next; once against the fp64 oracle; and with malformed
cu_seqlens, whose device status the caller reads with
gdn_chunk_fwd_noalloc_get_device_status.  This file is named to be collected
last.
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
    lib.gdn_chunk_fwd_noalloc_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    lib.gdn_chunk_fwd_noalloc_get_device_status.restype = ctypes.c_int
    return binding


def stream_ptr():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def noalloc_call(gdn, x, C, cu=None):
    cu = x["cu_seqlens"] if cu is None else cu
    p = gdn.problem_of(x["q"], x["v"], C, cu)
    o = torch.full_like(x["v"], float("nan"))
    ht = torch.full((p.N, p.Hv, p.K, p.V), float("nan"), dtype=torch.float32, device=x["q"].device)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p()
    st = gdn.load().gdn_chunk_fwd_noalloc(ctypes.byref(p), ptr(x["q"]), ptr(x["k"]), ptr(x["v"]), ptr(x["g"]),
                                          ptr(x["beta"]), ctypes.c_float(x["scale"]), ptr(x["h0"]), ptr(cu),
                                          ptr(o), ptr(ht), stream_ptr())
    return st, o, ht


def noalloc_status(gdn):
    out = ctypes.c_int(-1)
    st = gdn.load().gdn_chunk_fwd_noalloc_get_device_status(stream_ptr(), ctypes.byref(out))
    assert st == gdn.GDN_OK, gdn.status_string(st)
    return out.value


SCRATCH = (32 << 20) - 256   # the array less its status slot


def expected_path(gdn, p):
    """The path a gdn_chunk_fwd_noalloc call takes (None: it is refused)."""
    path = gdn.gdn_resolve_path(p)
    if path == "cp":
        path = "fused"
    if path != "staged" and gdn.gdn_chunk_fwd_workspace_size(p, path) <= SCRATCH:
        return path
    return "staged" if gdn.gdn_chunk_fwd_workspace_size(p, "staged") <= SCRATCH else None


# the window schedule (hand-over states in the scratch), a packed batch, an
# fp32 problem on the staged path, and the packed batch again
WINDOWS = (I.WORKLOADS[2].with_(B=16, T=2048), None)                        # bf16, H = 32, windows cut chains
VARLEN = (I.WORKLOADS[3].with_(Hqk=2, Hv=4, C=128), [70, 0, 5, 130, 300])   # bf16, GQA, varlen, C = 128
FP32 = (I.WORKLOADS[0], None)                                              # fp32, h0, C = 64
CASES = [WINDOWS, VARLEN, FP32, VARLEN]


def test_noalloc_matches_existing_entry_point_bit_for_bit(gdn):
    paths = []
    for w, lens in CASES:
        x = I.make_inputs(w, "cuda", lengths=lens)
        path = expected_path(gdn, gdn.problem_of(x["q"], x["v"], w.C, x["cu_seqlens"]))
        paths.append(path)
        st, o, ht = noalloc_call(gdn, x, w.C)
        assert st == gdn.GDN_OK, gdn.status_string(st)
        assert noalloc_status(gdn) == gdn.DEV_OK
        o_ref, ht_ref = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                          cu_seqlens=x["cu_seqlens"], C=w.C, path=path)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(ht, ht_ref)
    assert paths == ["fused", "fused1", "staged", "fused1"]


def test_noalloc_against_the_oracle(gdn, oracle_mod):
    w, lens = VARLEN
    x = I.make_inputs(w, "cpu", lengths=lens)
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    st, o, ht = noalloc_call(gdn, d, w.C)
    assert st == gdn.GDN_OK, gdn.status_string(st)
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                         cu_seqlens=x["cu_seqlens"])
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL[w.dtype]
    assert rel_fro(ht.cpu().numpy(), ht_ref) <= TOL[w.dtype]


def test_noalloc_reports_malformed_cu_seqlens(gdn):
    w, lens = VARLEN
    x = I.make_inputs(w, "cuda", lengths=lens)
    bad = x["cu_seqlens"].clone()
    bad[-1] = bad[-1] - 1          # cu[N] != T
    st, _, _ = noalloc_call(gdn, x, w.C, cu=bad)
    assert st == gdn.GDN_OK        # enqueued; the error is found on the device
    assert noalloc_status(gdn) == gdn.DEV_BAD_CU_SEQLENS
    assert noalloc_status(gdn) == gdn.DEV_OK    # read and cleared
    st, o, ht = noalloc_call(gdn, x, w.C)       # the next well-formed call is clean
    assert st == gdn.GDN_OK
    assert noalloc_status(gdn) == gdn.DEV_OK
    assert np.all(np.isfinite(o.float().cpu().numpy())) and np.all(np.isfinite(ht.cpu().numpy()))


def test_noalloc_rejects_problems_beyond_its_scratch(gdn):
    # fp32 inputs: no fused kernel, and a staged workspace above 32 MiB
    x = I.make_inputs(I.WORKLOADS[0].with_(B=2, T=4096, Hqk=4, Hv=4), "cuda")
    p = gdn.problem_of(x["q"], x["v"], 64)
    assert expected_path(gdn, p) is None
    assert gdn.gdn_chunk_fwd_workspace_size(p, "staged") > (32 << 20)
    st, _, _ = noalloc_call(gdn, x, 64)
    assert st == 5   # GDN_ERR_SCRATCH_LIMIT
    assert "static scratch" in gdn.status_string(st)
