"""Bounded waits of the fused kernel, exercised on the GPU without a fault.

The window schedule hands the state of a chain cut at a window boundary from
one CTA to another through a flag in the workspace.  The test hook
gdn_selftest_handover_timeout runs the fused pass with one window's flag never
raised and a 1 ms limit on the wait for it: the waiting window must give up,
record GDN_DEV_WAIT_TIMEOUT, leave exactly one chain unfinished, and the launch
must end; the next ordinary call on the same workspace must be exact.
"""
import ctypes

import pytest
import torch

from gated_deltanet_chunked_gdn_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    lib = binding.load()
    lib.gdn_selftest_handover_timeout.argtypes = ([ctypes.POINTER(binding.Problem), ctypes.c_int] +
                                                  [ctypes.c_void_p] * 5 +
                                                  [ctypes.c_float] + [ctypes.c_void_p] * 4 +
                                                  [ctypes.c_size_t, ctypes.c_int, ctypes.c_longlong,
                                                   ctypes.c_void_p])
    lib.gdn_selftest_handover_timeout.restype = ctypes.c_int
    return binding


CASES = {
    # 512 chains of 4 chunks over the 2 x SMs CTA slots: windows of more than
    # one chain's chunks, so window boundaries cut chains
    "d128": (I.WORKLOADS[2].with_(B=4, T=256, Hqk=128, Hv=128), "fused"),
    # the same over one CTA per SM (groups of 1 window: G = 1, one value slice)
    "d128_fused1": (I.WORKLOADS[2].with_(B=4, T=256, Hqk=128, Hv=128), "fused1"),
    # K = V = 256: 320 (chain, value slice) units of 3 chunks over one CTA per SM
    "d256": (I.WORKLOADS[4].with_(B=20, T=190, Hqk=2, Hv=8, h0=True), "fused1"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_handover_wait_times_out_and_the_next_call_is_exact(gdn, name):
    w, path = CASES[name]
    x = I.make_inputs(w, "cuda")
    p = gdn.problem_of(x["q"], x["v"], w.C)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(p, path), dtype=torch.uint8, device="cuda")
    call = lambda: gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"], C=w.C,
                                     path=path, workspace=ws)
    o_ref, ht_ref = call()
    assert gdn.gdn_get_device_status(p, path, ws) == gdn.DEV_OK

    o = torch.full_like(o_ref, float("nan"))
    ht = torch.full_like(ht_ref, float("nan"))
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    lib = gdn.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = gdn.GDN_ERR_UNSUPPORTED
    for window in range(1, 64):
        st = lib.gdn_selftest_handover_timeout(ctypes.byref(p), gdn.PATHS[path], ptr(x["q"]), ptr(x["k"]), ptr(x["v"]),
                                               ptr(x["g"]),
                                               ptr(x["beta"]), ctypes.c_float(x["scale"]), ptr(x["h0"]), ptr(o),
                                               ptr(ht), ptr(ws), ctypes.c_size_t(ws.numel()), window,
                                               ctypes.c_longlong(1_000_000), stream)
        if st != gdn.GDN_ERR_UNSUPPORTED:
            break
    assert st == gdn.GDN_OK, gdn.status_string(st)
    torch.cuda.synchronize()          # the launch ends
    assert gdn.gdn_get_device_status(p, path, ws) == gdn.DEV_WAIT_TIMEOUT

    # exactly the chain the window gave up on is unfinished; every other chain is exact
    unfinished = torch.isnan(ht).flatten(2).any(-1)          # [N, Hv]
    assert int(unfinished.sum()) == 1
    done = ~unfinished
    assert torch.equal(ht[done], ht_ref[done])
    n, h = [int(i) for i in unfinished.nonzero()[0]]
    keep = torch.ones_like(o_ref, dtype=torch.bool)
    keep[n, :, h] = False
    assert torch.equal(o[keep], o_ref[keep])

    # the next ordinary call on the same workspace clears the schedule and is exact
    o2, ht2 = call()
    assert gdn.gdn_get_device_status(p, path, ws) == gdn.DEV_OK
    assert torch.equal(o2, o_ref) and torch.equal(ht2, ht_ref)
