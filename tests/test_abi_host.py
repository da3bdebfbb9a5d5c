"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/gdn.h declares, sizes workspaces, and rejects bad arguments
before any CUDA call."""
import ctypes
import os
import re

import pytest

from gated_deltanet_chunked_gdn_gb300 import binding as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = b.load()
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"libgdn.so does not export {n}"
    assert set(b.EXPORTED) <= set(names)
    assert b.gdn_version().startswith("gdn")


def test_status_strings():
    for s in range(5):
        assert b.status_string(s)
    assert b.status_string(99) == "unknown status"


def P(**kw):
    base = dict(B=2, T=300, N=2, Hqk=2, Hv=4, K=128, V=128, C=64, dtype="bf16", varlen=0)
    base.update(kw)
    return b.problem(**base)


@pytest.mark.parametrize("bad", [dict(Hv=3), dict(K=96), dict(V=32), dict(C=32), dict(B=0), dict(T=0),
                                 dict(Hqk=0), dict(varlen=1, B=2), dict(varlen=1, N=0), dict(dtype=7)])
def test_invalid_problems_have_no_workspace(bad):
    p = P(**bad)
    if "dtype" in bad:
        p.dt = 7
    assert b.gdn_chunk_fwd_workspace_size(p, "auto") == 0
    assert b.gdn_chunk_fwd_workspace_size(p, "staged") == 0


def test_workspace_matches_staged_layout():
    p = P()
    L = b.gdn_staged_layout(p)
    assert L.nc_max == 2 * 5
    assert b.gdn_chunk_fwd_workspace_size(p, "staged") == L.total
    offs = [L.tables, L.status, L.gamma, L.A, L.Tinv, L.W, L.U, L.S0, L.Vn, L.total]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.Vn - L.S0 == 4 * L.nc_max * 4 * 128 * 128
    pv = P(B=1, T=1000, N=7, varlen=1)
    assert b.gdn_staged_layout(pv).nc_max == -(-1000 // 64) + 7


def call(p, path=0, ptrs=None, ws_bytes=1 << 30, ws=1 << 20, stage=None):
    """Calls with fake (never dereferenced) device addresses; every case here
    must be rejected by host validation before any CUDA call."""
    lib = b.load()
    x = ptrs or {}
    a = lambda k_, d: ctypes.c_void_p(x.get(k_, d))
    args = [ctypes.byref(p), path if stage is None else stage, a("q", 1 << 12), a("k", 2 << 12), a("v", 3 << 12),
            a("g", 4 << 12), a("beta", 5 << 12), ctypes.c_float(0.1), a("h0", 0), a("cu", 0), a("o", 6 << 12),
            a("ht", 0), ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes), ctypes.c_void_p(0)]
    fn = lib.gdn_chunk_fwd if stage is None else lib.gdn_chunk_fwd_staged
    return fn(*args)


def test_rejects_null_and_misaligned_pointers():
    p = P()
    assert call(p, ptrs={"q": 0}) == b.GDN_ERR_INVALID_ARG
    assert call(p, ptrs={"o": 0}) == b.GDN_ERR_INVALID_ARG
    assert call(p, ptrs={"q": (1 << 12) + 8}) == b.GDN_ERR_INVALID_ARG     # TMA wants 16-byte alignment
    assert call(p, ptrs={"g": (4 << 12) + 2}) == b.GDN_ERR_INVALID_ARG
    assert call(p, ws=(1 << 20) + 128) == b.GDN_ERR_INVALID_ARG           # workspace must be 256-aligned


def test_rejects_small_workspace_and_bad_shapes():
    p = P()
    need = b.gdn_chunk_fwd_workspace_size(p, "staged")
    assert call(p, path=1, ws_bytes=need - 1) == b.GDN_ERR_INVALID_ARG
    assert call(P(Hv=6, Hqk=4)) == b.GDN_ERR_INVALID_ARG
    assert call(P(K=512)) == b.GDN_ERR_INVALID_ARG
    assert call(p, path=9) == b.GDN_ERR_INVALID_ARG


def test_varlen_needs_cu_seqlens_and_fixed_forbids_it():
    assert call(P(B=1, N=3, varlen=1)) == b.GDN_ERR_INVALID_ARG                 # no cu_seqlens
    assert call(P(), ptrs={"cu": 7 << 12}) == b.GDN_ERR_INVALID_ARG             # cu_seqlens with fixed length


def test_staged_rejects_bad_stop_point():
    assert call(P(), stage=7) == b.GDN_ERR_INVALID_ARG
    assert call(P(), stage=-1) == b.GDN_ERR_INVALID_ARG


def test_fused_path_reports_unsupported_problems():
    # fp32 inputs and head dims other than 128 are outside the fused kernel.
    p = P(dtype="f32")
    assert b.gdn_chunk_fwd_workspace_size(p, "fused") == 0
    assert b.gdn_resolve_path(p) == "staged"
    assert call(p, path=2) == b.GDN_ERR_UNSUPPORTED


def conv_call(x=1 << 12, weight=2 << 12, bias=0, W=4, state=3 << 12, slots=2, idx=0, init=0, cu=0, N=2, B=2, T=16,
              D=64, dt=1, act=1, y=4 << 12):
    """gdn_causal_conv1d_fwd with fake (never dereferenced) device addresses;
    every case below must fail host validation before any CUDA call."""
    lib = b.load()
    v = ctypes.c_void_p
    return lib.gdn_causal_conv1d_fwd(v(x), v(weight), v(bias), W, v(state), slots, v(idx), v(init), v(cu), N, B, T,
                                     D, dt, act, v(y), v(0))


def test_conv1d_rejects_bad_arguments():
    bad = b.GDN_ERR_INVALID_ARG
    assert conv_call(D=12) == bad                    # channels must come in 16-byte vectors of bf16
    assert conv_call(W=0) == bad and conv_call(W=5) == bad
    assert conv_call(weight=0) == bad
    assert conv_call(x=0) == bad and conv_call(y=0) == bad
    assert conv_call(x=(1 << 12) + 8) == bad         # 16-byte alignment
    assert conv_call(state=(3 << 12) + 4) == bad
    assert conv_call(bias=(5 << 12) + 2) == bad
    assert conv_call(slots=1) == bad                 # identity slot map needs a slot per sequence
    assert conv_call(N=3) == bad                     # fixed length: N == B
    assert conv_call(cu=6 << 12, B=2) == bad         # packed batches have B == 1
    assert conv_call(dt=7) == bad and conv_call(act=2) == bad


def test_bwd_workspace_covers_both_forms():
    # the backward picks its form at call time (the chunked one needs 16-byte
    # aligned q, k, v and dout), so the queried size must cover the token
    # recurrence's checkpoints too: 64 KB a value head for every 64 tokens
    # (plus one a sequence) when K = V = 128
    for p in (P(B=256, T=8192, N=256, Hqk=32, Hv=32), P(B=2, T=300, N=2), P(B=1, T=5000, N=7, varlen=1)):
        slots = (p.B * p.T + 63) // 64 + p.N
        assert b.gdn_chunk_bwd_workspace_size(p) >= slots * p.Hv * p.K * p.V * 4
    # K = 64 only has the token recurrence
    q = P(K=64, V=64)
    slots = (q.B * q.T + 63) // 64 + q.N
    assert b.gdn_chunk_bwd_workspace_size(q) >= slots * q.Hv * 64 * 64 * 4
