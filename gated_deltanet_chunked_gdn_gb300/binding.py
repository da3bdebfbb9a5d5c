"""Thin ctypes binding over libgdn.so (include/gdn.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, outputs and the workspace are allocated with torch when the caller
does not pass them, and everything else runs in the library's CUDA kernels.
There is no CPU fallback: a missing library or a CPU tensor raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE = range(5)
GDN_F32, GDN_BF16 = 0, 1
PATHS = {"auto": 0, "staged": 1, "fused": 2, "cp": 3, "fused1": 4}
PATH_NAMES = {v: k for k, v in PATHS.items()}
DEV_OK, DEV_BAD_CU_SEQLENS, DEV_WAIT_TIMEOUT = 0, 1, 2
STAGES = {"prepare": 0, "cumsum": 1, "kkt": 2, "solve_tril": 3, "wy_fast": 4, "chunk_h": 5, "chunk_o": 6}

EXPORTED = ["gdn_chunk_fwd_workspace_size", "gdn_chunk_fwd", "gdn_chunk_fwd_staged", "gdn_staged_layout",
            "gdn_get_device_status", "gdn_resolve_path", "gdn_status_string", "gdn_version", "gdn_recurrent_fwd",
            "gdn_causal_conv1d_fwd", "gdn_chunk_bwd_workspace_size", "gdn_chunk_bwd",
            "gdn_chunk_bwd_get_device_status", "gdn_chunk_fwd_host_workspace_size", "gdn_chunk_fwd_host",
            "gdn_chunk_fwd_host_get_device_status"]


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("N", ctypes.c_int), ("Hqk", ctypes.c_int),
                ("Hv", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int), ("C", ctypes.c_int),
                ("dt", ctypes.c_int), ("varlen", ctypes.c_int)]


class StagedLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("tables", "status", "gamma", "A", "Tinv", "W", "U", "S0", "Vn",
                                               "total")] + [("nc_max", ctypes.c_int)]


class GDNError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libgdn.so")


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgdn.so (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libgdn.so not built ({path}); run __graft_entry__.build()")
            from . import build as _build
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(Problem)
        vp, fp, i32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        lib.gdn_chunk_fwd_workspace_size.argtypes = [P, ctypes.c_int]
        lib.gdn_chunk_fwd_workspace_size.restype = ctypes.c_size_t
        call = [P, ctypes.c_int, vp, vp, vp, fp, fp, ctypes.c_float, fp, i32p, vp, fp, vp, ctypes.c_size_t, vp]
        lib.gdn_chunk_fwd.argtypes = call
        lib.gdn_chunk_fwd.restype = ctypes.c_int
        lib.gdn_chunk_fwd_staged.argtypes = call
        lib.gdn_chunk_fwd_staged.restype = ctypes.c_int
        lib.gdn_staged_layout.argtypes = [P, ctypes.POINTER(StagedLayout)]
        lib.gdn_staged_layout.restype = ctypes.c_int
        lib.gdn_get_device_status.argtypes = [P, ctypes.c_int, vp, vp, ctypes.POINTER(ctypes.c_int)]
        lib.gdn_get_device_status.restype = ctypes.c_int
        lib.gdn_resolve_path.argtypes = [P]
        lib.gdn_resolve_path.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_recurrent_fwd.argtypes = [P, vp, vp, vp, fp, fp, fp, fp, ctypes.c_float, fp, i32p, ctypes.c_int,
                                          i32p, vp, vp]
        lib.gdn_recurrent_fwd.restype = ctypes.c_int
        lib.gdn_causal_conv1d_fwd.argtypes = [vp, fp, fp, ctypes.c_int, vp, ctypes.c_int, i32p, i32p, i32p,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, vp, vp]
        lib.gdn_causal_conv1d_fwd.restype = ctypes.c_int
        lib.gdn_chunk_bwd_workspace_size.argtypes = [P]
        lib.gdn_chunk_bwd_workspace_size.restype = ctypes.c_size_t
        lib.gdn_chunk_bwd.argtypes = [P, vp, vp, vp, fp, fp, ctypes.c_float, fp, i32p, vp, fp, fp, fp, fp, fp, fp, fp,
                                      vp, ctypes.c_size_t, vp]
        lib.gdn_chunk_bwd.restype = ctypes.c_int
        lib.gdn_chunk_bwd_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
        lib.gdn_chunk_bwd_get_device_status.restype = ctypes.c_int
        lib.gdn_chunk_fwd_host_workspace_size.argtypes = [P, i32p, ctypes.c_int, ctypes.c_int]
        lib.gdn_chunk_fwd_host_workspace_size.restype = ctypes.c_size_t
        lib.gdn_chunk_fwd_host.argtypes = [P, ctypes.c_int, ctypes.c_int, vp, vp, vp, fp, fp, ctypes.c_float, fp, i32p,
                                           vp, fp, vp, ctypes.c_size_t, vp]
        lib.gdn_chunk_fwd_host.restype = ctypes.c_int
        lib.gdn_chunk_fwd_host_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
        lib.gdn_chunk_fwd_host_get_device_status.restype = ctypes.c_int
        lib.gdn_version.argtypes = []
        lib.gdn_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(s: int) -> str:
    return load().gdn_status_string(int(s)).decode()


def gdn_version() -> str:
    return load().gdn_version().decode()


@dataclass
class Shapes:
    B: int
    T: int
    N: int
    Hqk: int
    Hv: int
    K: int
    V: int


def problem(B, T, N, Hqk, Hv, K, V, C, dtype, varlen) -> Problem:
    dt = GDN_F32 if dtype in (torch.float32, "f32", GDN_F32) else GDN_BF16
    return Problem(int(B), int(T), int(N), int(Hqk), int(Hv), int(K), int(V), int(C), dt, int(bool(varlen)))


def problem_of(q, v, C, cu_seqlens=None) -> Problem:
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    return problem(B, T, N, Hqk, Hv, K, V, C, q.dtype, cu_seqlens is not None)


def gdn_chunk_fwd_workspace_size(p: Problem, path: str = "auto") -> int:
    return int(load().gdn_chunk_fwd_workspace_size(ctypes.byref(p), PATHS[path]))


def gdn_resolve_path(p: Problem) -> str:
    return PATH_NAMES[int(load().gdn_resolve_path(ctypes.byref(p)))]


def gdn_staged_layout(p: Problem) -> StagedLayout:
    out = StagedLayout()
    st = load().gdn_staged_layout(ctypes.byref(p), ctypes.byref(out))
    if st:
        raise GDNError(st, "gdn_staged_layout")
    return out


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p()


def _check_inputs(q, k, v, g, beta, h0, cu_seqlens):
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0), ("cu_seqlens", cu_seqlens)):
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dtype not in (torch.float32, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float32 or bfloat16")
    for name, t in (("g", g), ("beta", beta), ("h0", h0)):
        if t is not None and t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    if k.shape != q.shape or v.shape[:2] != (B, T) or g.shape != (B, T, Hv) or beta.shape != (B, T, Hv):
        raise ValueError("shape mismatch among q, k, v, g, beta")
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if h0 is not None and h0.shape != (N, Hv, K, V):
        raise ValueError(f"h0 must be [N, Hv, K, V] = {(N, Hv, K, V)}")


def _alloc_ws(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks.
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def gdn_chunk_fwd(q, k, v, g, beta, scale: Optional[float] = None, h0=None, cu_seqlens=None, C: int = 64,
                  path: str = "auto", o=None, ht=None, output_final_state: bool = True, workspace=None,
                  stream=None):
    """Chunked Gated DeltaNet forward.  Returns (o, ht); ht is None when
    ``output_final_state`` is False.  ``scale`` defaults to K ** -0.5."""
    lib = load()
    _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    p = problem_of(q, v, C, cu_seqlens)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if o is None:
        o = torch.empty_like(v)
    if ht is None and output_final_state:
        ht = torch.empty((p.N, p.Hv, p.K, p.V), dtype=torch.float32, device=q.device)
    need = gdn_chunk_fwd_workspace_size(p, path)
    if need == 0:
        raise GDNError(GDN_ERR_UNSUPPORTED if path in ("fused", "cp", "fused1") else GDN_ERR_INVALID_ARG, "gdn_chunk_fwd_workspace_size")
    if workspace is None:
        workspace = _alloc_ws(need, q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    st = lib.gdn_chunk_fwd(ctypes.byref(p), PATHS[path], _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           ctypes.c_float(scale), _ptr(h0), _ptr(cu_seqlens), _ptr(o), _ptr(ht), _ptr(workspace),
                           ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(s))
    if st:
        raise GDNError(st, "gdn_chunk_fwd")
    return o, ht


def gdn_chunk_fwd_host_workspace_size(p: Problem, cu_seqlens=None, nsplit: int = 4, path: str = "auto") -> int:
    return int(load().gdn_chunk_fwd_host_workspace_size(ctypes.byref(p), _ptr(cu_seqlens), int(nsplit), PATHS[path]))


def gdn_chunk_fwd_host(q, k, v, g, beta, scale: Optional[float] = None, h0=None, cu_seqlens=None, C: int = 64,
                       path: str = "auto", nsplit: int = 4, o=None, ht=None, output_final_state: bool = True,
                       workspace=None, device=None, stream=None):
    """The forward pass on host (CPU) tensors, streamed through the GPU in
    ``nsplit`` sub-batches (pin the tensors for the copies to overlap the
    compute).  Returns host (o, ht) after the call has finished; ht is None
    when ``output_final_state`` is False."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("h0", h0), ("cu_seqlens", cu_seqlens)):
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous host tensor")
    p = problem_of(q, v, C, cu_seqlens)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    pin = q.is_pinned()
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, pin_memory=pin)
    if ht is None and output_final_state:
        ht = torch.empty((p.N, p.Hv, p.K, p.V), dtype=torch.float32, pin_memory=pin)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = gdn_chunk_fwd_host_workspace_size(p, cu_seqlens, nsplit, path)
    if need == 0:
        raise GDNError(GDN_ERR_INVALID_ARG, "gdn_chunk_fwd_host_workspace_size")
    if workspace is None:
        workspace = _alloc_ws(need, dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
    st = lib.gdn_chunk_fwd_host(ctypes.byref(p), PATHS[path], int(nsplit), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), ctypes.c_float(scale), _ptr(h0), _ptr(cu_seqlens), _ptr(o), _ptr(ht),
                                _ptr(workspace), ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(s))
    if st:
        raise GDNError(st, "gdn_chunk_fwd_host")
    torch.cuda.synchronize(dev)
    return o, ht


def gdn_chunk_fwd_host_get_device_status(workspace, stream=None) -> int:
    out = ctypes.c_int(0)
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device).cuda_stream
    st = load().gdn_chunk_fwd_host_get_device_status(_ptr(workspace), ctypes.c_void_p(s), ctypes.byref(out))
    if st:
        raise GDNError(st, "gdn_chunk_fwd_host_get_device_status")
    return out.value


def gdn_chunk_fwd_staged(q, k, v, g, beta, scale: Optional[float] = None, h0=None, cu_seqlens=None, C: int = 64,
                         stop_after: int | str = 6, workspace=None, stream=None):
    """Staged path up to ``stop_after``; returns (o, ht, workspace, layout)."""
    lib = load()
    _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    p = problem_of(q, v, C, cu_seqlens)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    stop = STAGES[stop_after] if isinstance(stop_after, str) else int(stop_after)
    layout = gdn_staged_layout(p)
    o = torch.zeros_like(v)
    ht = torch.zeros((p.N, p.Hv, p.K, p.V), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _alloc_ws(layout.total, q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    st = lib.gdn_chunk_fwd_staged(ctypes.byref(p), stop, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  ctypes.c_float(scale), _ptr(h0), _ptr(cu_seqlens), _ptr(o), _ptr(ht),
                                  _ptr(workspace), ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(s))
    if st:
        raise GDNError(st, "gdn_chunk_fwd_staged")
    return o, ht, workspace, layout


def staged_view(workspace: torch.Tensor, layout: StagedLayout, p: Problem, name: str) -> torch.Tensor:
    """A typed view of one staged intermediate inside ``workspace``."""
    nc, H, C, K, V = layout.nc_max, p.Hv, p.C, p.K, p.V
    shapes = {"gamma": (nc, H, C), "A": (nc, H, C, C), "Tinv": (nc, H, C, C), "W": (nc, H, C, K),
              "U": (nc, H, C, V), "S0": (nc, H, K, V), "Vn": (nc, H, C, V)}
    if name == "tables":
        n = p.N + 1 + 3 * nc + 1
        t = workspace[layout.tables: layout.tables + 4 * n].view(torch.int32)
        return {"seq_chunk0": t[: p.N + 1], "chunk_seq": t[p.N + 1: p.N + 1 + nc],
                "chunk_tok0": t[p.N + 1 + nc: p.N + 1 + 2 * nc], "chunk_len": t[p.N + 1 + 2 * nc: p.N + 1 + 3 * nc],
                "nc": t[-1:]}
    shape = shapes[name]
    off = getattr(layout, name)
    numel = 1
    for d in shape:
        numel *= d
    return workspace[off: off + 4 * numel].view(torch.float32).view(shape)


def gdn_get_device_status(p: Problem, path: str, workspace: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int(0)
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device).cuda_stream
    st = load().gdn_get_device_status(ctypes.byref(p), PATHS[path], _ptr(workspace), ctypes.c_void_p(s),
                                      ctypes.byref(out))
    if st:
        raise GDNError(st, "gdn_get_device_status")
    return int(out.value)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=True,
                           cu_seqlens=None, chunk_size: int = 64):
    """Framework-style entry: (o, final_state) like the pages' integration call."""
    return gdn_chunk_fwd(q, k, v, g, beta, scale=scale, h0=initial_state, cu_seqlens=cu_seqlens, C=chunk_size,
                         output_final_state=output_final_state)


def gdn_recurrent_fwd(q, k, v, a, b, A_log, state, dt_bias=None, scale: Optional[float] = None,
                      state_indices=None, cu_seqlens=None, o=None, stream=None):
    """Fused gated recurrent (decode) step.  ``state`` [slots, Hv, K, V] fp32 is
    updated in place; returns o.  g = -exp(A_log) softplus(a + dt_bias),
    beta = sigmoid(b), then the gated delta rule token by token."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("A_log", A_log), ("state", state),
                    ("dt_bias", dt_bias), ("state_indices", state_indices), ("cu_seqlens", cu_seqlens)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    for name, t in (("a", a), ("b", b), ("A_log", A_log), ("state", state), ("dt_bias", dt_bias)):
        if t is not None and t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    p = problem_of(q, v, 64, cu_seqlens)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if o is None:
        o = torch.empty_like(v)
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    st = lib.gdn_recurrent_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                               _ptr(dt_bias), ctypes.c_float(scale), _ptr(state), _ptr(state_indices),
                               int(state.shape[0]), _ptr(cu_seqlens), _ptr(o), ctypes.c_void_p(s))
    if st:
        raise GDNError(st, "gdn_recurrent_fwd")
    return o


ACTIVATIONS = {None: 0, "none": 0, "silu": 1}
DTYPES = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16}


def gdn_causal_conv1d_fwd(x, weight, bias=None, activation="silu", conv_state=None, cache_indices=None,
                          has_initial_state=None, cu_seqlens=None, y=None, stream=None):
    """Causal depthwise convolution with a carried state.  x [B, T, D] (bf16
    or fp32; packed with cu_seqlens when B == 1), weight [D, W] fp32, bias [D]
    fp32.  ``conv_state`` [slots, W-1, D] (dtype of x) is read and then
    updated in place; returns y (shape and dtype of x)."""
    lib = load()
    for name, t in (("x", x), ("weight", weight), ("bias", bias), ("conv_state", conv_state),
                    ("cache_indices", cache_indices), ("has_initial_state", has_initial_state),
                    ("cu_seqlens", cu_seqlens)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    for name, t in (("weight", weight), ("bias", bias)):
        if t is not None and t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32")
    for name, t in (("cache_indices", cache_indices), ("has_initial_state", has_initial_state),
                    ("cu_seqlens", cu_seqlens)):
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    if x.dtype not in DTYPES:
        raise ValueError("x must be float32 or bfloat16")
    if conv_state is not None and conv_state.dtype != x.dtype:
        raise ValueError("conv_state must have the dtype of x")
    B, T, D = x.shape
    W = int(weight.shape[1])
    N = int(cu_seqlens.numel()) - 1 if cu_seqlens is not None else B
    if y is None:
        y = torch.empty_like(x)
    slots = int(conv_state.shape[0]) if conv_state is not None else 0
    s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
    st = lib.gdn_causal_conv1d_fwd(_ptr(x), _ptr(weight), _ptr(bias), W, _ptr(conv_state), slots,
                                   _ptr(cache_indices), _ptr(has_initial_state), _ptr(cu_seqlens), N, B, T, D,
                                   DTYPES[x.dtype], ACTIVATIONS[activation], _ptr(y), ctypes.c_void_p(s))
    if st:
        raise GDNError(st, "gdn_causal_conv1d_fwd")
    return y


def gdn_chunk_bwd_workspace_size(p: Problem) -> int:
    return int(load().gdn_chunk_bwd_workspace_size(ctypes.byref(p)))


def gdn_chunk_bwd(q, k, v, g, beta, dout, scale: Optional[float] = None, h0=None, dht=None, cu_seqlens=None,
                  want_dh0: bool = True, workspace=None, stream=None) -> dict:
    """Backward of gdn_chunk_fwd for upstream gradients ``dout`` (dL/do, dtype of v)
    and ``dht`` (dL/dht, fp32 or None).  Returns fp32 gradients dq, dk
    [B,T,Hqk,K], dv [B,T,Hv,V], dg, dbeta [B,T,Hv] and dh0 [N,Hv,K,V] (None
    unless ``want_dh0``), plus the workspace under "workspace"."""
    lib = load()
    _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    for name, t in (("dout", dout), ("dht", dht)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dout.dtype != v.dtype or dout.shape != v.shape:
        raise ValueError("dout must match v in shape and dtype")
    if dht is not None and dht.dtype != torch.float32:
        raise ValueError("dht must be float32")
    p = problem_of(q, v, 64, cu_seqlens)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    need = gdn_chunk_bwd_workspace_size(p)
    if need == 0:
        raise GDNError(GDN_ERR_UNSUPPORTED, "gdn_chunk_bwd_workspace_size")
    if workspace is None:
        workspace = _alloc_ws(need, q.device)
    f32 = dict(dtype=torch.float32, device=q.device)
    out = {"dq": torch.empty(q.shape, **f32), "dk": torch.empty(k.shape, **f32), "dv": torch.empty(v.shape, **f32),
           "dg": torch.empty(g.shape, **f32), "dbeta": torch.empty(beta.shape, **f32),
           "dh0": torch.empty((p.N, p.Hv, p.K, p.V), **f32) if want_dh0 else None}
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    st = lib.gdn_chunk_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
                           _ptr(h0), _ptr(cu_seqlens), _ptr(dout), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]),
                           _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]),
                           _ptr(workspace), ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(s))
    if st:
        raise GDNError(st, "gdn_chunk_bwd")
    out["workspace"] = workspace
    return out


def gdn_chunk_bwd_get_device_status(workspace, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device).cuda_stream
    v = ctypes.c_int(0)
    st = load().gdn_chunk_bwd_get_device_status(_ptr(workspace), ctypes.c_void_p(s), ctypes.byref(v))
    if st:
        raise GDNError(st, "gdn_chunk_bwd_get_device_status")
    return int(v.value)
