"""fp64 CPU oracle for the Gated DeltaNet forward pass -- TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA library
(``gated_deltanet_chunked_gdn_gb300``) and never imports it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, OpenMP over
independent (sequence, value-head) chains); this file builds it with gcc and
marshals numpy arrays.  Forms:

* :func:`recurrent` -- the token recurrence (the operator's definition).
* :func:`chunked` -- the chunked form with an explicit Gauss-Jordan inverse.
* :func:`chunked_stages` -- the chunked form of one chain, returning every
  per-chunk intermediate (gamma, A, T, W, U, S0, V').
* :func:`recurrent_bwd` -- gradients of the token recurrence (reverse mode).

Tensor conventions (same as the library): q, k ``[B, T, Hqk, K]``;
v ``[B, T, Hv, V]``; g, beta ``[B, T, Hv]``; h0 / ht ``[N, Hv, K, V]``;
with ``cu_seqlens`` (length N+1) the batch is packed and B must be 1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_build/libgdn_oracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    common = [ctypes.c_int64, ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.oracle_recurrent.argtypes = common + [dp] * 5 + [ctypes.c_double, dp, dp, dp, i32p, ctypes.c_int, ctypes.c_int]
    lib.oracle_recurrent.restype = ctypes.c_int
    lib.oracle_chunked.argtypes = common + [ctypes.c_int] + [dp] * 5 + [ctypes.c_double, dp, dp, dp, i32p, ctypes.c_int, ctypes.c_int]
    lib.oracle_chunked.restype = ctypes.c_int
    lib.oracle_chunked_stages.argtypes = (common + [ctypes.c_int] + [dp] * 5 + [ctypes.c_double, dp, ctypes.c_int, ctypes.c_int]
                                          + [dp] * 9)
    lib.oracle_chunked_stages.restype = ctypes.c_int
    lib.oracle_recurrent_bwd.argtypes = common + [dp] * 5 + [ctypes.c_double] + [dp] * 9 + [ctypes.c_int]
    lib.oracle_recurrent_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


class Oracle:
    """The same entry points bound to another build of gdn_oracle.c (used by
    the mutation tests, which compile copies with a planted mistake)."""

    def __init__(self, so_path: str):
        self._lib = _bind(ctypes.CDLL(so_path))

    def recurrent(self, *a, **kw):
        return recurrent(*a, _lib=self._lib, **kw)

    def chunked(self, *a, **kw):
        return chunked(*a, _lib=self._lib, **kw)

    def recurrent_bwd(self, *a, **kw):
        return recurrent_bwd(*a, _lib=self._lib, **kw)


def _f64(x):
    if x is None:
        return None
    try:  # torch tensors (bf16 included) without importing torch here
        import torch  # noqa: WPS433 (local import keeps numpy-only callers light)
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", dtype=torch.float64).numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _prep(q, k, v, g, beta, h0, cu_seqlens):
    q, k, v, g, beta, h0 = (_f64(t) for t in (q, k, v, g, beta, h0))
    B, T, Hqk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    if cu_seqlens is None:
        N = B
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        cu = _i64(cu_seqlens)
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        N = cu.shape[0] - 1
    return q, k, v, g, beta, h0, cu, B, T, Hqk, K, Hv, V, N


def _chains(chains):
    if chains is None:
        return ctypes.POINTER(ctypes.c_int32)(), 0, None
    arr = np.ascontiguousarray(np.asarray(chains, dtype=np.int32))
    return arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(arr.shape[0]), arr


def recurrent(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chains=None, nthreads=0, _lib=None):
    """Token recurrence. Returns (o [B,T,Hv,V], ht [N,Hv,K,V]) as float64.

    ``chains``: optional list of chain ids ``n * Hv + h``; other chains' outputs
    are left as NaN.
    """
    q, k, v, g, beta, h0, cu, B, T, Hqk, K, Hv, V, N = _prep(q, k, v, g, beta, h0, cu_seqlens)
    o = np.full((B, T, Hv, V), np.nan if chains is not None else 0.0)
    ht = np.full((N, Hv, K, V), np.nan if chains is not None else 0.0)
    cp, nc, _keep = _chains(chains)
    rc = (_lib or _load()).oracle_recurrent(B * T, N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hqk, Hv, K, V,
                                  _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(h0),
                                  _ptr(o), _ptr(ht), cp, nc, int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_recurrent failed: {rc}")
    return o, ht


def recurrent_bwd(q, k, v, g, beta, scale, dout, h0=None, dht=None, cu_seqlens=None, nthreads=0, _lib=None):
    """Gradients of the token recurrence for upstream gradients ``dout``
    (dL/do, [B,T,Hv,V]) and ``dht`` (dL/dht, [N,Hv,K,V] or None).  Returns a
    dict of float64 arrays: dq, dk [B,T,Hqk,K]; dv [B,T,Hv,V]; dg, dbeta
    [B,T,Hv]; dh0 [N,Hv,K,V] (the gradient w.r.t. the initial state, zero
    state when h0 is None)."""
    q, k, v, g, beta, h0, cu, B, T, Hqk, K, Hv, V, N = _prep(q, k, v, g, beta, h0, cu_seqlens)
    do = _f64(dout)
    dh = _f64(dht)
    out = {"dq": np.zeros((B, T, Hqk, K)), "dk": np.zeros((B, T, Hqk, K)), "dv": np.zeros((B, T, Hv, V)),
           "dg": np.zeros((B, T, Hv)), "dbeta": np.zeros((B, T, Hv)), "dh0": np.zeros((N, Hv, K, V))}
    rc = (_lib or _load()).oracle_recurrent_bwd(B * T, N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hqk, Hv,
                                                K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                                _ptr(h0), _ptr(do), _ptr(dh), _ptr(out["dq"]), _ptr(out["dk"]),
                                                _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                                                _ptr(out["dh0"]), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_recurrent_bwd failed ({rc})")
    return out


def chunked(q, k, v, g, beta, scale, C, h0=None, cu_seqlens=None, chains=None, nthreads=0, _lib=None):
    """Naive chunked form (explicit inverse). Returns (o, ht) as float64."""
    q, k, v, g, beta, h0, cu, B, T, Hqk, K, Hv, V, N = _prep(q, k, v, g, beta, h0, cu_seqlens)
    o = np.full((B, T, Hv, V), np.nan if chains is not None else 0.0)
    ht = np.full((N, Hv, K, V), np.nan if chains is not None else 0.0)
    cp, nc, _keep = _chains(chains)
    rc = (_lib or _load()).oracle_chunked(B * T, N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hqk, Hv, K, V, int(C),
                                _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(h0),
                                _ptr(o), _ptr(ht), cp, nc, int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_chunked failed: {rc}")
    return o, ht


def chunked_stages(q, k, v, g, beta, scale, C, n, h, h0=None, cu_seqlens=None):
    """Chunked form of chain (n, h) with its per-chunk intermediates.

    Returns a dict with gamma [NT,C], A [NT,C,C], T [NT,C,C], W [NT,C,K],
    U [NT,C,V], S0 [NT,K,V], Vn [NT,C,V] (rows past a tail chunk's length are
    zero), plus o [B,T,Hv,V] (this chain's rows only) and ht [N,Hv,K,V].
    """
    q, k, v, g, beta, h0, cu, B, T, Hqk, K, Hv, V, N = _prep(q, k, v, g, beta, h0, cu_seqlens)
    L = int(cu[n + 1] - cu[n])
    NT = max(1, -(-L // C))
    out = {
        "gamma": np.zeros((NT, C)), "A": np.zeros((NT, C, C)), "T": np.zeros((NT, C, C)),
        "W": np.zeros((NT, C, K)), "U": np.zeros((NT, C, V)), "S0": np.zeros((NT, K, V)),
        "Vn": np.zeros((NT, C, V)),
    }
    o = np.full((B, T, Hv, V), np.nan)
    ht = np.full((N, Hv, K, V), np.nan)
    rc = _load().oracle_chunked_stages(B * T, N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hqk, Hv, K, V,
                                       int(C), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                       _ptr(h0), int(n), int(h), _ptr(o), _ptr(ht),
                                       *(_ptr(out[key]) for key in ("gamma", "A", "T", "W", "U", "S0", "Vn")))
    if rc:
        raise RuntimeError(f"oracle_chunked_stages failed: {rc}")
    out["o"], out["ht"] = o, ht
    return out


def gated_recurrent(q, k, v, a, b, A_log, dt_bias, scale, state, state_indices=None, cu_seqlens=None):
    """Decode-phase gated delta rule (the fused sigmoid-gating recurrent step of
    the TileLang x xLLM page): per token and value head
        g = -exp(A_log[h]) * softplus(a + dt_bias[h]),  beta = sigmoid(b),
    then the token recurrence from each sequence's slot of ``state``
    ([slots, Hv, K, V]).  Sequences whose slot is negative or out of range get
    zero outputs and leave the state untouched.  Returns (o, new_state), fp64.
    """
    a64, b64, A64 = _f64(a), _f64(b), _f64(A_log)
    d64 = _f64(dt_bias) if dt_bias is not None else np.zeros_like(A64)
    st = _f64(state)
    x = a64 + d64[None, None, :]
    g = -np.exp(A64)[None, None, :] * np.logaddexp(0.0, x)      # softplus(x) = log(1 + e^x)
    beta = 1.0 / (1.0 + np.exp(-b64))                            # sigmoid
    Bq = _f64(q).shape[0]
    N = (len(_i64(cu_seqlens)) - 1) if cu_seqlens is not None else Bq
    slots = _i64(state_indices) if state_indices is not None else np.arange(N)
    valid = (slots >= 0) & (slots < st.shape[0])
    h0 = np.zeros((N,) + st.shape[1:])
    h0[valid] = st[slots[valid]]
    o, ht = recurrent(q, k, v, g, beta, scale, h0=h0, cu_seqlens=cu_seqlens)
    new_state = st.copy()
    new_state[slots[valid]] = ht[valid]
    cu = _i64(cu_seqlens) if cu_seqlens is not None else None
    for n in np.nonzero(~valid)[0]:
        if cu is None:
            o[n] = 0.0
        else:
            o[0, cu[n]:cu[n + 1]] = 0.0
    return o, new_state


def causal_conv1d(x, weight, bias=None, activation="silu", conv_state=None, cache_indices=None,
                  has_initial_state=None, cu_seqlens=None):
    """Causal depthwise 1-D convolution with a carried convolution state (the
    causal_conv1d operator of the TileLang x xLLM page: each output token
    depends on the current and earlier tokens of its own sequence only; the
    last W-1 inputs are kept per sequence in ``conv_state`` for incremental
    decode; ``cache_indices`` picks each sequence's slot of the state pool).

    Shapes: x ``[B, T, D]`` (packed with ``cu_seqlens`` when B == 1),
    weight ``[D, W]``, bias ``[D]`` or None, conv_state ``[slots, W-1, D]``.
    For a sequence with inputs x_0..x_{L-1}, prepend its W-1 initial inputs
    (the slot's state when the sequence has one, zeros otherwise) to get
    ext_0..ext_{L+W-2}; then

        y_p[d] = act(bias[d] + sum_{w<W} weight[d, w] ext_{p+w}[d]),
        new state = ext_L .. ext_{L+W-2}   (the last W-1 inputs),

    with act = identity or SiLU (u * sigmoid(u)).  A sequence whose slot is
    negative has no state: zeros are prepended and no state is written.
    ``has_initial_state[n] == 0`` prepends zeros but still writes the slot.
    Returns (y fp64 [B, T, D], new conv_state fp64 or None).
    """
    xs, w = _f64(x), _f64(weight)
    B, T, D = xs.shape
    W = w.shape[1]
    b = _f64(bias) if bias is not None else np.zeros(D)
    if cu_seqlens is None:
        seqs = [(n, 0, T) for n in range(B)]
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = _i64(cu_seqlens)
        seqs = [(0, int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]
    st = _f64(conv_state) if conv_state is not None else None
    new_state = st.copy() if st is not None else None
    slots = _i64(cache_indices) if cache_indices is not None else np.arange(len(seqs))
    init_flag = _i64(has_initial_state) if has_initial_state is not None else np.ones(len(seqs), dtype=np.int64)
    y = np.zeros_like(xs)
    for n, (bi, s, e) in enumerate(seqs):
        L = e - s
        slot = int(slots[n]) if st is not None else -1
        init = np.zeros((W - 1, D))
        if slot >= 0 and init_flag[n] != 0:
            init = st[slot]
        ext = np.concatenate([init, xs[bi, s:e]], axis=0)
        acc = np.tile(b, (L, 1))
        for j in range(W):
            acc += w[:, j][None, :] * ext[j:j + L]
        if activation == "silu":
            acc = acc / (1.0 + np.exp(-acc))
        elif activation not in (None, "none"):
            raise ValueError(activation)
        y[bi, s:e] = acc
        if slot >= 0:
            new_state[slot] = ext[L:L + W - 1]
    return y, new_state
