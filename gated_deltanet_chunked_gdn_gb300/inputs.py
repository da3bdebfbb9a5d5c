"""Seeded synthetic inputs for the Gated DeltaNet chunked forward pass.

This module holds only input recipes (random draws, normalisation of the
draws, rounding to the storage dtype); none of the operator's arithmetic.  It
is the one module shared by the CUDA path's tests/benchmarks and by the CPU
oracle's tests.

Workloads (all synthetic; the pages measure a kernel bench of 16 sequences x
8192 tokens with H in {16, 32, 48, 64} -- MegaGDN-PTO walkthrough, "quick
start" bench command and the latency bar chart of the introduction):

====  ==================  ===========================================================
id    name                shape
====  ==================  ===========================================================
0     tiny_fp32           B=1, T=256, Hqk=Hv=2, K=V=64, C=64, fp32, h0 ~ N(0, 0.1)
1     gqa_prefill         B=1, T=4096, Hqk=16, Hv=32, K=V=128, C=64, bf16, h0 = None
2     batched_16x8192     B=16, T=8192, Hqk=Hv=H (16/32/48/64), K=V=128, C=128, bf16,
                          h0 ~ N(0, 0.1)
3     varlen_64           64 packed sequences, lengths log-uniform in [1, 16384],
                          Hqk=16, Hv=32, K=V=128, C=64, bf16, h0 ~ N(0, 0.1)
4     long_d256           B=4, T=32768, Hqk=8, Hv=32, K=V=256, C=64, bf16, h0 = None
====  ==================  ===========================================================

Value distributions: q, k ~ N(0, 1), then L2-normalised per (token, head) in
fp32 before rounding; v ~ N(0, 1); beta = sigmoid(N(0, 1)); g (a log-decay,
<= 0) = logsigmoid(N(0, 1)) / 4 for workload 0 and -softplus(N(0, 1)) *
exp(U(-4, 0)) otherwise; h0 ~ N(0, 0.1) (std 0.1).  g, beta and h0 are fp32;
q, k, v are rounded to the workload's dtype (round-to-nearest-even).
scale = K ** -0.5.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hqk: int
    Hv: int
    K: int
    V: int
    C: int
    dtype: str            # "f32" or "bf16"
    gate: str             # "logsigmoid4" or "softplus_exp"
    h0: bool              # random initial state, else None
    seed: int
    varlen_n: int = 0     # > 0: packed batch of this many sequences (B must be 1)
    varlen_max: int = 16384

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    0: Workload("tiny_fp32", 1, 256, 2, 2, 64, 64, 64, "f32", "logsigmoid4", True, 0),
    1: Workload("gqa_prefill", 1, 4096, 16, 32, 128, 128, 64, "bf16", "softplus_exp", False, 1),
    2: Workload("batched_16x8192", 16, 8192, 32, 32, 128, 128, 128, "bf16", "softplus_exp", True, 2),
    3: Workload("varlen_64", 1, 0, 16, 32, 128, 128, 64, "bf16", "softplus_exp", True, 3, varlen_n=64),
    4: Workload("long_d256", 4, 32768, 8, 32, 256, 256, 64, "bf16", "softplus_exp", False, 4),
}


def varlen_lengths(n: int, seed: int, max_len: int = 16384) -> list[int]:
    """Sequence lengths log-uniform in [1, max_len] (rounded, clamped).

    If the draw holds no length below 64 (shorter than one chunk) or none of at
    least max_len / 2, the first (resp. last) drawn length is replaced by 17
    (resp. max_len / 2 + 123) so that both regimes are always present.
    """
    gen = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.rand(n, generator=gen, dtype=torch.float64) * math.log(max_len)
    lens = [min(max(int(round(math.exp(x))), 1), max_len) for x in u.tolist()]
    if n >= 2 and not any(L < 64 for L in lens):
        lens[0] = 17
    if n >= 2 and not any(L >= max_len // 2 for L in lens):
        lens[-1] = max_len // 2 + 123
    return lens


def _normal(shape, gen, device, std=1.0):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32) * std


def make_inputs(w: Workload, device: str | torch.device = "cpu", lengths: Optional[list[int]] = None) -> dict:
    """Draw the inputs of workload ``w`` on ``device`` (the torch generator of
    that device, seeded with ``w.seed``; CPU and CUDA streams differ).

    Returns q, k [B,T,Hqk,K]; v [B,T,Hv,V]; g, beta [B,T,Hv] fp32; h0
    [N,Hv,K,V] fp32 or None; cu_seqlens int32 [N+1] or None; scale; C; N.
    """
    device = torch.device(device)
    if w.varlen_n > 0:
        lens = lengths if lengths is not None else varlen_lengths(w.varlen_n, w.seed, w.varlen_max)
        B, T, N = 1, int(sum(lens)), len(lens)
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    else:
        B, T, N, cu = w.B, w.T, w.B, None
    gen = torch.Generator(device=device).manual_seed(w.seed)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    q = _normal((B, T, w.Hqk, w.K), gen, device)
    q = (q / q.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(dt)
    k = _normal((B, T, w.Hqk, w.K), gen, device)
    k = (k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(dt)
    v = _normal((B, T, w.Hv, w.V), gen, device).to(dt)
    if w.gate == "logsigmoid4":
        g = torch.nn.functional.logsigmoid(_normal((B, T, w.Hv), gen, device)) / 4
    else:
        base = torch.nn.functional.softplus(_normal((B, T, w.Hv), gen, device))
        u = torch.rand((B, T, w.Hv), generator=gen, device=device, dtype=torch.float32) * 4.0 - 4.0
        g = -base * torch.exp(u)
    beta = torch.sigmoid(_normal((B, T, w.Hv), gen, device))
    h0 = _normal((N, w.Hv, w.K, w.V), gen, device, std=0.1) if w.h0 else None
    return {
        "q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(),
        "g": g.contiguous(), "beta": beta.contiguous(), "h0": h0,
        "cu_seqlens": cu.to(device) if cu is not None else None,
        "scale": w.K ** -0.5, "C": w.C, "N": N,
    }


def conv_channels(Hqk: int, Hv: int, K: int, V: int) -> int:
    """Channels of the convolution in front of a GDN layer: the q, k and v
    projections side by side (2 Hqk K + Hv V)."""
    return 2 * Hqk * K + Hv * V


def make_conv_inputs(B: int, T: int, D: int, W: int, dtype: str, device="cpu", seed: int = 0,
                     lengths: Optional[list[int]] = None, slots: Optional[int] = None) -> dict:
    """Inputs of the causal convolution with a carried state: x ~ N(0, 1)
    [B, T, D] (or packed [1, sum(lengths), D] with cu_seqlens), weight ~
    N(0, 1/W) [D, W] fp32, bias ~ N(0, 0.1) [D] fp32, conv_state ~ N(0, 1)
    [slots, W-1, D] (slots defaults to the number of sequences), x and the
    state rounded to ``dtype``."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    cu = None
    if lengths is not None:
        B, T, N = 1, int(sum(lengths)), len(lengths)
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    else:
        N = B
    S = N if slots is None else slots
    x = _normal((B, T, D), gen, device).to(dt)
    weight = _normal((D, W), gen, device, std=W ** -0.5)
    bias = _normal((D,), gen, device, std=0.1)
    state = _normal((S, max(W - 1, 0), D), gen, device).to(dt)
    return {"x": x.contiguous(), "weight": weight.contiguous(), "bias": bias.contiguous(),
            "conv_state": state.contiguous(), "cu_seqlens": cu.to(device) if cu is not None else None, "N": N}
