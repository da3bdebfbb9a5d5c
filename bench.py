#!/usr/bin/env python
"""Throughput of the Gated DeltaNet chunked forward pass on GB300.

Workload: the pages' kernel bench shape -- 16 sequences x 8192 tokens,
Hqk = Hv = 32 (``--H``), K = V = 128, chunk C = 128, bf16 q/k/v/o, fp32
g/beta/h0/ht, synthetic seeded inputs generated on the device (4.4 GB of
compulsory traffic per step, far larger than the 129 MB L2, so no flush is
needed between steps).

One step = one ``gdn_chunk_fwd`` call over the whole batch (all stages of the
hot path).  Prints ONE JSON line (rank 0).  Multi-GPU (torchrun): every rank
runs its own independent batch (weak scaling, no data-path collective); the
timed region is bracketed by barriers and the max over ranks is reported.

``--impl reference`` times the fp64 CPU oracle on the host cores instead
(bounded samples of the same workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN chunk-fwd tokens/s (16x8192, H=32, K=V=128, bf16); % roofline"
L2_BYTES = 129 * 1000 * 1000   # GB300 L2


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def measured_traffic(op: str, units: float, fixed_bytes: float = 0.0):
    """DRAM bytes (read + write) per launch of op's kernels, from the committed
    ncu summary table (profiles/traffic.json); None when any of the kernels'
    sources changed since that capture.

    One formula: traffic = fixed_bytes + (D - F) * units / U, where D is the
    captured launch's DRAM bytes, U its size in units (sequences of 8192
    tokens, or pool entries for decode) and F the bytes of that launch that do
    not grow with its size (the record's ``fixed_bytes``: initial and final
    states); fixed_bytes is the same for the bench's own launch.  A capture
    taken at the bench's own size (units == U, F == fixed_bytes) is used as
    it is."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[op]
        for src, want in rec["sources"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != want:
                    return None
    except (OSError, KeyError, ValueError):
        return None
    F = float(rec.get("fixed_bytes", 0.0))
    return fixed_bytes + (rec["dram_bytes_per_launch"] - F) * units / rec["units"]


def algorithmic(B, T, Hqk, Hv, K, V, C, elem=2, h0=True, N=None):
    """Compulsory bytes and algorithmic FLOPs of one forward pass over B x T
    tokens in N sequences (N = B unless packed).

    Bytes: q, k, v, o in the input dtype, g and beta fp32, h0 and ht fp32.
    FLOPs (triangular products counted as half, KK^T / QK^T once per qk head):
    per token Hqk*(C*K + C*K) + Hv*(C*V + C*K + C*V + 6*K*V + C*C/3).
    """
    tokens = B * T
    N = B if N is None else N
    per_tok = 2 * Hqk * K * elem + 2 * Hv * V * elem + 8 * Hv
    state = N * Hv * K * V * 4 * (2 if h0 else 1)
    nbytes = tokens * per_tok + state
    flops = tokens * (Hqk * 2 * C * K + Hv * (2 * C * V + C * K + 6 * K * V + C * C / 3))
    return nbytes, flops


class ClockSampler:
    """nvidia-smi sampler for SM clocks, power and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        if self.error or not self.samples:
            return {"error": self.error or "no samples"}
        win = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15] or [self.samples[-1][1]]
        sm = [float(p[1]) for p in win if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in win if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        pw = [float(p[3]) for p in win if p[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win), "power_w_max": max(pw) if pw else None}


def aggregate(elapsed_s: float, tokens_per_rank_step: int, steps: int, world: int, device=None) -> tuple:
    """Whole-job throughput under weak scaling: every rank processed its own
    ``tokens_per_rank_step * steps`` tokens; the job took the slowest rank's
    time (max over ranks).  Returns (value tokens/s, max elapsed s)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_s = float(t.item())
    return world * tokens_per_rank_step * steps / elapsed_s, elapsed_s


def gpu_uuid(dev: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:  # noqa: BLE001 - fall back to the ordinal
        return str(dev)


def cpu_oracle_sample(x: dict, w, nthreads: int, budget_s: float, n_chains: int | None = None) -> dict:
    """Time the fp64 oracle on whole (sequence, head) chains of ``x``.

    With ``n_chains`` unset, one chain is first timed on one thread and the
    sample is sized to about ``budget_s`` CPU-seconds (a multiple of the
    thread count, at most every chain of ``x``).
    """
    from oracle import oracle
    oracle.build()
    H = w.Hv
    Bx = x["q"].shape[0]
    if x.get("cu_seqlens") is not None:
        return cpu_oracle_sample_packed(oracle, x, w, nthreads, budget_s)
    if n_chains is None:
        s0 = {k: x[k][0:1].cpu() for k in ("q", "k", "v", "g", "beta")}
        h0 = x["h0"][0:1].cpu() if x["h0"] is not None else None
        t = time.perf_counter()
        oracle.recurrent(s0["q"], s0["k"], s0["v"], s0["g"], s0["beta"], x["scale"], h0=h0, chains=[0], nthreads=1)
        t1 = time.perf_counter() - t
        n = max(1, int(budget_s / max(t1, 1e-3)))      # budget in CPU-seconds
        n = max(1, (n // nthreads) * nthreads) if n >= nthreads else n
    else:
        n = n_chains
    n = min(n, Bx * H)
    nseq = math.ceil(n / H)
    sub = {k: x[k][:nseq].cpu() for k in ("q", "k", "v", "g", "beta")}
    hs = x["h0"][:nseq].cpu() if x["h0"] is not None else None
    t = time.perf_counter()
    oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], x["scale"], h0=hs,
                     chains=list(range(n)), nthreads=nthreads)
    wall = time.perf_counter() - t
    tokens = n * w.T / H        # token positions of all Hv heads
    return {"value": tokens / wall, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n} (sequence, head) chains of {w.T} tokens of the {w.B}x{w.T} H={H} workload, "
                      f"fp64 recurrence, {nthreads} threads, {wall:.2f} s wall",
            "wall_s": wall, "chains": n}


def cpu_oracle_sample_packed(oracle, x: dict, w, nthreads: int, budget_s: float) -> dict:
    """The oracle on whole (sequence, head) chains of a packed batch, taken in
    (sequence, head) order until about ``budget_s`` CPU-seconds of work, sized
    from one chain of the longest sequence timed on one thread; tokens are
    counted as in the metric (token positions of all Hv heads)."""
    H = w.Hv
    cu = x["cu_seqlens"].cpu().tolist()
    lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    host = {k: x[k].cpu() for k in ("q", "k", "v", "g", "beta")}
    h0 = x["h0"].cpu() if x["h0"] is not None else None
    cuc = x["cu_seqlens"].cpu()
    nmax = max(range(len(lens)), key=lambda i: lens[i])
    t = time.perf_counter()
    oracle.recurrent(host["q"], host["k"], host["v"], host["g"], host["beta"], x["scale"], h0=h0, cu_seqlens=cuc,
                     chains=[nmax * H], nthreads=1)
    per_tok = (time.perf_counter() - t) / max(lens[nmax], 1)
    want = budget_s / max(per_tok, 1e-9)       # chain-tokens the budget buys
    chains, ctoks = [], 0
    for c in range(len(lens) * H):
        if ctoks >= want:
            break
        chains.append(c)
        ctoks += lens[c // H]
    t = time.perf_counter()
    oracle.recurrent(host["q"], host["k"], host["v"], host["g"], host["beta"], x["scale"], h0=h0, cu_seqlens=cuc,
                     chains=chains, nthreads=nthreads)
    wall = time.perf_counter() - t
    tokens = ctoks / H
    return {"value": tokens / wall, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{len(chains)} (sequence, head) chains ({ctoks} chain-tokens) of the packed "
                      f"{len(lens)}-sequence workload, fp64 recurrence, {nthreads} threads, {wall:.2f} s wall",
            "wall_s": wall, "chains": len(chains)}


def run_reference(args, rank: int, world: int) -> None:
    if rank != 0:
        return
    import torch
    from gated_deltanet_chunked_gdn_gb300 import inputs as I
    w = I.WORKLOADS[2].with_(Hqk=args.H, Hv=args.H)
    nthreads = os.cpu_count() or 1
    # Each step: one chain per host thread, drawn from the same recipe (only
    # the sequences the sample needs are generated).
    nseq = math.ceil(nthreads / w.Hv)
    x = I.make_inputs(w.with_(B=nseq), "cpu")
    for _ in range(args.warmup):
        cpu_oracle_sample(x, w, nthreads, 0.0, n_chains=nthreads)
    vals, walls = [], []
    for _ in range(args.steps):
        r = cpu_oracle_sample(x, w, nthreads, 0.0, n_chains=nthreads)
        vals.append(r["value"])
        walls.append(r["wall_s"])
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.median(walls),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"batched_{w.B}x8192_H{args.H}", "B": w.B, "T": w.T, "Hqk": w.Hqk, "Hv": w.Hv,
                   "K": w.K, "V": w.V, "C": w.C, "sample": r["sample"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    del torch
    print(json.dumps(line), flush=True)


def timed(step, steps, world, dev, stream):
    """Time `steps` calls of step() with CUDA events on `stream`, clocks
    sampled meanwhile; returns (seconds over all steps, max over ranks, clocks)."""
    import torch
    import torch.distributed as dist
    sampler = ClockSampler(gpu_uuid(dev.index or 0))
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()
    return ev0.elapsed_time(ev1) / 1000.0, sampler.summary(t_wall0, t_wall1)


def hbm_roofline(nbytes: float, sec_per_launch: float, kernel: str, traffic=None) -> dict:
    pk = peaks()
    achieved = nbytes / sec_per_launch / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic, "peak_source": pk["source"], "kernel": kernel,
            "alg_bytes": nbytes, "t_hbm_ms": 1e3 * nbytes / (pk["hbm_gbs"] * 1e9)}


def run_conv1d(args, rank, world, dev):
    """Causal conv1d in front of a 32-head GDN layer: 16 x 8192 tokens,
    D = 2*32*128 + 32*128 channels, W = 4, SiLU, bf16, a 16-slot state pool.
    One step = one gdn_causal_conv1d_fwd call (convolution + state update)."""
    import torch
    from gated_deltanet_chunked_gdn_gb300 import binding
    from gated_deltanet_chunked_gdn_gb300 import inputs as I
    B, T, W = args.B, 8192, 4
    D = I.conv_channels(32, 32, 128, 128)
    d = I.make_conv_inputs(B, T, D, W, "bf16", device=dev, seed=2 + rank)
    y = torch.empty_like(d["x"])
    stream = torch.cuda.current_stream(dev)

    def step(x=d["x"]):
        binding.gdn_causal_conv1d_fwd(x, d["weight"], d["bias"], "silu", conv_state=d["conv_state"], y=y,
                                      stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sec, clocks = timed(step, args.steps, world, dev, stream)
    value, sec_total = aggregate(sec, B * T, args.steps, world, dev)
    sec_step = sec_total / args.steps
    nbytes = 2 * (B * T * D * 2) + D * W * 4 + D * 4 + 2 * B * (W - 1) * D * 2
    x_host = d["x"].cpu().pin_memory()
    y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    x_dev = torch.empty_like(d["x"])

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        step(x_dev)
        y_host.copy_(y, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(time.perf_counter() - t0, B * T, args.e2e_steps, world, dev)
    line = {
        "metric": "causal conv1d tokens/s (16x8192, D=12288, W=4, SiLU, bf16); % roofline", "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"conv1d_{B}x{T}_D{D}_W{W}", "B": B, "T": T, "D": D, "W": W, "activation": "silu",
                   "parallelism": f"dp{world} (independent batches)",
                   "l2": f"inputs larger than L2 ({nbytes / 1e9:.1f} GB compulsory traffic per step)"},
        "roofline": hbm_roofline(nbytes, sec_step, "conv1d_kernel + conv1d_state_kernel (one step)",
                                 traffic=measured_traffic("conv1d", B * T / 8192)),
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": x_host.numel() * 2,
                "d2h_bytes_per_step": y_host.numel() * 2, "steps": args.e2e_steps},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle as O
        xs, ws_, bs_, st_ = d["x"][0].cpu(), d["weight"].cpu(), d["bias"].cpu(), d["conv_state"][:1].cpu()
        Ds, done, t0 = 512, 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds:
            c = (done * Ds) % D
            O.causal_conv1d(xs[None, :, c:c + Ds], ws_[c:c + Ds], bs_[c:c + Ds], "silu", conv_state=st_[:, :, c:c + Ds])
            done += 1
        el = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": done * T * Ds / D / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{done} blocks of {T} tokens x {Ds} channels of sequence 0"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_decode(args, rank, world, dev):
    """Gated decode step: 512 sequences x 1 token, Hqk = Hv = 32, K = V = 128,
    bf16 q/k/v/o, fp32 state pool (2 GB read + written per step, larger than
    L2).  One step = one gdn_recurrent_fwd call."""
    import torch
    from gated_deltanet_chunked_gdn_gb300 import binding
    N, H, K = 512, 32, 128
    gen = torch.Generator(device=dev).manual_seed(2 + rank)
    rn = lambda *s_, dt=torch.float32: torch.randn(*s_, generator=gen, device=dev, dtype=torch.float32).to(dt)
    q = torch.nn.functional.normalize(rn(N, 1, H, K), dim=-1).to(torch.bfloat16)
    k = torch.nn.functional.normalize(rn(N, 1, H, K), dim=-1).to(torch.bfloat16)
    v = rn(N, 1, H, K, dt=torch.bfloat16)
    a, b_ = rn(N, 1, H), rn(N, 1, H)
    A_log, dt_bias = rn(H) * 0.5, rn(H) * 0.1
    state = rn(N, H, K, K) * 0.1
    o = torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.gdn_recurrent_fwd(q, k, v, a, b_, A_log, state, dt_bias=dt_bias, o=o, stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sec, clocks = timed(step, args.steps, world, dev, stream)
    value, sec_total = aggregate(sec, N, args.steps, world, dev)
    sec_step = sec_total / args.steps
    nbytes = 2 * N * H * K * K * 4 + 4 * N * H * K * 2 + 2 * N * H * 4 + 2 * H * 4
    line = {
        "metric": "gated decode step tokens/s (512 seqs x 1 token, H=32, K=V=128, fp32 state); % roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode_{N}x1_H{H}", "N": N, "H": H, "K": K, "V": K,
                   "parallelism": f"dp{world} (independent batches)",
                   "l2": f"state pool larger than L2 ({nbytes / 1e9:.2f} GB per step)"},
        "roofline": hbm_roofline(nbytes, sec_step, "gdn_recurrent_kernel (the step's only launch)",
                                 traffic=measured_traffic("decode", N)),
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


BWDC_LAUNCHES = 34          # kernels of one sequence group of the chunked backward (gdn_bwdc.cu)
BWDC_GROUP_BYTES = 16 << 30  # the chunked backward's per-group workspace budget


def run_bwd(args, rank, world, dev):
    """Backward pass on the 16 x 8192, 32-head batch (bf16 inputs, fp32
    gradients).  One step = one gdn_chunk_bwd call (the chunked backward for
    this equal-length K = V = 128 batch, in sequence groups).  Algorithmic
    FLOPs per (token, value head): one forward step of the recurrence (4 K V)
    and one reverse step (16 K V)."""
    import torch
    from gated_deltanet_chunked_gdn_gb300 import binding
    from gated_deltanet_chunked_gdn_gb300 import inputs as I
    packed = args.workload == "varlen_64"
    if packed:
        w = I.WORKLOADS[3].with_(seed=3 + rank)
    else:
        w = I.WORKLOADS[2].with_(B=args.B, Hqk=args.H, Hv=args.H, seed=2 + rank)
    x = I.make_inputs(w, dev)
    N = x["N"]
    gen = torch.Generator(device=dev).manual_seed(7 + rank)
    do = torch.randn(x["v"].shape, generator=gen, device=dev).to(x["v"].dtype)
    dht = torch.randn((N, w.Hv, w.K, w.V), generator=gen, device=dev)
    p = binding.problem_of(x["q"], x["v"], 64, x["cu_seqlens"])
    ws = torch.empty(binding.gdn_chunk_bwd_workspace_size(p), dtype=torch.uint8, device=dev)
    if packed:
        # one group with the chunk tables built on the device (the bound of this
        # batch, about 28 K (chunk, head) pairs, is within the packed budget)
        groups, launches = 1, BWDC_LAUNCHES + 1
    else:
        # sequence groups of the chunked backward: as many whole sequences as fit
        # its budget, from the workspace of one sequence
        p1 = binding.problem_of(x["q"][:1], x["v"][:1], 64)
        per_seq = binding.gdn_chunk_bwd_workspace_size(p1)
        group = max(1, min(w.B, BWDC_GROUP_BYTES // max(per_seq, 1)))
        groups, launches = -(-w.B // group), BWDC_LAUNCHES
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.gdn_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, scale=x["scale"], h0=x["h0"], dht=dht,
                              cu_seqlens=x["cu_seqlens"], workspace=ws, stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sec, clocks = timed(step, args.steps, world, dev, stream)
    tokens = x["q"].shape[0] * x["q"].shape[1]
    value, sec_total = aggregate(sec, tokens, args.steps, world, dev)
    sec_step = sec_total / args.steps
    flops = 20.0 * w.K * w.V * tokens * w.Hv
    in_bytes = sum(t.numel() * t.element_size() for t in (x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], do, dht)
                   if t is not None)
    achieved = flops / sec_step / 1e12
    # the products run on the tensor cores as tf32 (nominal dense tf32 : bf16 = 1.1 : 2.25 PFLOP/s);
    # a long step, so the sustained bf16 figure
    pk = peaks()
    tf32_peak = pk["bf16_tflops_sustained"] * 1.1 / 2.25
    line = {
        "metric": ("GDN backward tokens/s (varlen_64, Hqk=16, Hv=32, K=V=128, bf16 inputs, fp32 gradients)" if packed
                   else "GDN backward tokens/s (16x8192, H=32, K=V=128, bf16 inputs, fp32 gradients)"), "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": (f"bwd_varlen_{N}seqs_{tokens}tok_Hqk{w.Hqk}_Hv{w.Hv}" if packed
                                else f"bwd_{w.B}x{w.T}_H{w.Hv}"), "B": x["q"].shape[0], "T": x["q"].shape[1], "N": N,
                   "Hqk": w.Hqk, "Hv": w.Hv, "K": w.K,
                   "V": w.V, "parallelism": f"dp{world} (independent batches)",
                   "l2": f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB of inputs and upstream gradients per step)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tf32_peak, "unit": "TFLOP/s",
                     "frac": achieved / tf32_peak, "traffic": None,
                     "peak_source": f"measured bf16 sustained x nominal tf32/bf16 ratio ({pk['source']})",
                     "kernel": "chunked backward, all launches of one step (mma.sync tf32, three terms)",
                     "alg_flops": flops},
        "gpu_launches": launches * groups * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--H", type=int, default=32, choices=[16, 32, 48, 64])
    ap.add_argument("--path", default="auto", choices=["auto", "staged", "fused", "fused1"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-split", type=int, default=8,
                    help="sub-batches of the end-to-end leg (host buffers streamed through the GPU)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--B", type=int, default=16, help="batch override (profiling runs only; the metric is B=16)")
    ap.add_argument("--T", type=int, default=None,
                    help="sequence length override of the batched (8192) or long_d256 (32768) workload "
                         "(profiling runs only)")
    ap.add_argument("--workload", default="batched_16x8192",
                    choices=["batched_16x8192", "gqa_prefill_1x4096", "long_1x32768", "varlen_64", "long_d256"],
                    help="chunk_fwd shape: the headline 16 x 8192 batch, one long GQA sequence (1 x 4096 or "
                         "1 x 32768 tokens, 16 qk / 32 value heads), where AUTO takes the chunk-parallel path, "
                         "64 packed sequences of log-uniform lengths in [1, 16384] (16 qk / 32 value heads), or "
                         "the large-head-dim prefill: 4 x 32768 tokens, 8 qk / 32 value heads, K = V = 256")
    ap.add_argument("--op", default="chunk_fwd", choices=["chunk_fwd", "conv1d", "decode", "bwd"],
                    help="chunk_fwd: the GDN chunked forward (the headline); conv1d / decode: the neighbouring "
                         "ops of the same layer, each with its own JSON line")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from gated_deltanet_chunked_gdn_gb300 import binding
    from gated_deltanet_chunked_gdn_gb300 import inputs as I

    binding.load()
    if args.op != "chunk_fwd":
        {"conv1d": run_conv1d, "decode": run_decode, "bwd": run_bwd}[args.op](args, rank, world, dev)
        if world > 1:
            dist.destroy_process_group()
        return
    if args.workload == "batched_16x8192":
        w = I.WORKLOADS[2].with_(B=args.B, T=args.T or 8192, Hqk=args.H, Hv=args.H, seed=2 + rank)
        wname = f"batched_{w.B}x{w.T}_H{args.H}"
    elif args.workload == "varlen_64":
        w = I.WORKLOADS[3].with_(seed=3 + rank)
    elif args.workload == "long_d256":
        w = I.WORKLOADS[4].with_(T=args.T or 32768, seed=4 + rank)
        wname = f"long_d256_{w.B}x{w.T}_Hqk{w.Hqk}_Hv{w.Hv}"
    else:
        T = 4096 if args.workload == "gqa_prefill_1x4096" else 32768
        w = I.WORKLOADS[1].with_(T=T, seed=1 + rank)
        wname = f"gqa_prefill_1x{T}_Hqk{w.Hqk}_Hv{w.Hv}"
    x = I.make_inputs(w, dev)
    Bx, Tx = x["q"].shape[0], x["q"].shape[1]   # the packed batch is [1, total tokens]
    if args.workload == "varlen_64":
        wname = f"varlen_{x['N']}seqs_{Tx}tok_Hqk{w.Hqk}_Hv{w.Hv}"
    p = binding.problem_of(x["q"], x["v"], w.C, x["cu_seqlens"])
    path = args.path if args.path != "auto" else binding.gdn_resolve_path(p)
    o = torch.empty_like(x["v"])
    ht = torch.empty((p.N, p.Hv, p.K, p.V), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.gdn_chunk_fwd_workspace_size(p, path), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(q=x["q"], k=x["k"], v=x["v"], g=x["g"], beta=x["beta"], h0=x["h0"]):
        binding.gdn_chunk_fwd(q, k, v, g, beta, x["scale"], h0=h0, cu_seqlens=x["cu_seqlens"], C=w.C, path=path,
                              o=o, ht=ht, workspace=ws, stream=stream.cuda_stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st = binding.gdn_get_device_status(p, path, ws)
    if st != binding.DEV_OK:
        raise RuntimeError(f"device status {st} after warm-up")

    sampler = ClockSampler(gpu_uuid(local))
    sampler.start()
    time.sleep(0.3)
    # inputs smaller than about twice the L2 are timed step by step with the
    # L2 flushed (a 512 MB write) between steps, outside the timed spans
    in_bytes, _ = algorithmic(Bx, Tx, w.Hqk, w.Hv, w.K, w.V, w.C, 2, h0=x["h0"] is not None, N=x["N"])
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if in_bytes < 2 * L2_BYTES else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush is not None else 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    if flush is None:
        evs[0][0].record(stream)
        for _ in range(args.steps):
            step()
        evs[0][1].record(stream)
    else:
        for e_a, e_b in evs:
            flush.zero_()
            e_a.record(stream)
            step()
            e_b.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms = sum(e_a.elapsed_time(e_b) for e_a, e_b in evs)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    tokens_step = Bx * Tx
    value, sec_total = aggregate(ms / 1000.0, tokens_step, args.steps, world, dev)
    ms_step = 1000.0 * sec_total / args.steps

    # End to end through the public API: the C-ABI call on host buffers
    # (gdn_chunk_fwd_host: inputs in pinned host memory, the batch streamed
    # through the GPU in sub-batches whose copies overlap the compute, o and ht
    # back in host memory), every step.
    host = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    if x["h0"] is not None:
        host["h0"] = x["h0"].cpu().pin_memory()
    cu_host = x["cu_seqlens"].cpu() if x["cu_seqlens"] is not None else None
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    ht_host = torch.empty(ht.shape, dtype=ht.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * o_host.element_size() + ht_host.numel() * ht_host.element_size()
    p_host = binding.problem_of(host["q"], host["v"], w.C, cu_host)
    ws_host = torch.empty(binding.gdn_chunk_fwd_host_workspace_size(p_host, cu_host, args.e2e_split, path),
                          dtype=torch.uint8, device=dev)

    def e2e_step():
        binding.gdn_chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], x["scale"],
                                   h0=host.get("h0"), cu_seqlens=cu_host, C=w.C, path=path, nsplit=args.e2e_split,
                                   o=o_host, ht=ht_host, workspace=ws_host, device=dev,
                                   stream=stream.cuda_stream)

    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(time.perf_counter() - t0, tokens_step, args.e2e_steps, world, dev)

    pk = peaks()
    # the fused and chunk-parallel kernels run 64-token chunks whatever C the
    # call asks for (the result does not depend on C): their FLOPs are counted
    # at the chunk length they execute
    C_exec = 64 if path in ("fused", "fused1", "cp") else w.C
    nbytes, flops = algorithmic(Bx, Tx, w.Hqk, w.Hv, w.K, w.V, C_exec, 2, h0=x["h0"] is not None, N=x["N"])
    _, flops_req = algorithmic(Bx, Tx, w.Hqk, w.Hv, w.K, w.V, w.C, 2, h0=x["h0"] is not None, N=x["N"])
    state_bytes = x["N"] * w.Hv * w.K * w.V * 4 * (2 if x["h0"] is not None else 1)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    sec = ms_step / 1000.0
    if bound == "hbm":
        achieved, peak, unit = nbytes / sec / 1e9, pk["hbm_gbs"], "GB/s"
        peak_kind = "HBM copy"
    else:
        # a tensor-bound step is one long launch: the sustained bf16 figure
        achieved, peak, unit = flops / sec / 1e12, pk["bf16_tflops_sustained"], "TFLOP/s"
        peak_kind = "bf16 sustained"
    # a packed batch adds the longest-first ranking launch before a fused pass
    ranked = path in ("fused", "fused1") and x["cu_seqlens"] is not None and 1 < x["N"] <= 16384
    launches = {"staged": 7, "fused": 1, "fused1": 1, "cp": 4}[path] + (1 if ranked else 0)
    line = {
        "metric": METRIC if args.workload == "batched_16x8192" else f"GDN chunk-fwd tokens/s ({wname}, bf16); % roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wname, "B": Bx, "T": Tx, "N": x["N"], "Hqk": w.Hqk, "Hv": w.Hv,
                   "K": w.K, "V": w.V, "C": w.C, "C_executed": C_exec, "path": path,
                   "parallelism": f"dp{world} (independent batches)",
                   "l2": (f"inputs larger than L2 ({nbytes / 1e9:.2f} GB compulsory traffic per step)"
                          if flush is None else "L2 flushed (512 MB write) before every timed step")},
        "tflops_alg": flops / sec / 1e12,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": (measured_traffic("fused", w.B * w.T / 8192 * w.Hv / 32, state_bytes)
                                 if path == "fused" and args.workload == "batched_16x8192" else
                                 measured_traffic("fused1_d256", w.B * w.T / 32768, state_bytes)
                                 if path in ("fused", "fused1") and args.workload == "long_d256" else
                                 measured_traffic("fused1_varlen64", 1, state_bytes)
                                 if path == "fused1" and args.workload == "varlen_64" else
                                 measured_traffic({"gqa_prefill_1x4096": "cp_1x4096",
                                                   "long_1x32768": "cp_1x32768"}.get(args.workload, ""), 1)
                                 if path == "cp" else None),
                     "peak_source": f"{pk['source']} ({peak_kind})",
                     "kernel": (("gdn_fused1_kernel" if (w.K == 256 or path == "fused1") else "gdn_fused_kernel") +
                                (" (after the ranking launch of the packed batch)" if ranked
                                 else " (the step's only launch)")) if path in ("fused", "fused1")
                     else "gdn_chunk_fwd call (all launches of one step)",
                     "alg_bytes": nbytes, "alg_flops": flops, "alg_flops_at_requested_C": flops_req,
                     "t_hbm_ms": 1e3 * t_hbm, "t_tensor_ms": 1e3 * t_tc},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps, "call": f"gdn_chunk_fwd_host, {args.e2e_split} sub-batches"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k_: v_ for k_, v_ in cpu_oracle_sample(x, w, os.cpu_count() or 1,
                                                                       args.cpu_seconds).items()
                                if k_ in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
