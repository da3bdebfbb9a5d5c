"""GPU parity: the CUDA library against the fp64 oracle on the same seeded
inputs, through the C ABI (the Python binding only marshals arguments).

Bar (the operator's accuracy targets): relative Frobenius error on both o and ht of at
most 1e-4 for fp32 inputs and 5e-3 for bf16 inputs (fp32 state); chunk
tables bit-exact.
"""
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
    binding.load()
    return binding


# Reduced versions of the five workloads: several chunks, a ragged tail, GQA,
# empty and sub-chunk sequences, both head dims, both dtypes.
SMALL = {
    "tiny_fp32": (I.WORKLOADS[0], None),
    "gqa_prefill": (I.WORKLOADS[1].with_(T=300, Hqk=2, Hv=4), None),
    "batched_C128": (I.WORKLOADS[2].with_(B=2, T=333, Hqk=2, Hv=2), None),
    "varlen": (I.WORKLOADS[3].with_(Hqk=2, Hv=4), [5, 64, 200, 1, 0, 129, 63]),
    "long_d256": (I.WORKLOADS[4].with_(B=1, T=200, Hqk=1, Hv=4), None),
    "fp32_C128_gqa": (I.WORKLOADS[0].with_(B=2, T=150, Hqk=1, Hv=3, K=128, V=64, C=128), None),
}


def run_case(gdn, w, lens, path, device="cuda"):
    x = I.make_inputs(w, "cpu", lengths=lens)
    d = {k_: (v_.to(device) if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                              cu_seqlens=d["cu_seqlens"], C=w.C, path=path)
    torch.cuda.synchronize()
    return x, o.float().cpu().numpy(), ht.cpu().numpy()


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("path", ["staged", "auto"])
def test_parity_small(gdn, oracle_mod, name, path):
    w, lens = SMALL[name]
    x, o, ht = run_case(gdn, w, lens, path)
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                         cu_seqlens=x["cu_seqlens"])
    tol = TOL[w.dtype]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(ht))
    assert rel_fro(o, o_ref) <= tol, rel_fro(o, o_ref)
    assert rel_fro(ht, ht_ref) <= tol, rel_fro(ht, ht_ref)


def test_h0_none_and_ht_skipped(gdn, oracle_mod):
    w = I.WORKLOADS[1].with_(T=130, Hqk=1, Hv=2)
    x = I.make_inputs(w, "cpu")
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], C=w.C,
                              output_final_state=False)
    assert ht is None
    o_ref, _ = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"])
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]


def test_state_passing_on_gpu(gdn, oracle_mod):
    """run(T1) then run(T2, h0=ht) on the GPU equals the oracle on T1+T2."""
    w = I.WORKLOADS[2].with_(B=1, T=400, Hqk=2, Hv=2, C=128, dtype="f32")
    x = I.make_inputs(w, "cpu")
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    T1 = 150
    sl = lambda t, a, b_: t[:, a:b_].contiguous()
    o1, ht1 = gdn.gdn_chunk_fwd(*(sl(d[n], 0, T1) for n in ("q", "k", "v", "g", "beta")), d["scale"], h0=d["h0"],
                                C=w.C)
    o2, ht2 = gdn.gdn_chunk_fwd(*(sl(d[n], T1, 400) for n in ("q", "k", "v", "g", "beta")), d["scale"], h0=ht1,
                                C=w.C)
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"])
    o = torch.cat([o1, o2], dim=1).cpu().numpy()
    assert rel_fro(o, o_ref) <= TOL["f32"]
    assert rel_fro(ht2.cpu().numpy(), ht_ref) <= TOL["f32"]


def test_chunk_tables_bit_exact(gdn):
    """The prepare stage's chunk tables equal a host computation exactly."""
    lens = [5, 0, 64, 65, 1, 128, 300, 0, 63]
    C = 64
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=1, K=64, V=64, dtype="f32")
    x = I.make_inputs(w, "cuda", lengths=lens)
    _, _, ws, layout = gdn.gdn_chunk_fwd_staged(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                                cu_seqlens=x["cu_seqlens"], C=C, stop_after="prepare")
    torch.cuda.synchronize()
    p = gdn.problem_of(x["q"], x["v"], C, x["cu_seqlens"])
    t = {k_: v_.cpu().numpy() for k_, v_ in gdn.staged_view(ws, layout, p, "tables").items()}
    seq_chunk0, seqs, tok0, ln = [0], [], [], []
    off = 0
    for n, L in enumerate(lens):
        nch = -(-L // C)
        for j in range(nch):
            seqs.append(n)
            tok0.append(off + j * C)
            ln.append(min(C, L - j * C))
        seq_chunk0.append(seq_chunk0[-1] + nch)
        off += L
    nc = seq_chunk0[-1]
    assert int(t["nc"][0]) == nc
    assert t["seq_chunk0"].tolist() == seq_chunk0
    assert t["chunk_seq"][:nc].tolist() == seqs
    assert t["chunk_tok0"][:nc].tolist() == tok0
    assert t["chunk_len"][:nc].tolist() == ln


def test_malformed_cu_seqlens_sets_device_status(gdn):
    """Decreasing offsets are caught by the prepare kernel: the device status
    word reports it and no stage runs (the output stays untouched)."""
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2, K=64, V=64, dtype="f32")
    x = I.make_inputs(w, "cuda", lengths=[10, 20, 30])
    bad = torch.tensor([0, 25, 20, 60], dtype=torch.int32, device="cuda")
    o = torch.full_like(x["v"], 7.0)
    p = gdn.problem_of(x["q"], x["v"], 64, bad)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(p, "staged"), dtype=torch.uint8, device="cuda")
    gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], cu_seqlens=bad, C=64, path="staged",
                      o=o, workspace=ws)
    assert gdn.gdn_get_device_status(p, "staged", ws) == gdn.DEV_BAD_CU_SEQLENS
    assert torch.all(o == 7.0)
    # a good call on the same workspace clears it
    gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], cu_seqlens=x["cu_seqlens"], C=64,
                      path="staged", o=o, workspace=ws)
    assert gdn.gdn_get_device_status(p, "staged", ws) == gdn.DEV_OK


STAGE_KEYS = [("gamma", "gamma", 1), ("A", "A", 2), ("Tinv", "T", 3), ("W", "W", 4), ("U", "U", 4),
              ("S0", "S0", 5), ("Vn", "Vn", 5)]


@pytest.mark.parametrize("C", [64, 128])
def test_stage_intermediates_match_oracle(gdn, oracle_mod, C):
    """Each stage of the staged path, stopped right after it, against the
    chunked oracle's intermediates for every chain (fp32 inputs)."""
    lens = [C + 37, 2, 2 * C]
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2, K=64, V=64, C=C, dtype="f32")
    x = I.make_inputs(w, "cpu", lengths=lens)
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    p = gdn.problem_of(d["q"], d["v"], C, d["cu_seqlens"])
    for key, okey, stop in STAGE_KEYS:
        _, _, ws, layout = gdn.gdn_chunk_fwd_staged(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                                    h0=d["h0"], cu_seqlens=d["cu_seqlens"], C=C, stop_after=stop)
        torch.cuda.synchronize()
        got = gdn.staged_view(ws, layout, p, key).cpu().numpy()
        c0 = 0
        for n, L in enumerate(lens):
            nt = -(-L // C)
            for h in range(w.Hv):
                ref = oracle_mod.chunked_stages(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], C, n, h,
                                                h0=x["h0"], cu_seqlens=x["cu_seqlens"])[okey]
                g_ = got[c0:c0 + nt, h].copy()
                if key == "Tinv":
                    # past a tail chunk's length (I + A) is the identity, so
                    # its inverse holds 1 on the diagonal there
                    tail = L - (nt - 1) * C
                    diag = np.arange(tail, C)
                    assert np.all(g_[-1, diag, diag] == 1.0)
                    g_[-1, diag, diag] = 0.0
                err = rel_fro(g_, ref) if np.linalg.norm(ref) > 0 else np.abs(g_).max()
                assert err < 1e-4, (key, n, h, err)
            c0 += nt


# ------------------------------------------------------------- fused path

FUSED_CASES = {
    "fixed_C64_ragged": (I.WORKLOADS[1].with_(B=2, T=333, Hqk=2, Hv=4), None),
    "fixed_C128_request": (I.WORKLOADS[2].with_(B=2, T=300, Hqk=2, Hv=2), None),
    "varlen_short_and_empty": (I.WORKLOADS[3].with_(Hqk=1, Hv=2), [5, 64, 200, 1, 0, 129, 63, 65]),
    "single_token": (I.WORKLOADS[2].with_(B=3, T=1, Hqk=1, Hv=1), None),
    "gqa4_h0": (I.WORKLOADS[2].with_(B=1, T=130, Hqk=1, Hv=4, C=64), None),
    # 320 chains of 3 chunks (ragged last chunk) over more chains than the GPU
    # holds CTAs: windows of 4 chunks, most chains cut in two and handed over
    "windows_cut_chains": (I.WORKLOADS[2].with_(B=40, T=190, Hqk=4, Hv=8, C=64), None),
    # 150 packed sequences of 0..299 tokens (empty ones included), GQA 2 -> 4
    "varlen_many_short": (I.WORKLOADS[3].with_(Hqk=2, Hv=4),
                          [int(n) for n in np.random.default_rng(5).integers(0, 300, 150)]),
    # K = V = 256 (value slices of 128 columns): ragged tail with GQA 4, h0,
    # short and empty packed sequences, V = 128, and windows that cut units
    "d256_fixed_ragged_gqa4": (I.WORKLOADS[4].with_(B=2, T=333, Hqk=1, Hv=4), None),
    "d256_gqa4_h0": (I.WORKLOADS[4].with_(B=1, T=200, Hqk=2, Hv=8, h0=True), None),
    "d256_varlen_short_and_empty": (I.WORKLOADS[4].with_(B=1, T=0, Hqk=1, Hv=4, h0=True, varlen_n=8),
                                    [5, 64, 200, 1, 0, 129, 63, 65]),
    "d256_V128_h0": (I.WORKLOADS[4].with_(B=2, T=150, Hqk=2, Hv=4, V=128, h0=True), None),
    # 320 (chain, slice) units of 3 chunks over 152 SMs: windows of 7 chunks
    "d256_windows_cut_units": (I.WORKLOADS[4].with_(B=20, T=190, Hqk=2, Hv=8, h0=True), None),
    # K = 128 with V = 256: two value slices per chain on the one-CTA kernel only
    "k128_v256_gqa2": (I.WORKLOADS[2].with_(B=2, T=200, Hqk=1, Hv=2, V=256), None),
}
# cases that only the one-CTA kernel runs (GDN_PATH_FUSED does not take K = 128 with V = 256)
FUSED1_ONLY = {"k128_v256_gqa2"}


@pytest.mark.parametrize("name", sorted(FUSED_CASES))
@pytest.mark.parametrize("path", ["fused", "fused1"])
def test_fused_parity(gdn, oracle_mod, name, path):
    """Both fused kernels (two CTAs per SM, K = V = 128; one CTA per SM, K in
    {128, 256}) on every case; for K = 256 both paths run the one-CTA kernel."""
    w, lens = FUSED_CASES[name]
    x = I.make_inputs(w, "cpu", lengths=lens)
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    p = gdn.problem_of(d["q"], d["v"], w.C, d["cu_seqlens"])
    assert gdn.gdn_resolve_path(p) in ("fused", "fused1")
    if path == "fused" and name in FUSED1_ONLY:
        assert gdn.gdn_chunk_fwd_workspace_size(p, "fused") == 0   # rejected up front
        return
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(p, path), dtype=torch.uint8, device="cuda")
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                              cu_seqlens=d["cu_seqlens"], C=w.C, path=path, workspace=ws)
    assert gdn.gdn_get_device_status(p, path, ws) == gdn.DEV_OK
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                         cu_seqlens=x["cu_seqlens"])
    o, ht = o.float().cpu().numpy(), ht.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(ht))
    assert rel_fro(o, o_ref) <= TOL["bf16"], rel_fro(o, o_ref)
    assert rel_fro(ht, ht_ref) <= TOL["bf16"], rel_fro(ht, ht_ref)


def _gate_pattern(kind, B, T, H, gen):
    """Per-token log-decays g (<= 0) that put the fused kernel's gating into
    each of its regimes: a 32-row block whose exponents span little (row x
    column factors), one that spans a lot (an exponential per element), and
    a mix of the two inside one chunk."""
    r = torch.arange(T) % 64
    if kind == "strong":
        return -(1.0 + 5.0 * torch.rand(B, T, H, generator=gen))
    if kind == "weak_then_strong":
        return torch.where((r < 32)[None, :, None], -0.02 * torch.ones(B, T, H), -3.0 * torch.ones(B, T, H))
    if kind == "strong_then_weak":
        return torch.where((r < 32)[None, :, None], -3.0 * torch.ones(B, T, H), -0.02 * torch.ones(B, T, H))
    if kind == "no_decay":
        return torch.zeros(B, T, H)
    if kind == "near_span_limit":
        # about 60 binary orders of magnitude across each 32-row block
        return -(1.3 + 0.1 * torch.rand(B, T, H, generator=gen))
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["strong", "weak_then_strong", "strong_then_weak", "no_decay", "near_span_limit"])
@pytest.mark.parametrize("path", ["fused", "fused1"])
def test_fused_gate_regimes(gdn, oracle_mod, kind, path):
    w = I.WORKLOADS[2].with_(B=2, T=200, Hqk=2, Hv=2, C=64)
    x = I.make_inputs(w, "cpu")
    x["g"] = _gate_pattern(kind, w.B, w.T, w.Hv, torch.Generator().manual_seed(7)).float().contiguous()
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    o, ht = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], C=64,
                              path=path)
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"])
    o, ht = o.float().cpu().numpy(), ht.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(ht))
    assert rel_fro(o, o_ref) <= TOL["bf16"], rel_fro(o, o_ref)
    assert rel_fro(ht, ht_ref) <= TOL["bf16"], rel_fro(ht, ht_ref)


def test_fused_leaves_rows_of_other_sequences_untouched(gdn):
    """A tail chunk's padding rows belong to the next sequence: the fused
    kernel must not store them.  Sequence 1 is empty-output-checked by giving
    the call an o prefilled with a sentinel and zero-length sequences."""
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    lens = [70, 0, 10]
    x = I.make_inputs(w, "cuda", lengths=lens)
    o = torch.full_like(x["v"], 3.0)
    gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                      cu_seqlens=x["cu_seqlens"], C=64, path="fused", o=o)
    torch.cuda.synchronize()
    assert torch.all(o != 3.0)   # every row of the packed batch written exactly by its own sequence
    # sequence 0 alone reproduces its rows: rows 64..69 were not clobbered by chunk padding
    o0, _ = gdn.gdn_chunk_fwd(x["q"][:, :70].contiguous(), x["k"][:, :70].contiguous(), x["v"][:, :70].contiguous(),
                              x["g"][:, :70].contiguous(), x["beta"][:, :70].contiguous(), x["scale"],
                              h0=x["h0"][:1].contiguous(), C=64, path="fused")
    assert torch.equal(o0, o[:, :70])


@pytest.mark.parametrize("path", ["fused", "fused1"])
def test_fused_malformed_cu_seqlens(gdn, path):
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    x = I.make_inputs(w, "cuda", lengths=[10, 20, 30])
    # sequence 1 runs past the end of the batch, sequence 2 has a negative length
    bad = torch.tensor([0, 10, 70, 60], dtype=torch.int32, device="cuda")
    p = gdn.problem_of(x["q"], x["v"], 64, bad)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(p, path), dtype=torch.uint8, device="cuda")
    o = torch.full_like(x["v"], 7.0)
    gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], cu_seqlens=bad, C=64, path=path,
                      o=o, workspace=ws)
    assert gdn.gdn_get_device_status(p, path, ws) == gdn.DEV_BAD_CU_SEQLENS
    # the malformed sequences wrote nothing; the valid one wrote its rows
    assert torch.all(o[:, 10:] == 7.0)
    assert not torch.any(o[:, :10] == 7.0)


@pytest.mark.parametrize("path", ["fused", "fused1"])
def test_fused_matches_staged(gdn, path):
    """Fused and staged paths agree with each other (both against the same
    seeded inputs) -- a cross-check independent of the oracle."""
    w = I.WORKLOADS[1].with_(T=500, Hqk=2, Hv=4)
    x = I.make_inputs(w, "cuda")
    args = (x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"])
    of, hf = gdn.gdn_chunk_fwd(*args, C=64, path=path)
    os_, hs = gdn.gdn_chunk_fwd(*args, C=64, path="staged")
    torch.cuda.synchronize()
    assert rel_fro(of.float().cpu().numpy(), os_.float().cpu().numpy()) < 5e-3
    assert rel_fro(hf.cpu().numpy(), hs.cpu().numpy()) < 5e-3


@pytest.mark.parametrize("path,case", [("fused", "windows_cut_chains"), ("fused1", "windows_cut_chains"),
                                       ("fused1", "d256_windows_cut_units"), ("fused1", "varlen_many_short"),
                                       ("fused", "varlen_many_short")])
def test_fused_runs_are_bit_identical(gdn, path, case):
    """No chain's arithmetic depends on scheduling (which CTA runs it, where a
    window boundary cuts it, what runs beside it), so repeated calls must agree
    bit for bit; a race between warps or CTAs would show up here."""
    w, lens = FUSED_CASES[case]
    x = I.make_inputs(w, "cuda", lengths=lens)
    runs = []
    for _ in range(4):
        o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                  cu_seqlens=x["cu_seqlens"], C=w.C, path=path)
        torch.cuda.synchronize()
        runs.append((o.clone(), ht.clone()))
    for o, ht in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(ht, runs[0][1])


@pytest.mark.parametrize("path", ["fused", "fused1"])
def test_packed_batch_longest_first_order(gdn, oracle_mod, path):
    """Packed batches run their longest sequences first (a device-side ranking
    of cu_seqlens, two ranking blocks here: 300 sequences).  Every chain must
    still run exactly once: sampled chains against the oracle, and the batch
    with its sequences in reverse order gives the same o and ht bit for bit,
    sequence by sequence."""
    gen = np.random.default_rng(11)
    lens = [int(x) for x in gen.integers(0, 150, size=300)]
    lens[7], lens[150], lens[299] = 1500, 1499, 1500   # the longest, with a tie
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    x = I.make_inputs(w, "cuda", lengths=lens)
    cu = x["cu_seqlens"].cpu().tolist()
    o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], C=w.C, path=path)
    # the same sequences packed in reverse order
    idx = torch.cat([torch.arange(cu[n], cu[n + 1]) for n in reversed(range(len(lens)))]).to("cuda")
    cu_r = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu_r[1:] = torch.cumsum(torch.tensor(lens[::-1], dtype=torch.int64), 0).to(torch.int32)
    tok = lambda t: t[:, idx].contiguous()
    o_r, ht_r = gdn.gdn_chunk_fwd(tok(x["q"]), tok(x["k"]), tok(x["v"]), tok(x["g"]), tok(x["beta"]), x["scale"],
                                  h0=x["h0"].flip(0).contiguous(), cu_seqlens=cu_r.to("cuda"), C=w.C, path=path)
    torch.cuda.synchronize()
    assert torch.equal(o_r, tok(o)) and torch.equal(ht_r, ht.flip(0))
    for n, h in [(7, 0), (150, 1), (299, 0), (0, 1), (200, 0), (256, 1)]:
        sl = slice(cu[n], cu[n + 1])
        sub = lambda t, hh: t[:, sl, hh:hh + 1].contiguous().cpu()
        o_ref, ht_ref = oracle_mod.recurrent(sub(x["q"], 0), sub(x["k"], 0), sub(x["v"], h), sub(x["g"], h),
                                             sub(x["beta"], h), x["scale"], h0=x["h0"][n:n + 1, h:h + 1].cpu())
        if o_ref.size:
            assert rel_fro(o[:, sl, h:h + 1].float().cpu().numpy(), o_ref) <= TOL["bf16"], (n, h)
        assert rel_fro(ht[n:n + 1, h:h + 1].cpu().numpy(), ht_ref) <= TOL["bf16"], (n, h)


@pytest.mark.parametrize("N", [16384, 16385])
@pytest.mark.parametrize("path", ["fused", "fused1"])
def test_packed_batch_order_at_its_size_limit(gdn, oracle_mod, N, path):
    """The longest-first ranking covers up to 16384 sequences (64 ranking
    blocks); one more keeps the index order.  Both sides of the limit: the
    reversed packing gives the same outputs bit for bit, and sampled chains
    match the oracle."""
    gen = np.random.default_rng(N)
    lens = [int(x) for x in gen.integers(0, 9, size=N)]
    lens[N // 3] = 200   # one sequence of several chunks
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    x = I.make_inputs(w, "cuda", lengths=lens)
    cu = x["cu_seqlens"].cpu().tolist()
    o, ht = gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                              cu_seqlens=x["cu_seqlens"], C=w.C, path=path)
    idx = torch.cat([torch.arange(cu[n], cu[n + 1]) for n in reversed(range(N))]).to("cuda")
    cu_r = torch.zeros(N + 1, dtype=torch.int32)
    cu_r[1:] = torch.cumsum(torch.tensor(lens[::-1], dtype=torch.int64), 0).to(torch.int32)
    tok = lambda t: t[:, idx].contiguous()
    o_r, ht_r = gdn.gdn_chunk_fwd(tok(x["q"]), tok(x["k"]), tok(x["v"]), tok(x["g"]), tok(x["beta"]), x["scale"],
                                  h0=x["h0"].flip(0).contiguous(), cu_seqlens=cu_r.to("cuda"), C=w.C, path=path)
    torch.cuda.synchronize()
    assert torch.equal(o_r, tok(o)) and torch.equal(ht_r, ht.flip(0))
    for n, h in [(N // 3, 0), (N // 3, 1), (0, 1), (N - 1, 0), (N // 2, 1)]:
        sl = slice(cu[n], cu[n + 1])
        sub = lambda t, hh: t[:, sl, hh:hh + 1].contiguous().cpu()
        o_ref, ht_ref = oracle_mod.recurrent(sub(x["q"], 0), sub(x["k"], 0), sub(x["v"], h), sub(x["g"], h),
                                             sub(x["beta"], h), x["scale"], h0=x["h0"][n:n + 1, h:h + 1].cpu())
        if o_ref.size:
            assert rel_fro(o[:, sl, h:h + 1].float().cpu().numpy(), o_ref) <= TOL["bf16"], (n, h)
        assert rel_fro(ht[n:n + 1, h:h + 1].cpu().numpy(), ht_ref) <= TOL["bf16"], (n, h)
