"""GPU parity of the causal convolution with a carried state (GPU).

The CUDA kernels, called through the C ABI, against the fp64 oracle on the
same seeded inputs.  Bar: the outputs differ from the oracle by at most one
unit in the last place of the output dtype plus fp32 rounding (each output
is an fp32 sum rounded once: bf16 relative 2^-8, fp32 relative 1e-5); the
new convolution states are copies of inputs, so they are compared bit for
bit.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_chunked_gdn_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    binding.load()
    return binding


def assert_close(got, ref, dtype):
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    if dtype == "bf16":
        bound = 2.0 ** -8 * np.abs(ref) + 1e-6
    else:
        bound = 1e-5 * np.abs(ref) + 1e-6
    err = np.abs(got - ref)
    assert np.all(err <= bound), float((err / (bound + 1e-300)).max())


def run_both(gdn, oracle_mod, d, activation, **kw):
    """Run the GPU op on a copy of the inputs and the oracle on the originals."""
    xs = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    state_gpu = xs["conv_state"].clone() if kw.get("use_state", True) else None
    extra = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items() if k != "use_state"}
    y = gdn.gdn_causal_conv1d_fwd(xs["x"], xs["weight"], xs["bias"], activation, conv_state=state_gpu,
                                  cu_seqlens=xs["cu_seqlens"], **extra)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle_mod.causal_conv1d(d["x"], d["weight"], d["bias"], activation,
                                            conv_state=d["conv_state"] if kw.get("use_state", True) else None,
                                            cu_seqlens=d["cu_seqlens"],
                                            **{k: v for k, v in kw.items() if k != "use_state"})
    return y, state_gpu, y_ref, s_ref


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("activation", ["none", "silu"])
def test_conv1d_fixed_batch(gdn, oracle_mod, dtype, W, activation):
    # T = 150 spans several 64-token runs and a ragged tail; D = 48 a partial CTA
    d = I.make_conv_inputs(3, 150, 48, W, dtype, seed=W)
    y, st, y_ref, s_ref = run_both(gdn, oracle_mod, d, activation)
    assert_close(y, y_ref, dtype)
    if W > 1:
        assert torch.equal(st.cpu(), torch.from_numpy(s_ref).to(st.dtype))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv1d_varlen_slots(gdn, oracle_mod, dtype):
    """Packed sequences (empty, shorter than the window, straddling thread
    runs), a permuted slot map with one sequence without a slot, and one
    sequence that starts from zeros but still writes its slot."""
    lens = [5, 1, 0, 130, 2, 64, 65, 3]
    d = I.make_conv_inputs(1, 0, 64, 4, dtype, seed=3, lengths=lens, slots=10)
    idx = torch.tensor([9, 0, 2, -1, 5, 7, 3, 4], dtype=torch.int32)
    init = torch.tensor([1, 1, 1, 1, 0, 1, 1, 0], dtype=torch.int32)
    y, st, y_ref, s_ref = run_both(gdn, oracle_mod, d, "silu", cache_indices=idx, has_initial_state=init)
    assert_close(y, y_ref, dtype)
    assert torch.equal(st.cpu(), torch.from_numpy(s_ref).to(st.dtype))


def test_conv1d_runs_across_sequences(gdn, oracle_mod):
    """Packed sequences longer and shorter than a thread's 256-token run, so
    that runs start inside sequences and hold several whole ones."""
    lens = [300, 255, 257, 1, 0, 600, 10, 256, 40]
    d = I.make_conv_inputs(1, 0, 96, 4, "bf16", seed=12, lengths=lens)
    y, st, y_ref, s_ref = run_both(gdn, oracle_mod, d, "silu")
    assert_close(y, y_ref, "bf16")
    assert torch.equal(st.cpu(), torch.from_numpy(s_ref).to(st.dtype))


def test_conv1d_without_state(gdn, oracle_mod):
    d = I.make_conv_inputs(2, 70, 32, 4, "bf16", seed=5)
    y, _, y_ref, _ = run_both(gdn, oracle_mod, d, "silu", use_state=False)
    assert_close(y, y_ref, "bf16")


def test_conv1d_decode_continues_prefill(gdn, oracle_mod):
    """Prefill of 40 tokens, then 5 single-token decode calls on the same
    state pool, equal one oracle pass over 45 tokens."""
    d = I.make_conv_inputs(4, 45, 64, 4, "bf16", seed=8)
    x = d["x"].cuda()
    w, b = d["weight"].cuda(), d["bias"].cuda()
    st = d["conv_state"].cuda().clone()
    ys = [gdn.gdn_causal_conv1d_fwd(x[:, :40].contiguous(), w, b, "silu", conv_state=st)]
    for t in range(40, 45):
        ys.append(gdn.gdn_causal_conv1d_fwd(x[:, t:t + 1].contiguous(), w, b, "silu", conv_state=st))
    torch.cuda.synchronize()
    y_ref, s_ref = oracle_mod.causal_conv1d(d["x"], d["weight"], d["bias"], "silu", conv_state=d["conv_state"])
    assert_close(torch.cat(ys, dim=1), y_ref, "bf16")
    assert torch.equal(st.cpu(), torch.from_numpy(s_ref).to(st.dtype))


def test_conv1d_malformed_cu_seqlens(gdn):
    """A sequence running past the batch and one with a negative length are
    skipped: their rows and slots keep what they held."""
    d = I.make_conv_inputs(1, 0, 32, 4, "bf16", seed=9, lengths=[10, 20, 30])
    x, w = d["x"].cuda(), d["weight"].cuda()
    bad = torch.tensor([0, 10, 70, 60], dtype=torch.int32, device="cuda")
    st = d["conv_state"].cuda().clone()
    before = st.clone()
    y = torch.full_like(x, 7.0)
    gdn.gdn_causal_conv1d_fwd(x, w, None, "none", conv_state=st, cu_seqlens=bad, y=y)
    torch.cuda.synchronize()
    assert torch.all(y[:, 10:] == 7.0)
    assert not torch.any(y[:, :10] == 7.0)
    assert torch.equal(st[1:], before[1:])
    assert not torch.equal(st[0], before[0])


def test_conv1d_rejects_bad_arguments(gdn):
    x = torch.zeros(1, 4, 12, dtype=torch.bfloat16, device="cuda")   # D % 8 != 0
    w = torch.zeros(12, 4, device="cuda")
    with pytest.raises(gdn.GDNError):
        gdn.gdn_causal_conv1d_fwd(x, w, None, "none")
    x = torch.zeros(1, 4, 16, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(16, 5, device="cuda")                              # W > 4
    with pytest.raises(gdn.GDNError):
        gdn.gdn_causal_conv1d_fwd(x, w, None, "none")


def test_conv1d_full_size_sampled(gdn, oracle_mod):
    """The 16 x 8192-token batch of a 32-head GDN layer (D = 2*32*128 + 32*128
    channels, W = 4, SiLU, bf16) in one call, as bench.py times it; sampled
    channel blocks of every sequence are recomputed by the oracle."""
    D = I.conv_channels(32, 32, 128, 128)
    d = I.make_conv_inputs(16, 8192, D, 4, "bf16", device="cuda", seed=2)
    st = d["conv_state"].clone()
    y = gdn.gdn_causal_conv1d_fwd(d["x"], d["weight"], d["bias"], "silu", conv_state=st)
    torch.cuda.synchronize()
    for c in (0, 4096, D - 64):
        sl = slice(c, c + 64)
        y_ref, s_ref = oracle_mod.causal_conv1d(d["x"][:, :, sl].cpu(), d["weight"][sl].cpu(), d["bias"][sl].cpu(),
                                                "silu", conv_state=d["conv_state"][:, :, sl].cpu())
        assert_close(y[:, :, sl], y_ref, "bf16")
        assert torch.equal(st[:, :, sl].cpu(), torch.from_numpy(s_ref).to(st.dtype))


@pytest.mark.parametrize("i", range(12))
def test_conv1d_random_draw(gdn, oracle_mod, i):
    """Seeded draws of dtype, window, channel count, activation, packed or
    equal lengths (across thread runs), slot map and initial-state flags."""
    r = np.random.default_rng(6600 + i)
    dtype = "bf16" if r.random() < 0.6 else "f32"
    W = int(r.integers(1, 5))
    D = 8 * int(r.integers(1, 40))
    act = "silu" if r.random() < 0.7 else "none"
    kw = {}
    if r.random() < 0.5:
        n = int(r.integers(1, 8))
        lens = [int(x) for x in r.integers(0, 600, size=n)]
        slots = n + int(r.integers(0, 3))
        d = I.make_conv_inputs(1, 0, D, W, dtype, seed=40 + i, lengths=lens, slots=slots)
        perm = r.permutation(slots)[:n].astype(np.int32)
        perm[r.random(n) < 0.2] = -1
        kw["cache_indices"] = torch.from_numpy(perm)
        kw["has_initial_state"] = torch.from_numpy((r.random(n) < 0.7).astype(np.int32))
    else:
        d = I.make_conv_inputs(int(r.integers(1, 4)), int(r.integers(1, 700)), D, W, dtype, seed=40 + i)
    y, st, y_ref, s_ref = run_both(gdn, oracle_mod, d, act, **kw)
    assert_close(y, y_ref, dtype)
    if W > 1:
        assert torch.equal(st.cpu(), torch.from_numpy(s_ref).to(st.dtype))
