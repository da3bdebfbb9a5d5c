"""GPU parity of the fused gated recurrent (decode) step against the fp64
oracle: single-token decode over a state pool with slot indirection, several
tokens per packed sequence, both dtypes, all head dims, and a prefill (chunked
kernel) followed by decode steps against the recurrence over the whole
sequence."""
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


def gating_inputs(B, T, Hv, seed):
    gen = torch.Generator().manual_seed(seed)
    a = torch.randn(B, T, Hv, generator=gen)
    b = torch.randn(B, T, Hv, generator=gen)
    A_log = torch.randn(Hv, generator=gen) * 0.5 - 1.0
    dt_bias = torch.randn(Hv, generator=gen) * 0.1
    return a, b, A_log, dt_bias


@pytest.mark.parametrize("dtype,K", [("bf16", 128), ("f32", 64), ("bf16", 256), ("f32", 128)])
def test_decode_step_state_pool(gdn, oracle_mod, dtype, K):
    w = I.WORKLOADS[1].with_(B=5, T=1, Hqk=2, Hv=4, K=K, V=K, dtype=dtype)
    x = I.make_inputs(w, "cpu")
    a, b, A_log, dt_bias = gating_inputs(5, 1, 4, 7)
    gen = torch.Generator().manual_seed(8)
    pool = torch.randn(9, 4, K, K, generator=gen) * 0.1
    slots = torch.tensor([3, 0, -1, 8, 5], dtype=torch.int32)          # sequence 2 has no slot
    o_ref, pool_ref = oracle_mod.gated_recurrent(x["q"], x["k"], x["v"], a, b, A_log, dt_bias, x["scale"], pool,
                                                 state_indices=slots)
    dev = lambda t: t.cuda().contiguous()
    state = dev(pool)
    o = gdn.gdn_recurrent_fwd(dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(a), dev(b), dev(A_log), state,
                              dt_bias=dev(dt_bias), scale=x["scale"], state_indices=dev(slots))
    torch.cuda.synchronize()
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL[dtype]
    assert rel_fro(state.cpu().numpy(), pool_ref) <= 1e-5      # fp32 state, fp32 arithmetic
    assert torch.all(o[2].float() == 0)


def test_decode_multi_token_varlen(gdn, oracle_mod):
    lens = [3, 0, 5, 1]
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2, K=128, V=128)
    x = I.make_inputs(w, "cpu", lengths=lens)
    T = sum(lens)
    a, b, A_log, _ = gating_inputs(1, T, 2, 9)
    pool = torch.randn(4, 2, 128, 128, generator=torch.Generator().manual_seed(10)) * 0.1
    o_ref, pool_ref = oracle_mod.gated_recurrent(x["q"], x["k"], x["v"], a, b, A_log, None, x["scale"], pool,
                                                 cu_seqlens=x["cu_seqlens"])
    state = pool.cuda()
    o = gdn.gdn_recurrent_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), a.cuda(), b.cuda(), A_log.cuda(), state,
                              scale=x["scale"], cu_seqlens=x["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]
    assert rel_fro(state.cpu().numpy(), pool_ref) <= 1e-5


def test_prefill_then_decode_matches_recurrence(gdn, oracle_mod):
    """Fused chunked prefill of T tokens, then three decode steps on its final
    state, against the recurrence over all T + 3 tokens."""
    T, steps = 200, 3
    w = I.WORKLOADS[1].with_(B=2, T=T + steps, Hqk=2, Hv=4)
    x = I.make_inputs(w, "cpu")
    a, b, A_log, dt_bias = gating_inputs(2, steps, 4, 11)
    g_dec = -np.exp(A_log.double().numpy())[None, None, :] * np.logaddexp(0.0, (a + dt_bias).double().numpy())
    beta_dec = torch.sigmoid(b.double()).numpy()
    g_full = np.concatenate([x["g"][:, :T].double().numpy(), g_dec], axis=1)
    b_full = np.concatenate([x["beta"][:, :T].double().numpy(), beta_dec], axis=1)
    o_ref, ht_ref = oracle_mod.recurrent(x["q"], x["k"], x["v"], g_full, b_full, x["scale"])
    d = {k_: x[k_].cuda() for k_ in ("q", "k", "v", "g", "beta")}
    sl = lambda t, s0, s1: t[:, s0:s1].contiguous()
    o_pre, ht = gdn.gdn_chunk_fwd(sl(d["q"], 0, T), sl(d["k"], 0, T), sl(d["v"], 0, T), sl(d["g"], 0, T),
                                  sl(d["beta"], 0, T), x["scale"], C=64)
    outs = [o_pre]
    for t in range(steps):
        outs.append(gdn.gdn_recurrent_fwd(sl(d["q"], T + t, T + t + 1), sl(d["k"], T + t, T + t + 1),
                                          sl(d["v"], T + t, T + t + 1), a[:, t:t + 1].contiguous().cuda(),
                                          b[:, t:t + 1].contiguous().cuda(), A_log.cuda(), ht,
                                          dt_bias=dt_bias.cuda(), scale=x["scale"]))
    torch.cuda.synchronize()
    o = torch.cat(outs, dim=1).float().cpu().numpy()
    assert rel_fro(o, o_ref) <= TOL["bf16"]
    assert rel_fro(ht.cpu().numpy(), ht_ref) <= TOL["bf16"]


@pytest.mark.parametrize("i", range(12))
def test_decode_random_draw(gdn, oracle_mod, i):
    """Seeded draws of dtype, head dims, GQA ratio, pool size, slot map (with
    sequences that have no slot), tokens per sequence and dt_bias."""
    r = np.random.default_rng(6100 + i)
    dtype = "bf16" if r.random() < 0.6 else "f32"
    K = int(r.choice([64, 128, 256]))
    V = int(r.choice([64, 128])) if K != 256 else int(r.choice([128, 256]))
    Hqk = int(r.choice([1, 2]))
    Hv = Hqk * int(r.choice([1, 2, 4]))
    n = int(r.integers(1, 7))
    lens = [int(x) for x in r.integers(0, 6, size=n)]
    w = I.WORKLOADS[3].with_(Hqk=Hqk, Hv=Hv, K=K, V=V, dtype=dtype, seed=700 + i)
    x = I.make_inputs(w, "cpu", lengths=lens)
    T = sum(lens)
    a, b, A_log, dt_bias = gating_inputs(1, T, Hv, 800 + i)
    if r.random() < 0.4:
        dt_bias = None
    slots_n = n + int(r.integers(0, 4))
    perm = r.permutation(slots_n)[:n].astype(np.int32)
    perm[r.random(n) < 0.2] = -1
    slots = torch.from_numpy(perm)
    pool = torch.randn(slots_n, Hv, K, V, generator=torch.Generator().manual_seed(900 + i)) * 0.1
    o_ref, pool_ref = oracle_mod.gated_recurrent(x["q"], x["k"], x["v"], a, b, A_log, dt_bias, x["scale"], pool,
                                                 state_indices=slots, cu_seqlens=x["cu_seqlens"])
    state = pool.cuda()
    o = gdn.gdn_recurrent_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), a.cuda(), b.cuda(), A_log.cuda(), state,
                              dt_bias=dt_bias.cuda() if dt_bias is not None else None, scale=x["scale"],
                              state_indices=slots.cuda(), cu_seqlens=x["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    if o_ref.size:
        assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL[dtype]
    assert rel_fro(state.cpu().numpy(), pool_ref) <= 1e-5
