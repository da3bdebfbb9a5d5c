"""GPU parity of the backward pass (gdn_chunk_bwd, through the C ABI) against
the fp64 oracle's reverse-mode gradients on the same seeded inputs and
upstream gradients.  The backward computes in fp32 from the stored inputs
(bf16 or fp32), so the bar is a relative Frobenius error of at most 1e-4 on
every gradient.  K = V = 128 takes the chunked backward (equal lengths in
sequence groups, packed sequences in one group with device-built chunk
tables); K = 64 the token-recurrence one."""
import numpy as np
import pytest
import torch

from conftest import rel_fro
from gated_deltanet_chunked_gdn_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_chunked_gdn_gb300 import binding
    binding.load()
    return binding


def upstream(x, N, Hv, K, V, seed, with_dht=True):
    gen = torch.Generator().manual_seed(seed)
    do = torch.randn(x["v"].shape, generator=gen).to(x["v"].dtype)
    dht = torch.randn((N, Hv, K, V), generator=gen) if with_dht else None
    return do, dht


def shifted(t):
    """A CUDA copy of t whose data starts 4 bytes past a 16-byte boundary."""
    flat = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
    off = (-(flat.data_ptr() % 16) + 4) % 16 // t.element_size()
    v = flat[off:off + t.numel()].view(t.shape)
    v.copy_(t.cuda())
    assert v.data_ptr() % 16 == 4
    return v


def check(gdn, oracle_mod, w, lens=None, with_h0=True, with_dht=True, seed=11, unaligned=False):
    x = I.make_inputs(w, "cpu", lengths=lens)
    if not with_h0:
        x["h0"] = None
    N = x["N"]
    do, dht = upstream(x, N, w.Hv, w.K, w.V, seed, with_dht)
    d = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    do_d = do.cuda()
    if unaligned:
        d["q"], d["k"], d["v"], do_d = shifted(x["q"]), shifted(x["k"]), shifted(x["v"]), shifted(do)
    r = gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do_d, scale=d["scale"], h0=d["h0"],
                          dht=dht.cuda() if dht is not None else None, cu_seqlens=d["cu_seqlens"])
    assert gdn.gdn_chunk_bwd_get_device_status(r["workspace"]) == gdn.DEV_OK
    ref = oracle_mod.recurrent_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], do, h0=x["h0"], dht=dht,
                                   cu_seqlens=x["cu_seqlens"])
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        got = r[key].cpu().numpy()
        assert np.all(np.isfinite(got)), key
        assert rel_fro(got, ref[key]) <= TOL, (key, rel_fro(got, ref[key]))


def test_bwd_fp32_gqa_ragged(gdn, oracle_mod):
    # 150 tokens: two full 64-token chunks and a tail, 16-token blocks and a tail; GQA 1 -> 2
    check(gdn, oracle_mod, I.WORKLOADS[0].with_(B=2, T=150, Hqk=1, Hv=2))


def test_bwd_fp32_chunked_gqa_ragged(gdn, oracle_mod):
    # equal lengths with K = V = 128: the chunked backward (150 tokens: two full
    # chunks and a 22-token tail; GQA 1 -> 2)
    check(gdn, oracle_mod, I.WORKLOADS[2].with_(B=2, T=150, Hqk=1, Hv=2, dtype="f32"))


def test_bwd_bf16_varlen_gqa(gdn, oracle_mod):
    check(gdn, oracle_mod, I.WORKLOADS[3].with_(Hqk=2, Hv=4), lens=[5, 64, 200, 1, 0, 129, 63, 65])


def test_bwd_fp32_chunked_varlen(gdn, oracle_mod):
    # packed sequences on the chunked form: several chunks with a ragged tail,
    # a one-token and an empty sequence, exactly one chunk
    check(gdn, oracle_mod, I.WORKLOADS[3].with_(Hqk=2, Hv=4, dtype="f32"), lens=[300, 1, 64, 0, 129])


def test_bwd_bf16_chunked_varlen_without_h0_and_dht(gdn, oracle_mod):
    check(gdn, oracle_mod, I.WORKLOADS[3].with_(Hqk=1, Hv=2), lens=[200, 65, 7], with_h0=False, with_dht=False)


def test_bwd_fp32_varlen_token_path(gdn, oracle_mod):
    # K = 64: packed sequences on the token recurrence
    check(gdn, oracle_mod, I.WORKLOADS[0].with_(Hqk=1, Hv=2), lens=[5, 70, 0, 130])


def test_bwd_unaligned_inputs_take_token_path(gdn, oracle_mod):
    # q, k, v and dout 4-byte aligned only: the chunked form needs 16-byte
    # alignment, so the token recurrence runs on a K = V = 128 problem
    check(gdn, oracle_mod, I.WORKLOADS[2].with_(B=2, T=130, Hqk=1, Hv=2), unaligned=True)


def test_bwd_without_h0_and_dht(gdn, oracle_mod):
    check(gdn, oracle_mod, I.WORKLOADS[2].with_(B=1, T=300, Hqk=2, Hv=2), with_h0=False, with_dht=False)


def test_bwd_long_sequence(gdn, oracle_mod):
    check(gdn, oracle_mod, I.WORKLOADS[2].with_(B=1, T=1000, Hqk=1, Hv=2))


def test_bwd_rejects_head_dim_256(gdn):
    w = I.WORKLOADS[4].with_(B=1, T=16, Hqk=1, Hv=1)
    x = I.make_inputs(w, "cuda")
    with pytest.raises(gdn.GDNError):
        gdn.gdn_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], torch.zeros_like(x["v"]))


def test_bwd_malformed_cu_seqlens(gdn):
    w = I.WORKLOADS[3].with_(Hqk=1, Hv=2)
    x = I.make_inputs(w, "cuda", lengths=[10, 20, 30])
    bad = torch.tensor([0, 10, 70, 60], dtype=torch.int32, device="cuda")
    r = gdn.gdn_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], torch.zeros_like(x["v"]), cu_seqlens=bad)
    assert gdn.gdn_chunk_bwd_get_device_status(r["workspace"]) == gdn.DEV_BAD_CU_SEQLENS


@pytest.mark.parametrize("B,chains", [(1, [(0, 0), (0, 31)]), (16, [(0, 5), (7, 12), (15, 31)])])
def test_bwd_fullsize_sampled_chains(gdn, oracle_mod, B, chains):
    # the bench's shape at full length (8192 tokens, 128 chunks a chain, H = 32;
    # B = 16 runs in sequence groups, the last holding one sequence): sampled
    # (sequence, head) chains against the oracle run on each chain alone (with
    # Hqk = Hv every gradient of head h depends on chain (n, h) only)
    w = I.WORKLOADS[2].with_(B=B)
    x = I.make_inputs(w, "cuda")
    gen = torch.Generator(device="cuda").manual_seed(13)
    do = torch.randn(x["v"].shape, generator=gen, device="cuda").to(x["v"].dtype)
    dht = torch.randn((B, w.Hv, w.K, w.V), generator=gen, device="cuda")
    r = gdn.gdn_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, scale=x["scale"], h0=x["h0"], dht=dht)
    assert gdn.gdn_chunk_bwd_get_device_status(r["workspace"]) == gdn.DEV_OK
    for n, h in chains:
        sl = lambda t: t[n:n + 1, :, h:h + 1].cpu()
        ref = oracle_mod.recurrent_bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]), x["scale"],
                                       sl(do), h0=x["h0"][n:n + 1, h:h + 1].cpu(), dht=dht[n:n + 1, h:h + 1].cpu())
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            got = sl(r[key]).numpy()
            assert rel_fro(got, ref[key]) <= TOL, (n, h, key, rel_fro(got, ref[key]))
        got = r["dh0"][n:n + 1, h:h + 1].cpu().numpy()
        assert rel_fro(got, ref["dh0"]) <= TOL, (n, h, "dh0", rel_fro(got, ref["dh0"]))


def test_bwd_fullsize_packed_sampled(gdn, oracle_mod):
    # the 64-sequence packed batch (51 606 tokens, Hqk = 16, Hv = 32) on the
    # chunked form with device-built tables: the longest sequence and one of
    # the shortest against the oracle, each with the G value heads of one q/k
    # head (dq and dk sum over them)
    w = I.WORKLOADS[3]
    x = I.make_inputs(w, "cuda")
    N, G = x["N"], w.Hv // w.Hqk
    cu = x["cu_seqlens"].cpu().tolist()
    lens = [cu[i + 1] - cu[i] for i in range(N)]
    gen = torch.Generator(device="cuda").manual_seed(17)
    do = torch.randn(x["v"].shape, generator=gen, device="cuda").to(x["v"].dtype)
    dht = torch.randn((N, w.Hv, w.K, w.V), generator=gen, device="cuda")
    r = gdn.gdn_chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, scale=x["scale"], h0=x["h0"], dht=dht,
                          cu_seqlens=x["cu_seqlens"])
    assert gdn.gdn_chunk_bwd_get_device_status(r["workspace"]) == gdn.DEV_OK
    longest = max(range(N), key=lambda i: lens[i])
    shortest = min((i for i in range(N) if lens[i] > 0), key=lambda i: lens[i])
    for n, hq in ((longest, 3), (shortest, 15)):
        a, e, hv = cu[n], cu[n + 1], slice(G * hq, G * hq + G)
        sq = lambda t: t[:, a:e, hq:hq + 1].cpu()
        sv = lambda t: t[:, a:e, hv].cpu()
        ref = oracle_mod.recurrent_bwd(sq(x["q"]), sq(x["k"]), sv(x["v"]), sv(x["g"]), sv(x["beta"]), x["scale"],
                                       sv(do), h0=x["h0"][n:n + 1, hv].cpu(), dht=dht[n:n + 1, hv].cpu())
        got = {"dq": sq(r["dq"]), "dk": sq(r["dk"]), "dv": sv(r["dv"]), "dg": sv(r["dg"]), "dbeta": sv(r["dbeta"]),
               "dh0": r["dh0"][n:n + 1, hv].cpu()}
        for key, val in got.items():
            assert rel_fro(val.numpy(), ref[key]) <= TOL, (n, lens[n], key, rel_fro(val.numpy(), ref[key]))


def draw_bwd(i):
    """Draw i of the randomised backward sweep: shape, GQA ratio, dtype, head
    dims (K = V = 128 takes the chunked backward, K = 64 the token recurrence),
    packed lengths, h0 and dht."""
    r = np.random.default_rng(5200 + i)
    dtype = "bf16" if r.random() < 0.6 else "f32"
    K = int(r.choice([64, 128]))
    V = 128 if K == 128 else int(r.choice([64, 128]))
    Hqk = int(r.choice([1, 2]))
    Hv = Hqk * int(r.choice([1, 2]))
    gate = "softplus_exp" if r.random() < 0.7 else "logsigmoid4"
    lens = None
    if r.random() < 0.5:
        n = int(r.integers(1, 6))
        lens = [int(x) for x in r.integers(0, 260, size=n)]
        w = I.Workload("random_bwd", 1, 0, Hqk, Hv, K, V, 64, dtype, gate, True, 500 + i, varlen_n=n)
    else:
        w = I.Workload("random_bwd", int(r.integers(1, 3)), int(r.integers(1, 260)), Hqk, Hv, K, V, 64, dtype, gate,
                       True, 500 + i)
    return w, lens, bool(r.random() < 0.7), bool(r.random() < 0.7)


@pytest.mark.parametrize("i", range(16))
def test_bwd_random_draw(gdn, oracle_mod, i):
    w, lens, with_h0, with_dht = draw_bwd(i)
    check(gdn, oracle_mod, w, lens=lens, with_h0=with_h0, with_dht=with_dht, seed=40 + i)
