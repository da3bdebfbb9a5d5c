"""Pins for the oracle's backward pass (no GPU).

The gradients of the token recurrence are checked against central finite
differences of the oracle's own forward (itself pinned in
test_oracle_pins.py) for L = <dout, o> + <dht, ht>, against the closed form
of the pure-decay case (beta = 0), and against the invariants of a reverse
pass (linear in the upstream gradients; a packed batch equals its sequences
run one by one).  A mutation test plants slips in a copy of the C oracle and
checks that some pin catches each.
"""
import os
import subprocess

import numpy as np
import pytest

from oracle import oracle as oracle_pkg

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gdn_oracle.c")


def problem(seed, B=1, T=6, Hqk=1, Hv=2, K=3, V=2, h0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hqk, K))
    k = rng.standard_normal((B, T, Hqk, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, V))
    g = -rng.random((B, T, Hv))
    beta = rng.random((B, T, Hv))
    N = B
    h = rng.standard_normal((N, Hv, K, V)) if h0 else None
    do = rng.standard_normal((B, T, Hv, V))
    dht = rng.standard_normal((N, Hv, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h), do, dht


def loss(ora, x, do, dht, scale, cu=None):
    o, ht = ora.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], scale, h0=x["h0"], cu_seqlens=cu)
    return float((o * do).sum() + (ht * dht).sum())


def check_finite_differences(ora, seed=0, h0=True, cu=None, T=6, B=1):
    x, do, dht = problem(seed, B=B, T=T, h0=h0)
    if cu is not None:
        dht = np.random.default_rng(seed + 1).standard_normal((len(cu) - 1,) + dht.shape[1:])
        if x["h0"] is not None:
            x["h0"] = np.random.default_rng(seed + 2).standard_normal((len(cu) - 1,) + x["h0"].shape[1:])
    scale = 0.7
    r = ora.recurrent_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], scale, do, h0=x["h0"], dht=dht, cu_seqlens=cu)
    names = ["q", "k", "v", "g", "beta"] + (["h0"] if x["h0"] is not None else [])
    eps = 1e-6
    for name in names:
        base = x[name]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            xp = dict(x), dict(x)
            plus, minus = base.copy(), base.copy()
            plus[idx] += eps
            minus[idx] -= eps
            xp[0][name], xp[1][name] = plus, minus
            num[idx] = (loss(ora, xp[0], do, dht, scale, cu) - loss(ora, xp[1], do, dht, scale, cu)) / (2 * eps)
        got = r["dh0"] if name == "h0" else r["d" + name]
        np.testing.assert_allclose(got, num, rtol=1e-6, atol=1e-7, err_msg=name)


def check_pure_decay_closed_form(ora):
    """beta = 0: S_t = e^{gamma_t} h0, so dq_t = scale e^{gamma_t} h0 dout_t,
    dv = 0, dh0 = e^{gamma_T} dht + sum_t scale e^{gamma_t} q_t dout_t^T."""
    x, do, dht = problem(3, T=5, Hv=1)
    x["beta"] = np.zeros_like(x["beta"])
    scale = 0.4
    r = ora.recurrent_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], scale, do, h0=x["h0"], dht=dht)
    gam = np.cumsum(x["g"][0, :, 0])
    h0 = x["h0"][0, 0]
    dq = np.stack([scale * np.exp(gam[t]) * h0 @ do[0, t, 0] for t in range(5)])
    np.testing.assert_allclose(r["dq"][0, :, 0], dq, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r["dv"], 0.0)
    dh0 = np.exp(gam[-1]) * dht[0, 0] + sum(scale * np.exp(gam[t]) * np.outer(x["q"][0, t, 0], do[0, t, 0])
                                            for t in range(5))
    np.testing.assert_allclose(r["dh0"][0, 0], dh0, rtol=1e-12, atol=1e-12)


def check_linear_in_upstream(ora):
    x, do, dht = problem(5)
    _, do2, dht2 = problem(6)
    f = lambda a, b: ora.recurrent_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.3, a, h0=x["h0"], dht=b)
    r1, r2, r12 = f(do, dht), f(do2, dht2), f(do + 2 * do2, dht + 2 * dht2)
    for key in r1:
        np.testing.assert_allclose(r12[key], r1[key] + 2 * r2[key], rtol=1e-10, atol=1e-10, err_msg=key)


def check_packed_equals_separate(ora):
    rng = np.random.default_rng(9)
    lens = [4, 0, 7, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    Tt = int(cu[-1])
    x, do, _ = problem(9, T=Tt)
    N = len(lens)
    x["h0"] = rng.standard_normal((N,) + x["h0"].shape[1:])
    dht = rng.standard_normal((N,) + x["h0"].shape[1:])
    r = ora.recurrent_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], 0.5, do, h0=x["h0"], dht=dht, cu_seqlens=cu)
    for n in range(N):
        sl = slice(cu[n], cu[n + 1])
        sub = {k_: (x[k_][:, sl] if k_ != "h0" else x["h0"][n:n + 1]) for k_ in x}
        rn = ora.recurrent_bwd(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], 0.5, do[:, sl],
                               h0=sub["h0"], dht=dht[n:n + 1])
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(r[key][:, sl], rn[key], rtol=1e-12, atol=1e-12, err_msg=key)
        np.testing.assert_allclose(r["dh0"][n], rn["dh0"][0], rtol=1e-12, atol=1e-12)


PINS = [lambda o: check_finite_differences(o), lambda o: check_finite_differences(o, seed=1, h0=False),
        check_pure_decay_closed_form, check_linear_in_upstream, check_packed_equals_separate]


def test_finite_differences_gqa(oracle_mod):
    check_finite_differences(oracle_mod)


def test_finite_differences_without_h0(oracle_mod):
    check_finite_differences(oracle_mod, seed=1, h0=False)


def test_finite_differences_packed(oracle_mod):
    check_finite_differences(oracle_mod, seed=2, cu=np.array([0, 3, 3, 7]), T=7)


def test_pure_decay_closed_form(oracle_mod):
    check_pure_decay_closed_form(oracle_mod)


def test_linear_in_upstream_gradients(oracle_mod):
    check_linear_in_upstream(oracle_mod)


def test_packed_equals_separate(oracle_mod):
    check_packed_equals_separate(oracle_mod)


MUTANTS = {
    "dk_sign": ("dkt[d] += -a * b * (gu + sw) + b * gv;", "dkt[d] += a * b * (gu + sw) + b * gv;"),
    "adjoint_no_decay": ("G[(int64_t)d * V + e] = a * (G[(int64_t)d * V + e] - b * kt[d] * w[e]);",
                         "G[(int64_t)d * V + e] = (G[(int64_t)d * V + e] - b * kt[d] * w[e]);"),
    "dbeta_missing_value_term": ("dbeta[t * Hv + h] = -a * wu + wv;", "dbeta[t * Hv + h] = -a * wu;"),
    "dq_from_previous_state": ("acc += Sc[(int64_t)d * V + e] * dot[e];", "acc += Sp[(int64_t)d * V + e] * dot[e];"),
    "dg_missing_chain_factor": ("dg[t * Hv + h] = a * (gs - b * wu);", "dg[t * Hv + h] = (gs - b * wu);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_bwd_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, old
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mpath), "-o", str(so), "-lm"],
                   check=True)
    mutant = oracle_pkg.Oracle(str(so))
    caught = 0
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught += 1
    assert caught >= 1, f"no pin caught mutant {name}"
