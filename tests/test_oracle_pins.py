"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: hand-derived
worked examples, closed forms of special cases, invariants of the delta rule,
the second (chunked) form written independently, and library routines.  The
cases are chosen so that a plausible slip (a dropped decay, a sign flip, a
transposed state, the wrong GQA head, the output taken before the update, a
wrong chunk boundary) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from conftest import rel_fro

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
TOL = 1e-10


def rand_inputs(rng, B, T, Hqk, Hv, K, V, h0=True, gate_scale=1.0):
    q = rng.standard_normal((B, T, Hqk, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, Hqk, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv)))) * gate_scale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv))))
    h = 0.1 * rng.standard_normal((B, Hv, K, V)) if h0 else None
    return q, k, v, g, beta, h


# ----------------------------------------------------------------- golden

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("form", ["recurrent", "chunked_C1", "chunked_C2"])
def test_hand_worked_examples(oracle_mod, case, form):
    T = len(case["g"])
    K, V = case["K"], case["V"]
    q = np.array(case["q"]).reshape(1, T, 1, K)
    k = np.array(case["k"]).reshape(1, T, 1, K)
    v = np.array(case["v"]).reshape(1, T, 1, V)
    g = np.array(case["g"]).reshape(1, T, 1)
    beta = np.array(case["beta"]).reshape(1, T, 1)
    h0 = np.array(case["h0"]).reshape(1, 1, K, V)
    if form == "recurrent":
        o, ht = oracle_mod.recurrent(q, k, v, g, beta, case["scale"], h0=h0)
    else:
        C = int(form[-1])
        o, ht = oracle_mod.chunked(q, k, v, g, beta, case["scale"], C, h0=h0)
    np.testing.assert_allclose(o.reshape(T, V), np.array(case["o"]), atol=1e-12, rtol=0)
    np.testing.assert_allclose(ht.reshape(K, V), np.array(case["ht"]), atol=1e-12, rtol=0)


# ------------------------------------------------- chunked form == recurrence

@pytest.mark.parametrize("C", [1, 4, 16, 64, 128])
@pytest.mark.parametrize("seed", [0, 1])
def test_chunked_equals_recurrent(oracle_mod, C, seed):
    rng = np.random.default_rng(100 + seed)
    # T = 301 spans several chunks of every C and leaves a ragged tail.
    q, k, v, g, beta, h0 = rand_inputs(rng, 2, 301, 2, 4, 16, 12)
    o_r, ht_r = oracle_mod.recurrent(q, k, v, g, beta, 0.25, h0=h0)
    o_c, ht_c = oracle_mod.chunked(q, k, v, g, beta, 0.25, C, h0=h0)
    assert rel_fro(o_c, o_r) < TOL
    assert rel_fro(ht_c, ht_r) < TOL


def test_chunked_equals_recurrent_varlen(oracle_mod):
    rng = np.random.default_rng(7)
    lens = [5, 0, 64, 1, 130, 63, 200]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, _ = rand_inputs(rng, 1, T, 1, 2, 8, 8, h0=False)
    h0 = 0.1 * rng.standard_normal((len(lens), 2, 8, 8))
    o_r, ht_r = oracle_mod.recurrent(q, k, v, g, beta, 0.5, h0=h0, cu_seqlens=cu)
    for C in (16, 64):
        o_c, ht_c = oracle_mod.chunked(q, k, v, g, beta, 0.5, C, h0=h0, cu_seqlens=cu)
        assert rel_fro(o_c, o_r) < TOL
        assert rel_fro(ht_c, ht_r) < TOL


def test_recurrent_matches_strong_decay_dynamic_range(oracle_mod):
    """g as negative as the bf16 workloads produce (cumsum over a chunk far
    below -88): the chunked form must still agree (no overflow in e^{-gamma})."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, 256, 1, 1, 8, 8, gate_scale=4.0)
    o_r, ht_r = oracle_mod.recurrent(q, k, v, g, beta, 1.0, h0=h0)
    o_c, ht_c = oracle_mod.chunked(q, k, v, g, beta, 1.0, 128, h0=h0)
    assert np.all(np.isfinite(o_c))
    assert rel_fro(o_c, o_r) < TOL and rel_fro(ht_c, ht_r) < TOL


# ------------------------------------------------------------- closed forms

@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_beta_zero_is_pure_decay(oracle_mod, form):
    """beta = 0: S_T = exp(sum g) h0 and o_t = scale exp(sum_{s<=t} g_s) h0^T q_t."""
    rng = np.random.default_rng(11)
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, 90, 1, 1, 6, 5)
    beta[:] = 0.0
    scale = 0.3
    if form == "recurrent":
        o, ht = oracle_mod.recurrent(q, k, v, g, beta, scale, h0=h0)
    else:
        o, ht = oracle_mod.chunked(q, k, v, g, beta, scale, 32, h0=h0)
    G = np.cumsum(g[0, :, 0])
    H = h0[0, 0]
    o_ref = scale * np.exp(G)[:, None] * (q[0, :, 0, :] @ H)
    assert rel_fro(o[0, :, 0, :], o_ref) < TOL
    assert rel_fro(ht[0, 0], math.exp(G[-1]) * H) < TOL


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_delta_rule_overwrite_orthonormal_keys(oracle_mod, form):
    """g = 0, beta = 1, orthonormal keys: each write replaces the value stored
    under its key, so S_T = (I - sum k_i k_i^T) h0 + sum k_i v_i^T, and
    querying with q_t = k_t returns scale * v_t."""
    rng = np.random.default_rng(5)
    K, V, T = 16, 7, 12
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:, :T].T                       # T orthonormal rows
    k = keys.reshape(1, T, 1, K)
    q = k.copy()
    v = rng.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    h0 = rng.standard_normal((1, 1, K, V))
    scale = 0.7
    if form == "recurrent":
        o, ht = oracle_mod.recurrent(q, k, v, g, beta, scale, h0=h0)
    else:
        o, ht = oracle_mod.chunked(q, k, v, g, beta, scale, 5, h0=h0)
    P = keys.T @ keys
    S_ref = (np.eye(K) - P) @ h0[0, 0] + keys.T @ v[0, :, 0, :]
    assert rel_fro(ht[0, 0], S_ref) < TOL
    assert rel_fro(o[0, :, 0, :], scale * v[0, :, 0, :]) < TOL


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_householder_reflection_preserves_state(oracle_mod, form):
    """g = 0, beta = 2, unit keys, v = 0: each step applies the reflection
    I - 2 k k^T (orthogonal), so S_T = H_T ... H_1 h0 (checked against an
    explicit matrix product) and ||S_T||_F = ||h0||_F."""
    rng = np.random.default_rng(9)
    K, V, T = 8, 3, 20
    k = rng.standard_normal((1, T, 1, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q = rng.standard_normal((1, T, 1, K))
    v = np.zeros((1, T, 1, V))
    g = np.zeros((1, T, 1))
    beta = np.full((1, T, 1), 2.0)
    h0 = rng.standard_normal((1, 1, K, V))
    if form == "recurrent":
        _, ht = oracle_mod.recurrent(q, k, v, g, beta, 1.0, h0=h0)
    else:
        _, ht = oracle_mod.chunked(q, k, v, g, beta, 1.0, 8, h0=h0)
    M = np.eye(K)
    for t in range(T):
        kt = k[0, t, 0]
        M = (np.eye(K) - 2.0 * np.outer(kt, kt)) @ M
    assert rel_fro(ht[0, 0], M @ h0[0, 0]) < TOL
    assert abs(np.linalg.norm(ht) - np.linalg.norm(h0)) < 1e-10 * np.linalg.norm(h0)


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_fixed_point_when_values_match_predictions(oracle_mod, form):
    """g = 0, beta = 1 and v_t = h0^T k_t: every write stores what is already
    there, so S_t = h0 for all t and o_t = scale h0^T q_t."""
    rng = np.random.default_rng(21)
    K, V, T = 10, 6, 40
    q, k, _, _, _, h0 = rand_inputs(rng, 1, T, 1, 1, K, V)
    v = np.einsum("tk,kv->tv", k[0, :, 0, :], h0[0, 0]).reshape(1, T, 1, V)
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    if form == "recurrent":
        o, ht = oracle_mod.recurrent(q, k, v, g, beta, 0.5, h0=h0)
    else:
        o, ht = oracle_mod.chunked(q, k, v, g, beta, 0.5, 16, h0=h0)
    assert rel_fro(ht[0, 0], h0[0, 0]) < TOL
    assert rel_fro(o[0, :, 0, :], 0.5 * q[0, :, 0, :] @ h0[0, 0]) < TOL


# ---------------------------------------------------------------- structure

@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_state_passing_resumes(oracle_mod, form):
    """run(T1) then run(T2, h0 = ht) equals run(T1 + T2)."""
    rng = np.random.default_rng(13)
    q, k, v, g, beta, h0 = rand_inputs(rng, 2, 150, 2, 2, 8, 8)
    f = (lambda *a, **kw: oracle_mod.recurrent(*a, **kw)) if form == "recurrent" else \
        (lambda *a, **kw: oracle_mod.chunked(*a[:6], 64, *a[6:], **kw))
    o, ht = f(q, k, v, g, beta, 0.5, h0=h0)
    T1 = 77
    o1, ht1 = f(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], beta[:, :T1], 0.5, h0=h0)
    o2, ht2 = f(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], beta[:, T1:], 0.5, h0=ht1)
    assert rel_fro(np.concatenate([o1, o2], axis=1), o) < TOL
    assert rel_fro(ht2, ht) < TOL


def test_varlen_equals_per_sequence_runs(oracle_mod):
    rng = np.random.default_rng(17)
    lens = [3, 0, 70, 129]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, beta, _ = rand_inputs(rng, 1, sum(lens), 2, 4, 8, 4, h0=False)
    h0 = 0.1 * rng.standard_normal((len(lens), 4, 8, 4))
    o, ht = oracle_mod.recurrent(q, k, v, g, beta, 1.0, h0=h0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        s = slice(cu[n], cu[n + 1])
        if L == 0:
            np.testing.assert_array_equal(ht[n], h0[n])
            continue
        on, htn = oracle_mod.recurrent(q[:, s], k[:, s], v[:, s], g[:, s], beta[:, s], 1.0, h0=h0[n:n + 1])
        assert rel_fro(o[:, s], on) < TOL
        assert rel_fro(ht[n], htn[0]) < TOL


def test_gqa_maps_value_head_to_group(oracle_mod):
    """Value head h reads q/k head h // (Hv/Hqk): equal to repeating each qk
    head G times (repeat_interleave), not tiling them."""
    rng = np.random.default_rng(19)
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, 50, 2, 6, 8, 8)
    o, ht = oracle_mod.recurrent(q, k, v, g, beta, 1.0, h0=h0)
    qr, kr = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    o2, ht2 = oracle_mod.recurrent(qr, kr, v, g, beta, 1.0, h0=h0)
    assert rel_fro(o, o2) < TOL and rel_fro(ht, ht2) < TOL
    qt, kt = np.tile(q, (1, 1, 3, 1)), np.tile(k, (1, 1, 3, 1))
    o3, _ = oracle_mod.recurrent(qt, kt, v, g, beta, 1.0, h0=h0)
    assert rel_fro(o3, o) > 1e-3   # the tiled mapping is a different operator


def test_linearity_in_h0_and_v(oracle_mod):
    """For fixed q, k, g, beta the map (h0, v) -> (o, ht) is linear, and o is
    linear in q."""
    rng = np.random.default_rng(23)
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, 60, 1, 1, 8, 8)
    _, _, v2, _, _, h02 = rand_inputs(rng, 1, 60, 1, 1, 8, 8)
    a, b = 0.7, -1.9
    o1, s1 = oracle_mod.recurrent(q, k, v, g, beta, 1.0, h0=h0)
    o2, s2 = oracle_mod.recurrent(q, k, v2, g, beta, 1.0, h0=h02)
    o3, s3 = oracle_mod.recurrent(q, k, a * v + b * v2, g, beta, 1.0, h0=a * h0 + b * h02)
    assert rel_fro(o3, a * o1 + b * o2) < TOL
    assert rel_fro(s3, a * s1 + b * s2) < TOL
    q2 = rng.standard_normal(q.shape)
    o4, _ = oracle_mod.recurrent(a * q + b * q2, k, v, g, beta, 1.0, h0=h0)
    o5, _ = oracle_mod.recurrent(q2, k, v, g, beta, 1.0, h0=h0)
    assert rel_fro(o4, a * o1 + b * o5) < TOL


def test_output_uses_post_update_state(oracle_mod):
    """With h0 = 0 and T = 1 the output must see the token's own write:
    o_1 = scale * beta (k.q) v (exp(g) drops out since h0 = 0)."""
    rng = np.random.default_rng(29)
    q, k, v, g, beta, _ = rand_inputs(rng, 1, 1, 1, 1, 8, 5, h0=False)
    o, _ = oracle_mod.recurrent(q, k, v, g, beta, 0.9, h0=None)
    ref = 0.9 * beta[0, 0, 0] * float(k[0, 0, 0] @ q[0, 0, 0]) * v[0, 0, 0]
    assert rel_fro(o[0, 0, 0], ref) < TOL


# --------------------------------------------------- chunked intermediates

def test_stage_intermediates(oracle_mod):
    """Per-chunk intermediates of the chunked form: gamma is the in-chunk
    cumsum (numpy cumsum), A is strictly lower triangular, T is the inverse of
    I + A (numpy.linalg.inv), S0 of chunk c equals the recurrence's state after
    c*C tokens, and the tail chunk's padding rows are zero."""
    rng = np.random.default_rng(31)
    C, T = 16, 53
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, T, 1, 2, 8, 6)
    st = oracle_mod.chunked_stages(q, k, v, g, beta, 0.5, C, 0, 1, h0=h0)
    NT = st["gamma"].shape[0]
    assert NT == 4
    for c in range(NT):
        n = min(C, T - c * C)
        np.testing.assert_allclose(st["gamma"][c, :n], np.cumsum(g[0, c * C:c * C + n, 1]), rtol=0, atol=1e-12)
        A = st["A"][c, :n, :n]
        assert np.all(np.triu(A) == 0.0)
        Tinv = np.linalg.inv(np.eye(n) + A)
        assert rel_fro(st["T"][c, :n, :n], Tinv) < TOL
        if c > 0:
            _, ht = oracle_mod.recurrent(q[:, :c * C], k[:, :c * C], v[:, :c * C], g[:, :c * C],
                                         beta[:, :c * C], 0.5, h0=h0)
            assert rel_fro(st["S0"][c], ht[0, 1]) < TOL
        else:
            np.testing.assert_array_equal(st["S0"][0], h0[0, 1])
    tail = T - (NT - 1) * C
    assert np.all(st["W"][-1, tail:] == 0) and np.all(st["Vn"][-1, tail:] == 0)


def test_stage_wy_terms_against_the_recurrence(oracle_mod):
    """W, U and V' of every chunk, pinned by the token recurrence rather than
    by their own formulas.  Unrolling S_t = e^{g_t} S_{t-1} + k_t d_t^T with
    d_t = beta_t (v_t - e^{g_t} S_{t-1}^T k_t) over a chunk gives V' = U - W S0
    with V'_t = d_t: so the dumped V' must equal d_t computed from the
    recurrence's own states S_{t-1}, and U - W S0 must equal it for two
    different initial states h0 (whose chunk-start states differ by a
    full-rank K x V matrix, K <= V), which fixes W and U uniquely."""
    rng = np.random.default_rng(37)
    C, T, K, V, h = 16, 45, 6, 8, 1
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, T, 1, 2, K, V)

    def run(init):
        st = oracle_mod.chunked_stages(q, k, v, g, beta, 0.5, C, 0, h, h0=init)
        d = np.zeros((T, V))
        for t in range(T):
            if t == 0:
                S = init[0, h] if init is not None else np.zeros((K, V))
            else:
                _, ht = oracle_mod.recurrent(q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t], 0.5, h0=init)
                S = ht[0, h]
            d[t] = beta[0, t, h] * (v[0, t, h] - math.exp(g[0, t, h]) * (S.T @ k[0, t, 0]))
        return st, d

    a, da = run(h0)
    b, db = run(None)
    for c in range(a["gamma"].shape[0]):
        n = min(C, T - c * C)
        rows = slice(c * C, c * C + n)
        for st, d in ((a, da), (b, db)):
            assert rel_fro(st["Vn"][c, :n], d[rows]) < TOL
            assert rel_fro(st["U"][c, :n] - st["W"][c, :n] @ st["S0"][c], d[rows]) < TOL
        # the dumps of U and W do not depend on the initial state
        np.testing.assert_array_equal(a["W"][c], b["W"][c])
        np.testing.assert_array_equal(a["U"][c], b["U"][c])
        assert np.linalg.matrix_rank(a["S0"][c] - b["S0"][c]) == K


# -------------------------------------------------------- decode (gated) step

def test_gated_decode_hand_example(oracle_mod):
    case = json.load(open(GOLDEN))["decode_cases"][0]
    K, V = case["K"], case["V"]
    q = np.array(case["q"]).reshape(1, 1, 1, K)
    k = np.array(case["k"]).reshape(1, 1, 1, K)
    v = np.array(case["v"]).reshape(1, 1, 1, V)
    a = np.array(case["a"]).reshape(1, 1, 1)
    b = np.array(case["b"]).reshape(1, 1, 1)
    st = np.array(case["state"]).reshape(1, 1, K, V)
    o, new = oracle_mod.gated_recurrent(q, k, v, a, b, np.array(case["A_log"]), np.array(case["dt_bias"]),
                                        case["scale"], st)
    np.testing.assert_allclose(o.reshape(V), np.array(case["o"]).reshape(V), atol=1e-12, rtol=0)
    np.testing.assert_allclose(new.reshape(K, V), np.array(case["new_state"]), atol=1e-12, rtol=0)


def test_gated_decode_continues_prefill(oracle_mod):
    """Prefill of T tokens (chunked form) followed by one gated decode step on
    the resulting state equals the recurrence over T + 1 tokens whose last
    gate / beta come from the gating formula; state slots are honoured and an
    out-of-range slot leaves its state untouched with zero output."""
    rng = np.random.default_rng(41)
    T, K, V, Hv = 40, 8, 6, 2
    q, k, v, g, beta, _ = rand_inputs(rng, 3, T + 1, 1, Hv, K, V, h0=False)
    a = rng.standard_normal((3, 1, Hv))
    b = rng.standard_normal((3, 1, Hv))
    A_log = rng.standard_normal(Hv) * 0.5
    dt_bias = rng.standard_normal(Hv) * 0.1
    _, ht = oracle_mod.chunked(q[:, :T], k[:, :T], v[:, :T], g[:, :T], beta[:, :T], 0.3, 16)
    pool = rng.standard_normal((5, Hv, K, V))
    slots = np.array([4, 1, 7])            # sequence 2 has no slot
    pool[4], pool[1] = ht[0], ht[1]
    o1, new = oracle_mod.gated_recurrent(q[:, T:], k[:, T:], v[:, T:], a, b, A_log, dt_bias, 0.3, pool,
                                         state_indices=slots)
    g_last = -np.exp(A_log)[None, None, :] * np.logaddexp(0.0, a + dt_bias[None, None, :])
    beta_last = 1.0 / (1.0 + np.exp(-b))
    g_full = np.concatenate([g[:, :T], g_last], axis=1)
    b_full = np.concatenate([beta[:, :T], beta_last], axis=1)
    o_ref, ht_ref = oracle_mod.recurrent(q, k, v, g_full, b_full, 0.3)
    assert rel_fro(o1[:2], o_ref[:2, T:]) < TOL
    assert rel_fro(new[4], ht_ref[0]) < TOL and rel_fro(new[1], ht_ref[1]) < TOL
    assert np.all(o1[2] == 0.0)
    untouched = [0, 2, 3]
    np.testing.assert_array_equal(new[untouched], pool[untouched])
