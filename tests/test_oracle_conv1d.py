"""Pins for the oracle's causal convolution with a carried state (no GPU).

The operator is the causal_conv1d of the TileLang x xLLM page: a depthwise
convolution along the sequence in which each output token sees only the
current and earlier tokens of its own sequence, with the last W-1 inputs kept
per sequence (``conv_state``, slot chosen by ``cache_indices``) so that decode
can continue where prefill stopped.  The pins check the oracle against hand
worked examples, numpy's convolution, and the state-carrying invariants
(splitting a sequence anywhere, or running it token by token, changes
nothing).  Each pin is a function of the convolution under test, so that the
mutation test below can hand it a copy of the oracle with a planted slip.
"""
import inspect
import json
import os
import textwrap

import numpy as np
import pytest

from oracle import oracle as oracle_pkg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["conv1d_cases"]


def check_hand_examples(conv):
    for c in _cases():
        W = len(c["weight"])
        x = np.array(c["x"], dtype=np.float64).reshape(1, -1, 1)
        w = np.array(c["weight"]).reshape(1, W)
        st = np.array(c["state"]).reshape(1, W - 1, 1) if W > 1 else None
        y, new = conv(x, w, np.array([c["bias"]]), c["activation"], conv_state=st)
        np.testing.assert_allclose(y.reshape(-1), c["y"], rtol=0, atol=1e-12)
        if st is not None:
            np.testing.assert_allclose(new.reshape(-1), c["new_state"], rtol=0, atol=1e-12)


def check_matches_numpy_convolve(conv):
    """Zero state, no activation, no bias: channel d is numpy's full
    convolution of x[:, d] with the reversed taps, cut to the first T outputs."""
    rng = np.random.default_rng(3)
    for W in (1, 2, 4, 5):
        x = rng.standard_normal((2, 37, 6))
        w = rng.standard_normal((6, W))
        y, _ = conv(x, w, None, "none")
        for b in range(2):
            for d in range(6):
                ref = np.convolve(x[b, :, d], w[d, ::-1])[:37]
                np.testing.assert_allclose(y[b, :, d], ref, rtol=0, atol=1e-12)


def check_silu_closed_form(conv):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 11, 3))
    w = rng.standard_normal((3, 1))
    b = rng.standard_normal(3)
    y, _ = conv(x, w, b, "silu")
    u = x * w[:, 0] + b
    np.testing.assert_allclose(y, u / (1.0 + np.exp(-u)), rtol=1e-14, atol=1e-14)


def check_split_anywhere(conv):
    """Running a sequence in pieces (each piece starting from the state the
    previous one left, pieces shorter than W-1 and empty ones included)
    equals one run over the whole sequence; so does the final state."""
    rng = np.random.default_rng(7)
    W, D, L = 4, 5, 23
    x = rng.standard_normal((1, L, D))
    w = rng.standard_normal((D, W))
    b = rng.standard_normal(D)
    s0 = rng.standard_normal((1, W - 1, D))
    y_all, s_all = conv(x, w, b, "silu", conv_state=s0)
    for cuts in ([0, 1, 2, 23], [0, 10, 10, 12, 23], [0, 22, 23], [0, 3, 4, 5, 6, 23]):
        st = s0.copy()
        pieces = []
        for a, e in zip(cuts[:-1], cuts[1:]):
            y, st = conv(x[:, a:e], w, b, "silu", conv_state=st)
            pieces.append(y)
        np.testing.assert_allclose(np.concatenate(pieces, axis=1), y_all, rtol=0, atol=1e-12)
        np.testing.assert_allclose(st, s_all, rtol=0, atol=0)


def check_packed_equals_separate(conv):
    """A packed batch (cu_seqlens) with a permuted slot map equals separate
    runs of each sequence on its own slot; a sequence with slot -1 starts from
    zeros and writes nothing; has_initial_state = 0 starts from zeros but
    still writes its slot."""
    rng = np.random.default_rng(11)
    W, D = 3, 4
    lens = [5, 1, 0, 9, 2]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.standard_normal((1, cu[-1], D))
    w = rng.standard_normal((D, W))
    pool = rng.standard_normal((6, W - 1, D))
    slots = np.array([4, 0, 2, -1, 5])
    init = np.array([1, 1, 1, 1, 0])
    y, new = conv(x, w, None, "none", conv_state=pool, cache_indices=slots, has_initial_state=init, cu_seqlens=cu)
    for n, L in enumerate(lens):
        xs = x[:, cu[n]:cu[n + 1]]
        if slots[n] < 0:
            yn, _ = conv(xs, w, None, "none")
        else:
            st = pool[slots[n]][None] if init[n] else np.zeros((1, W - 1, D))
            yn, sn = conv(xs, w, None, "none", conv_state=st)
            np.testing.assert_array_equal(new[slots[n]], sn[0])
        np.testing.assert_allclose(y[:, cu[n]:cu[n + 1]], yn, rtol=0, atol=1e-12)
    untouched = [s for s in range(6) if s not in slots]
    np.testing.assert_array_equal(new[untouched], pool[untouched])
    # an empty sequence leaves its state as it was
    np.testing.assert_array_equal(new[2], pool[2])


def check_decode_equals_prefill(conv):
    """Token-by-token calls (decode) reproduce one prefill call."""
    rng = np.random.default_rng(13)
    W, D, L = 4, 3, 9
    x = rng.standard_normal((2, L, D))
    w = rng.standard_normal((D, W))
    b = rng.standard_normal(D)
    s0 = rng.standard_normal((2, W - 1, D))
    y_all, s_all = conv(x, w, b, "silu", conv_state=s0)
    st = s0.copy()
    for t in range(L):
        y, st = conv(x[:, t:t + 1], w, b, "silu", conv_state=st)
        np.testing.assert_allclose(y[:, 0], y_all[:, t], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(st, s_all)


PINS = [check_hand_examples, check_matches_numpy_convolve, check_silu_closed_form, check_split_anywhere,
        check_packed_equals_separate, check_decode_equals_prefill]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_conv1d_pin(pin):
    pin(oracle_pkg.causal_conv1d)


# ------------------------------------------------------- mutation check

MUTANTS = {
    "taps_reversed": ("acc += w[:, j][None, :] * ext[j:j + L]", "acc += w[:, W - 1 - j][None, :] * ext[j:j + L]"),
    "state_one_row_early": ("new_state[slot] = ext[L:L + W - 1]", "new_state[slot] = ext[L - 1:L + W - 2]"),
    "initial_flag_ignored": ("if slot >= 0 and init_flag[n] != 0:", "if slot >= 0:"),
    "sigmoid_not_silu": ("acc = acc / (1.0 + np.exp(-acc))", "acc = 1.0 / (1.0 + np.exp(-acc))"),
    "bias_dropped": ("acc = np.tile(b, (L, 1))", "acc = np.zeros((L, D))"),
    "state_not_carried": ("init = st[slot]", "init = np.zeros((W - 1, D))"),
}


def _mutant(old, new):
    src = textwrap.dedent(inspect.getsource(oracle_pkg.causal_conv1d))
    assert src.count(old) == 1, old
    ns = dict(vars(oracle_pkg))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["causal_conv1d"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_conv1d_mutant_is_caught(name):
    conv = _mutant(*MUTANTS[name])
    caught = 0
    for pin in PINS:
        try:
            pin(conv)
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught >= 1, f"no pin caught mutant {name}"
