"""Pins of the oracle's confidence (softmax-plus-argmax over the vocabulary)
against things other than itself: a direct softmax in plain Python, closed
forms, SciPy's softmax, and the invariants of the definition."""
import math

import numpy as np
import pytest

import oracle


def _brute(row):
    """Softmax written out with math.exp (no max subtraction), then its
    largest probability and the first index holding the largest logit."""
    e = [math.exp(v) for v in row]
    z = sum(e)
    probs = [t / z for t in e]
    best = max(row)
    return row.index(best), max(probs)


def test_brute_force_small_rows():
    rng = np.random.default_rng(0)
    for V in (1, 2, 3, 7, 12):
        x = rng.normal(0, 3, size=(5, V))
        arg, conf = oracle.confidence(x)
        for r in range(5):
            a, c = _brute([float(v) for v in x[r]])
            assert arg[r] == a
            assert abs(conf[r] - c) <= 1e-14 * max(1.0, c)


def test_closed_forms():
    V = 1000
    # uniform logits: every token has probability 1/V; the first is the argmax
    arg, conf = oracle.confidence(np.full((1, V), 3.25))
    assert arg[0] == 0 and abs(conf[0] - 1.0 / V) < 1e-15
    # one logit a above V-1 zeros: e^a / (e^a + V - 1)
    for a in (0.5, 4.0, 20.0):
        x = np.zeros((1, V))
        x[0, 417] = a
        arg, conf = oracle.confidence(x)
        want = math.exp(a) / (math.exp(a) + V - 1)
        assert arg[0] == 417 and abs(conf[0] - want) < 1e-14
    # two tied maxima: the lower index wins; each has probability 1/(2 + rest)
    x = np.full((1, 16), -2.0)
    x[0, 9] = x[0, 3] = 1.5
    arg, conf = oracle.confidence(x)
    assert arg[0] == 3
    assert abs(conf[0] - 1.0 / (2 + 14 * math.exp(-3.5))) < 1e-15


def test_minus_inf_entries_and_rows():
    x = np.array([[-np.inf, 0.0, -np.inf, 0.0], [-np.inf] * 4])
    arg, conf = oracle.confidence(x)
    assert arg[0] == 1 and abs(conf[0] - 0.5) < 1e-15    # masked tokens have probability 0
    assert arg[1] == 0 and conf[1] == 0.0                  # no distribution at all


def test_against_scipy_softmax_large_vocab():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(1)
    x = rng.normal(0, 2.5, size=(3, 262144))
    arg, conf = oracle.confidence(x)
    p = scipy_special.softmax(x, axis=1)
    assert np.array_equal(arg, p.argmax(axis=1))
    assert np.allclose(conf, p.max(axis=1), rtol=1e-12, atol=0)


def test_invariants_shift_and_permutation():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1.7, size=(4, 999))
    arg, conf = oracle.confidence(x)
    # adding a constant to every logit of a row leaves the distribution unchanged
    arg2, conf2 = oracle.confidence(x + np.array([[100.0], [-50.0], [0.25], [7.0]]))
    assert np.array_equal(arg, arg2) and np.allclose(conf, conf2, rtol=1e-12)
    # permuting the vocabulary moves the argmax with it and keeps the confidence
    perm = rng.permutation(999)
    arg3, conf3 = oracle.confidence(x[:, perm])
    assert np.array_equal(perm[arg3], arg) and np.allclose(conf, conf3, rtol=1e-12)
    # confidence is a probability of the top token: 1/V <= conf <= 1
    assert np.all(conf >= 1.0 / 999 - 1e-15) and np.all(conf <= 1.0)
