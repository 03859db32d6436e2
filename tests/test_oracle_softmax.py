"""Pins of the oracle's temperature softmax (CPU only)."""

import math

import numpy as np
import pytest

from oracle import softmax


def test_two_token_closed_form():
    for a, b, T in [(0.0, 1.0, 1.0), (3.5, -2.0, 0.3), (10.0, 10.0, 0.7), (-4.0, 7.0, 2.0)]:
        _, logz, logp = softmax.row_stats(np.array([a, b]), T)
        p0 = 1.0 / (1.0 + math.exp((b - a) / T))
        assert abs(math.exp(logp[0]) - p0) < 1e-15
        assert abs(math.exp(logp[1]) - (1 - p0)) < 1e-15
        assert abs(logz - math.log(math.exp(a / T) + math.exp(b / T))) < 1e-12


def test_three_token_closed_form_with_minus_inf():
    l = np.array([1.0, -np.inf, 2.0])
    p = softmax.probs(l, 0.5)
    e = [math.exp(2.0), 0.0, math.exp(4.0)]
    assert p[1] == 0.0
    assert abs(p[0] - e[0] / (e[0] + e[2])) < 1e-15
    assert abs(p[2] - e[2] / (e[0] + e[2])) < 1e-15


def test_normalisation_and_logz_against_fsum():
    rng = np.random.default_rng(0)
    for T in (0.3, 0.7, 1.0, 1.7):
        l = (rng.standard_normal(5000) * 2.5).astype(np.float32)
        m, logz, logp = softmax.row_stats(l, T)
        assert abs(math.fsum(np.exp(logp)) - 1.0) < 1e-12
        ref = m / T + math.log(math.fsum(math.exp((float(v) - m) / T) for v in l))
        assert abs(logz - ref) < 1e-12 * max(1.0, abs(ref))


def test_logz_against_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(1)
    l = (rng.standard_normal(300) * 3).astype(np.float32)
    for T in (0.3, 1.0):
        _, logz, logp = softmax.row_stats(l, T)
        z = mp.fsum(mp.exp(mp.mpf(float(v)) / T) for v in l)
        assert abs(logz - float(mp.log(z))) < 1e-13 * abs(float(mp.log(z)))
        k = int(np.argmax(l))
        assert abs(logp[k] - float(mp.mpf(float(l[k])) / T - mp.log(z))) < 1e-13


def test_row_validity():
    assert softmax.row_is_valid([0.0, -np.inf, 1.0])
    assert not softmax.row_is_valid([0.0, np.nan])
    assert not softmax.row_is_valid([0.0, np.inf])
    assert not softmax.row_is_valid([-np.inf, -np.inf])


def test_argmax_lowest_index_on_ties():
    assert softmax.argmax_lowest([1.0, 3.0, 3.0, 2.0]) == 1
    assert softmax.argmax_lowest([5.0, 5.0]) == 0
    assert softmax.argmax_lowest([-np.inf, -1.0]) == 1
