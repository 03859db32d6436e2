"""Pins of the oracle's Markov bias and confidence / pick-k controller (CPU only)."""

import itertools
import json
import math
import os

import numpy as np

from oracle import confidence, markov


def test_markov_bias_against_brute_force_loops():
    rng = np.random.default_rng(0)
    rows, V, R = 4, 9, 5
    d = rng.standard_normal((rows, V))
    w1 = rng.standard_normal((V, R)) * 0.1
    w2 = rng.standard_normal((R, V)) * 0.1
    prev = rng.integers(0, V, rows)
    out = markov.markov_bias(d, prev, w1, w2)
    for r in range(rows):
        for v in range(V):
            ref = math.fsum([d[r, v]] + [w1[prev[r], j] * w2[j, v] for j in range(R)])
            assert abs(out[r, v] - ref) < 1e-15


def test_markov_bias_special_cases():
    rng = np.random.default_rng(1)
    V, R = 12, 4
    d = rng.standard_normal((3, V))
    w2 = rng.standard_normal((R, V))
    w1 = np.zeros((V, R))
    w1[5, 2] = 1.0                                   # one-hot row: bias = W2[2]
    out = markov.markov_bias(d, [5, 0, 5], w1, w2)
    assert np.array_equal(out[0], d[0] + w2[2]) and np.array_equal(out[1], d[1])
    assert np.array_equal(markov.markov_bias(d, [1, 2, 3], w1 + 1, np.zeros((R, V))), d)
    bad = markov.markov_bias(d, [0, V, -1], w1, w2)   # invalid prev -> NaN row
    assert np.isfinite(bad[0]).all() and np.isnan(bad[1]).all() and np.isnan(bad[2]).all()


def test_prefix_survival_worked_example(golden_dir):
    with open(os.path.join(golden_dir, "prefix_survival.json")) as f:
        g = json.load(f)
    a = confidence.prefix_survival(g["c"])
    half = 0.5 * 10.0 ** -g["printed_decimals"]
    for got, printed in zip(a, g["a_printed"]):
        assert abs(got - printed) <= half + 1e-12
    assert (np.diff(a) <= 0).all()


def test_pick_k_worked_example_with_linear_table():
    """c = (.95, .90, .85, .40) with verify_ms[n] = 12 + 2.6 n: expected tokens per ms for
    n = 0..4 drafts are 1/14.6, 1.95/17.2, 2.805/19.8, 3.53175/22.4, 3.82245/25.0, so the
    controller verifies n = 3 drafts."""
    ratios = [1 / 14.6, 1.95 / 17.2, 2.805 / 19.8, 3.53175 / 22.4, 3.82245 / 25.0]
    assert int(np.argmax(ratios)) == 3
    table = 12.0 + 2.6 * np.arange(800)
    a = confidence.prefix_survival([[0.95, 0.90, 0.85, 0.40]])
    k, best = confidence.pick_k_per_stream(a, table)
    assert k[0] == 3 and abs(best[0] - ratios[3]) < 1e-12
    for n in range(5):
        assert abs(confidence.expected_tokens(a[0], n) / table[n + 1] - ratios[n]) < 1e-12


def test_tokens_per_step_identity(golden_dir):
    with open(os.path.join(golden_dir, "tokens_per_step.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        a = case["a"]
        got = confidence.expected_tokens(a, len(a))
        tol = 0.5 * 10.0 ** -case["printed_decimals"] + len(a) * 0.0005
        assert abs(got - case["tokens_per_step"]) <= tol, case["name"]


def test_sigmoid_closed_forms():
    assert confidence.sigmoid(0.0) == 0.5
    for x in (0.3, 2.0, 15.0, 700.0):
        assert abs(confidence.sigmoid(x) + confidence.sigmoid(-x) - 1.0) < 1e-15
    assert abs(confidence.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    h = np.zeros((1, 2, 3))
    h[0, 1] = [1.0, 2.0, 3.0]
    c = confidence.confidence(h, [0.5, -0.25, 0.1], 0.2)
    assert c[0, 0] == confidence.sigmoid(0.2)
    assert abs(c[0, 1] - confidence.sigmoid(0.5 - 0.5 + 0.3 + 0.2)) < 1e-15


def _brute_force_batch(a, table):
    B, kmax = a.shape
    best = -1.0
    for ks in itertools.product(range(kmax + 1), repeat=B):
        e = sum(confidence.expected_tokens(a[b], ks[b]) for b in range(B))
        best = max(best, e / table[B + sum(ks)])
    return best


def test_batch_greedy_is_exactly_optimal():
    rng = np.random.default_rng(3)
    for trial in range(40):
        B, kmax = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        a = confidence.prefix_survival(rng.uniform(0.2, 1.0, (B, kmax)))
        base = rng.uniform(0.5, 12)
        slope = rng.uniform(0.05, 3.0)
        table = base + slope * np.arange(B + B * kmax + 1) + rng.uniform(0, 0.2, B + B * kmax + 1).cumsum()
        k, m, v = confidence.pick_k_batch(a, table)
        assert abs(v - _brute_force_batch(a, table)) < 1e-12
        assert k.sum() == m and (k <= kmax).all()
        e = sum(confidence.expected_tokens(a[b], k[b]) for b in range(B))
        assert abs(e / table[B + m] - v) < 1e-12


def test_per_stream_pick_matches_brute_force():
    rng = np.random.default_rng(4)
    a = confidence.prefix_survival(rng.uniform(0.3, 1.0, (20, 5)))
    table = 12.0 + 2.6 * np.arange(10)
    k, _ = confidence.pick_k_per_stream(a, table)
    for b in range(20):
        vals = [confidence.expected_tokens(a[b], n) / table[n + 1] for n in range(6)]
        assert k[b] == int(np.argmax(vals))


def test_batch_order_keeps_per_stream_prefixes():
    rng = np.random.default_rng(5)
    c = rng.uniform(0.5, 1.0, (6, 4))
    c[2, 1:] = 1.0                                    # equal a values inside one stream
    a = confidence.prefix_survival(c)
    order = confidence.batch_order(a)
    for m in range(len(order) + 1):
        chosen = order[:m]
        for b in range(6):
            js = sorted(j for bb, j in chosen if bb == b)
            assert js == list(range(len(js)))


def test_cu_from_k():
    assert list(confidence.cu_from_k([2, 0, 3])) == [0, 2, 2, 5]
    assert list(confidence.cu_from_k([])) == [0]
