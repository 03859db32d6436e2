"""The oracle's Markov walk (P1 "MTP, DSpark and Block Verification, Explained", §3 "The Markov
fix-up" and Figure 2) pinned on the CPU.

* Distribution: at V = 4, N = 3 the walk's token sequences, over many steps (the draft-side
  Philox uniforms), follow the product of the conditional softmaxes
  prod_i softmax((l_i + W1[t_{i-1}] W2) / T)(t_i), t_{-1} = the anchor, written out here
  with plain numpy (chi-square).  A planted mistake - biasing every slot by token 0 instead
  of the previous sample - fails the same check.
* Greedy closed form: with W1 the identity and W2 a scaled cyclic shift, the bias makes
  prev + 1 (mod V) the argmax, so T = 0 walks anchor + 1, anchor + 2, ...
* Statuses: an anchor outside [0, V), a negative temperature.
"""

import itertools

import numpy as np
import pytest
from scipy import stats

from oracle import markov as om


def _setup(seed=3, V=4, N=3, R=4):
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((N, V))
    w1 = rng.standard_normal((V, R)) * 0.8
    w2 = rng.standard_normal((R, V)) * 0.8
    return d, w1, w2


def _exact(d, w1, w2, anchor, T):
    """P(t_0 .. t_{N-1}) from the conditional softmaxes, written out directly."""
    N, V = d.shape
    probs = {}
    for seq in itertools.product(range(V), repeat=N):
        prev, p = anchor, 1.0
        for i, t in enumerate(seq):
            z = (d[i] + w1[prev] @ w2) / T
            e = np.exp(z - z.max())
            p *= e[t] / e.sum()
            prev = t
        probs[seq] = p
    return probs


def _chi2_pvalue(walk_fn, steps=6000, T=0.8, anchor=1):
    d, w1, w2 = _setup()
    exact = _exact(d, w1, w2, anchor, T)
    counts = dict.fromkeys(exact, 0)
    for st in range(steps):
        r = walk_fn(d, anchor, w1, w2, T, 11, st, 5)
        counts[tuple(r["tokens"])] += 1
    keys = sorted(exact)
    obs = np.array([counts[k] for k in keys], np.float64)
    exp = np.array([exact[k] for k in keys]) * steps
    big = exp >= 5
    o = np.append(obs[big], obs[~big].sum())
    e = np.append(exp[big], exp[~big].sum())
    return stats.chisquare(o, e).pvalue


def test_walk_sequences_follow_the_conditional_softmaxes():
    assert abs(sum(_exact(*_setup(), 1, 0.8).values()) - 1.0) < 1e-12
    assert _chi2_pvalue(om.walk) > 1e-4


def test_planted_walk_without_the_previous_token_is_caught(monkeypatch):
    real = om.markov_bias
    monkeypatch.setattr(om, "markov_bias", lambda d, prev, w1, w2: real(d, [0] * len(prev), w1, w2))
    assert _chi2_pvalue(om.walk) < 1e-6


def test_greedy_walk_closed_form():
    V, N = 6, 5
    d = np.zeros((N, V))
    w1 = np.eye(V)
    w2 = np.roll(np.eye(V), 1, axis=1) * 3.0      # W1[p] @ W2 = 3 e_{(p + 1) mod V}
    r = om.walk(d, 2, w1, w2, 0.0, 0, 0, 0)
    assert r["status"] == "ok" and r["tokens"] == [3, 4, 5, 0, 1]
    assert np.array_equal(r["biased"][0], 3.0 * np.eye(V)[3])
    assert all(w == [t] for w, t in zip(r["windows"], r["tokens"]))


def test_walk_statuses():
    d, w1, w2 = _setup()
    assert om.walk(d, 4, w1, w2, 1.0, 0, 0, 0)["status"] == "bad_anchor"
    assert om.walk(d, -1, w1, w2, 1.0, 0, 0, 0)["status"] == "bad_anchor"
    assert om.walk(d, 0, w1, w2, -0.5, 0, 0, 0)["status"] == "bad_temperature"
    bad = d.copy()
    bad[1, 2] = np.nan
    r = om.walk(bad, 0, w1, w2, 1.0, 0, 0, 0)
    assert r["status"] == "bad_row" and len(r["tokens"]) == 1
