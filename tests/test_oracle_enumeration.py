"""The oracle's verify rules pinned by exact enumeration and by their uniform-driven path.

* Losslessness (P1 "MTP, DSpark and Block Verification, Explained", §4: the output
  distribution is unchanged; Figure 3: both verifiers are lossless): for random conditional
  tables at V = 8 and N <= 3, the emitted sequence, continued by target sampling, has
  exactly the target's distribution (to 1e-12).
* Optimality (P1 §4 "Block verification": never worse than the token-level test):
  E[tau]_block >= E[tau]_token.
* Sensitivity: the same check rejects the readings that were not taken (unweighted
  residual, unclipped running product), so it pins the chosen ones.
* The uniform-driven oracle (Philox uniforms, inverse-CDF draws) agrees with the exact
  outcome probabilities (chi-square).
"""

import itertools
import math

import numpy as np
import pytest
from scipy import stats

from oracle import verify
from tests import enumeration as en


@pytest.mark.parametrize("V,N,seed", [(8, 1, 0), (8, 2, 1), (8, 3, 2), (4, 3, 3), (8, 3, 4)])
def test_lossless_both_rules(V, N, seed):
    rng = np.random.default_rng(seed)
    P, Q = en.random_tables(V, N, rng, alpha=0.7)
    for fn in (en.tokenwise_outcomes, en.block_outcomes):
        dist, _ = en.emitted_distribution(P, Q, V, N, fn)
        assert abs(sum(dist.values()) - 1.0) < 1e-12
        assert en.max_violation(P, V, N, dist) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_block_never_worse_than_tokenwise(seed):
    V, N = 6, 3
    rng = np.random.default_rng(100 + seed)
    P, Q = en.random_tables(V, N, rng, alpha=0.5 + seed * 0.3)
    _, e_tok = en.emitted_distribution(P, Q, V, N, en.tokenwise_outcomes)
    _, e_blk = en.emitted_distribution(P, Q, V, N, en.block_outcomes)
    assert e_blk >= e_tok - 1e-12


def test_h_in_unit_interval_and_bounded_by_w():
    rng = np.random.default_rng(7)
    V, N = 8, 3
    P, Q = en.random_tables(V, N, rng, alpha=0.4)
    for x in itertools.product(range(V), repeat=N):
        p = [P[x[:i]] for i in range(N + 1)]
        q = [Q[x[:i]] for i in range(N)]
        w = verify.running_weights([math.log(p[i][x[i]] / q[i][x[i]]) for i in range(N)])
        r = [float("nan")] + [float(np.sum(verify.residual_weights(w[i], p[i], q[i])))
                              for i in range(1, N)]
        h = verify.block_h(w, r)
        for i in range(1, N + 1):
            assert 0.0 <= h[i] <= w[i] + 1e-15 <= 1.0 + 1e-15


def test_unweighted_residual_is_not_lossless(monkeypatch):
    """Planted mistake (in the oracle, on the CPU): drop the w_i weight of the residual."""
    V, N = 4, 3
    P, Q = en.random_tables(V, N, np.random.default_rng(11), alpha=0.7)
    real = verify.residual_weights
    monkeypatch.setattr(verify, "residual_weights", lambda w, p, q: real(1.0, p, q))
    dist, _ = en.emitted_distribution(P, Q, V, N, en.block_outcomes)
    assert en.max_violation(P, V, N, dist) > 1e-3


def test_unclipped_running_product_is_invalid(monkeypatch):
    """Planted mistake: read the page's exp(cumulative_log_p) without the clip at 1."""
    V, N = 4, 3
    P, Q = en.random_tables(V, N, np.random.default_rng(12), alpha=0.7)
    monkeypatch.setattr(verify, "running_weights",
                        lambda lr: [math.exp(v) for v in np.concatenate([[0.0], np.cumsum(lr)])])
    bad = False
    for x in itertools.product(range(V), repeat=N):
        p = [P[x[:i]] for i in range(N + 1)]
        q = [Q[x[:i]] for i in range(N)]
        for _, _, pr in en.block_outcomes(p, q, list(x)):
            bad |= not (0.0 <= pr <= 1.0)
    if not bad:
        dist, _ = en.emitted_distribution(P, Q, V, N, en.block_outcomes)
        bad = en.max_violation(P, V, N, dist) > 1e-3
    assert bad


def test_tokenwise_rule_without_residual_is_not_lossless(monkeypatch):
    """Planted mistake: resample the correction from p instead of the residual."""
    V, N = 4, 2
    P, Q = en.random_tables(V, N, np.random.default_rng(13), alpha=0.7)
    monkeypatch.setattr(verify, "residual_weights", lambda w, p, q: np.asarray(p, np.float64))
    dist, _ = en.emitted_distribution(P, Q, V, N, en.tokenwise_outcomes)
    assert en.max_violation(P, V, N, dist) > 1e-3


def _chi2_against_exact(rule, outcomes_fn, seed, M):
    V, N = 6, 3
    rng = np.random.default_rng(seed)
    P, Q = en.random_tables(V, N, rng, alpha=0.8)
    x = []
    for i in range(N):                       # one draft string drawn from Q
        x.append(int(rng.choice(V, p=Q[tuple(x)])))
    p = [P[tuple(x[:i])] for i in range(N + 1)]
    q = [Q[tuple(x[:i])] for i in range(N)]
    expected = {}
    for t, ydist, pr in outcomes_fn(p, q, x):
        for y in range(V):
            if ydist[y] * pr > 0:
                expected[(t, y)] = expected.get((t, y), 0.0) + ydist[y] * pr
    q_rows = [np.log(v) for v in q]
    p_rows = [np.log(v) for v in p]
    counts = {}
    for step in range(M):
        r = verify.verify_stream(rule, q_rows, p_rows, x, 1.0, seed=99, step=step, stream=5)
        assert r["status"] == verify.STATUS_OK
        assert r["emitted"][:r["tau"]] == x[:r["tau"]]
        key = (r["tau"], r["emitted"][-1])
        assert key in expected, key
        counts[key] = counts.get(key, 0) + 1
    keys = sorted(expected)
    obs = np.array([counts.get(k, 0) for k in keys], float)
    exp = np.array([expected[k] * M for k in keys])
    big = exp >= 5                            # pool sparse cells
    obs_b = np.append(obs[big], obs[~big].sum())
    exp_b = np.append(exp[big], exp[~big].sum())
    if exp_b[-1] == 0:
        obs_b, exp_b = obs_b[:-1], exp_b[:-1]
    return stats.chisquare(obs_b, exp_b).pvalue


def test_uniform_driven_tokenwise_matches_enumeration():
    assert _chi2_against_exact(verify.RULE_TOKENWISE, en.tokenwise_outcomes, 21, 6000) > 1e-4


def test_uniform_driven_block_matches_enumeration():
    assert _chi2_against_exact(verify.RULE_BLOCK, en.block_outcomes, 22, 6000) > 1e-4
