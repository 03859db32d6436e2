"""Exact enumeration of the verify rules on tiny vocabularies (test helper, CPU only).

Given conditional tables P(.|prefix) for prefixes of length 0..N and Q(.|prefix) for
prefixes of length 0..N-1, enumerate every draft string x ~ Q and every outcome of a rule,
with the outcome probabilities written in closed form:

* token-wise: P[accept slot i | slot i reached] = min(1, p_i(x_i) / q_i(x_i));
* block: with independent uniforms eta_1..eta_N and tau = max{i: eta_i <= h_i},
  P[tau = t] = h_t * prod_{j>t} (1 - h_j) for t >= 1 and prod_{j>=1} (1 - h_j) for t = 0.

The per-slot quantities (w, r, h, the residual distribution) come from the oracle's own
functions; the result is compared with the target's own sequential distribution, which
involves none of them.
"""

import itertools
import math

import numpy as np

from oracle import verify


def random_tables(V, N, rng, alpha=1.0):
    P, Q = {}, {}
    for L in range(N + 1):
        for pre in itertools.product(range(V), repeat=L):
            P[pre] = rng.dirichlet(np.full(V, alpha))
            if L < N:
                Q[pre] = rng.dirichlet(np.full(V, alpha))
    return P, Q


def _norm(w):
    w = np.asarray(w, np.float64)
    return w / w.sum()


def tokenwise_outcomes(p, q, x):
    """[(tau, Y-distribution, probability)] for one draft string."""
    n = len(x)
    out, reach = [], 1.0
    for i in range(n):
        a = min(1.0, p[i][x[i]] / q[i][x[i]])
        if a < 1.0:
            out.append((i, _norm(verify.residual_weights(1.0, p[i], q[i])), reach * (1 - a)))
        reach *= a
    out.append((n, np.asarray(p[n]), reach))
    return out


def block_outcomes(p, q, x):
    n = len(x)
    log_rho = [math.log(p[i][x[i]]) - math.log(q[i][x[i]]) for i in range(n)]
    w = verify.running_weights(log_rho)
    r = [float("nan")] + [float(np.sum(verify.residual_weights(w[i], p[i], q[i])))
                          for i in range(1, n)]
    h = verify.block_h(w, r)
    out = []
    for t in range(n + 1):
        pr = h[t] if t >= 1 else 1.0
        for j in range(t + 1, n + 1):
            pr *= 1.0 - h[j]
        if pr == 0.0:
            continue
        if t == n:
            y = np.asarray(p[n])
        else:
            y = _norm(verify.residual_weights(w[t], p[t], q[t]))
        out.append((t, y, pr))
    return out


def emitted_distribution(P, Q, V, N, outcomes_fn):
    """Distribution over emitted token tuples (length 1..N+1) and E[tau]."""
    dist, e_tau = {}, 0.0
    for x in itertools.product(range(V), repeat=N):
        px = 1.0
        for i in range(N):
            px *= Q[x[:i]][x[i]]
        if px == 0.0:
            continue
        p = [P[x[:i]] for i in range(N + 1)]
        q = [Q[x[:i]] for i in range(N)]
        for t, ydist, pr in outcomes_fn(p, q, list(x)):
            e_tau += px * pr * t
            for y in range(V):
                if ydist[y] > 0:
                    key = x[:t] + (y,)
                    dist[key] = dist.get(key, 0.0) + px * pr * ydist[y]
    return dist, e_tau


def max_violation(P, V, N, dist):
    """max over s in V^(N+1) of |P_method(s) - P_target(s)|, after extending each emitted
    prefix with target sampling."""
    worst = 0.0
    for s in itertools.product(range(V), repeat=N + 1):
        target = 1.0
        for k in range(N + 1):
            target *= P[s[:k]][s[k]]
        method = 0.0
        for t in range(N + 1):
            pre = s[:t + 1]
            if pre in dist:
                ext = 1.0
                for k in range(t + 1, N + 1):
                    ext *= P[s[:k]][s[k]]
                method += dist[pre] * ext
        worst = max(worst, abs(method - target))
    return worst
