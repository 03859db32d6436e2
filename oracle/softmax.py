"""Temperature softmax of one logit row, in float64.

Test infrastructure (see ``oracle/__init__``).

P1 ("MTP, DSpark and Block Verification, Explained"), §4 "Verification: the guarantee": the
rules compare the target's distribution p_i and the drafter's q_i at each position; the lane
samples at temperature 1.0 (§5), and temperature 0 takes the greedy path (§4 "Greedy is a
different code path").  The same temperature T is applied to draft and target logits.

    p(v) = exp(l_v / T) / sum_u exp(l_u / T)

computed as exp((l_v - m)/T - log Z') with m = max_v l_v and Z' = sum_u exp((l_u - m)/T).
logZ below is the natural log of sum_u exp(l_u / T) = m/T + log Z'.

A row is invalid when it holds a NaN or +inf, or when every entry is -inf.
"""

import math

import numpy as np


def row_is_valid(l):
    """True iff the row has no NaN, no +inf and at least one finite entry."""
    l = np.asarray(l, dtype=np.float64)
    if l.size == 0:
        return False
    if np.isnan(l).any() or np.isposinf(l).any():
        return False
    return bool(np.isfinite(l).any())


def argmax_lowest(l):
    """Index of the largest entry; on ties the lowest index (numpy's first occurrence)."""
    return int(np.argmax(np.asarray(l, dtype=np.float64)))


def row_stats(l, T):
    """Softmax statistics of a valid row at temperature T > 0.

    Returns (m, logZ, logp) where logp is the float64 log-probability vector
    (-inf where the logit is -inf).
    """
    l = np.asarray(l, dtype=np.float64)
    T = float(T)
    m = float(np.max(l))
    z = (l - m) / T                     # -inf entries stay -inf
    log_zp = math.log(float(np.sum(np.exp(z))))
    logp = z - log_zp
    return m, m / T + log_zp, logp


def probs(l, T):
    """p = softmax(l / T) as a float64 vector (row must be valid, T > 0)."""
    return np.exp(row_stats(l, T)[2])
