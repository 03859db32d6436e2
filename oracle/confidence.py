"""Confidence head, prefix survival and the adaptive-verification controller, in float64.

Test infrastructure (see ``oracle/__init__``).

P2 "MTP Heads and Confidence Heads", §7 "Only Then Comes the Confidence Head":
    c_k = sigmoid(Linear(h_k)) = 1 / (1 + exp(-(h_k . w + beta)))
is the conditional acceptance probability of draft k given all earlier drafts accepted.
§9 "Why It Is Called Prefix Survival Probability": a_j = prod_{i<=j} c_i (non-increasing).
P1 §6 "The arithmetic you need before tuning k": tokens/step = 1 + sum_p a_p, so verifying
the first n drafts of a stream is expected to yield E_n = 1 + sum_{j<=n} a_j tokens.
P3 "Teaching the Speculator What a Draft Costs", "The controller, and the table it reads
from": before each step pick the count with the best expected tokens per millisecond, the
cost read from verify_ms[num_tokens].

Per-stream mode (mode 0; the reading used for the adaptive-verification workload):
    k_b = argmax_{n in 0..kmax} E_n / verify_ms[n + 1]     (n drafts + 1 bonus token;
                                                          ties -> the smaller n)
Batch mode (mode 1; the figure text after P2 §9: "greedily add candidates in descending
a_j ... truncating the low-confidence tail"): order all (stream, j) by (a desc, stream asc,
j asc), S_m = sum of the first m, m* = argmax_m (B + S_m) / verify_ms[B + m] (ties -> the
smaller m), k_b = number of stream b's entries among the first m*.  Because a is
non-increasing along j, every such prefix keeps each stream's selection a prefix.
"""

import math

import numpy as np


def sigmoid(x):
    x = float(x)
    if x >= 0:
        return 1.0 / (1.0 + math.exp(-x))
    e = math.exp(x)
    return e / (1.0 + e)


def confidence(hidden, w, beta):
    """c [B, kmax] from hidden [B, kmax, H], w [H] and the scalar bias beta."""
    h = np.asarray(hidden, np.float64)
    wv = np.asarray(w, np.float64)
    logits = h @ wv + float(beta)
    return np.vectorize(sigmoid, otypes=[np.float64])(logits)


def prefix_survival(c):
    """a [.., kmax] = cumulative product of c along the last axis."""
    return np.cumprod(np.asarray(c, np.float64), axis=-1)


def expected_tokens(a_row, n):
    """E_n = 1 + sum of the first n prefix-survival values of one stream."""
    return 1.0 + float(sum(float(v) for v in a_row[:n]))


def pick_k_per_stream(a, verify_ms):
    """k [B] (mode 0) and the winning ratio per stream."""
    a = np.asarray(a, np.float64)
    B, kmax = a.shape
    k = np.zeros(B, np.int32)
    best = np.zeros(B)
    for b in range(B):
        bn, bv = 0, -math.inf
        for n in range(kmax + 1):
            v = expected_tokens(a[b], n) / float(verify_ms[n + 1])
            if v > bv:
                bn, bv = n, v
        k[b], best[b] = bn, bv
    return k, best


def batch_order(a):
    """The (stream, j) entries in the batch mode's order (a desc, stream asc, j asc)."""
    a = np.asarray(a, np.float64)
    B, kmax = a.shape
    entries = [(-a[b, j], b, j) for b in range(B) for j in range(kmax)]
    entries.sort()
    return [(b, j) for _, b, j in entries]


def pick_k_batch(a, verify_ms):
    """k [B] (mode 1), m* and the winning batch ratio."""
    a = np.asarray(a, np.float64)
    B, kmax = a.shape
    order = batch_order(a)
    best_m, best_v = 0, B / float(verify_ms[B])
    s = 0.0
    for m in range(1, len(order) + 1):
        b, j = order[m - 1]
        s += a[b, j]
        v = (B + s) / float(verify_ms[B + m])
        if v > best_v:
            best_m, best_v = m, v
    k = np.zeros(B, np.int32)
    for b, _ in order[:best_m]:
        k[b] += 1
    return k, best_m, best_v


def cu_from_k(k):
    """Exclusive prefix sum: cu [B+1] with cu[0] = 0."""
    k = np.asarray(k, np.int64)
    return np.concatenate([[0], np.cumsum(k)]).astype(np.int32)
