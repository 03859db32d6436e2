"""The Markov head's low-rank previous-token logit bias, in float64.

Test infrastructure (see ``oracle/__init__``).

P2 "MTP Heads and Confidence Heads", §6 "Why the Markov Head Helps": the head is a low-rank
logit bias B = W1 @ W2 (default rank 256) added to the current draft logits according to the
previous token.  P1 "MTP, DSpark and Block Verification, Explained", §3 "The Markov fix-up"
and Figure 2: it is sampling-time arithmetic that biases slot i's logits by the token
sampled at slot i-1 (slot 0 by the anchor).  So for draft row r with previous token prev_r:

    l~[r, v] = l[r, v] + sum_j W1[prev_r, j] * W2[j, v]

Readings: the bias is added to the logits before the temperature is applied (the page says
it "biases each slot's logits"); prev is an explicit input per row.  A row whose prev token
lies outside [0, V) has no defined bias: its output row is all NaN (a downstream verify then
reports that row as invalid).

The walk (P1 §3 "The Markov fix-up", Figure 2: "slot 1 bias(t0)", ...): the drafter's forward
gives N slot logits l_0 .. l_{N-1} at once; the walk then goes left to right, biasing slot i
by the token sampled at slot i-1 (slot 0 by the anchor, the last token the target emitted)
and sampling t_i from softmax(l~_i / T).  Readings where the page is terse: the draw is the
verify's inverse CDF (the smallest v with C(v) >= U R over softmax weights) with the
draft-side uniform of (stream, slot) (Philox word 2, see ``philox``); T = 0 takes the argmax
(lowest index on ties), as the greedy verify does.
"""

import numpy as np

from . import philox
from .softmax import argmax_lowest, row_is_valid, row_stats
from .verify import inverse_cdf, temperature_ok


def markov_bias(draft_logits, prev_tokens, W1, W2):
    """float64 [rows, V] = draft + W1[prev] @ W2 (rows with an invalid prev become NaN)."""
    d = np.asarray(draft_logits, np.float64)
    prev = np.asarray(prev_tokens, np.int64)
    w1 = np.asarray(W1, np.float64)
    w2 = np.asarray(W2, np.float64)
    V = w2.shape[1]
    ok = (prev >= 0) & (prev < w1.shape[0]) & (prev < V)
    gathered = w1[np.where(ok, prev, 0)]
    out = d + gathered @ w2
    out[~ok] = np.nan
    return out


def walk(draft_logits, anchor, W1, W2, T, seed, step, stream):
    """The Markov walk of one stream, in float64.

    draft_logits [N, V] (the drafter's unbiased slot logits), anchor (token), W1 [V, R],
    W2 [R, V], T (0 = greedy).  Returns a dict: status ("ok", "bad_anchor", "bad_temperature",
    "bad_row"), tokens [N] (int), biased [N, V] float64 (the rows the draft q is taken from),
    windows [N] (the admissible tokens of each draw: more than one is a near tie, and every
    later slot then depends on which one the sampler took).
    """
    d = np.asarray(draft_logits, np.float64)
    n, V = d.shape
    out = {"status": "ok", "tokens": [], "biased": np.full((n, V), np.nan), "windows": []}
    if not temperature_ok(T):
        out["status"] = "bad_temperature"
        return out
    if not (0 <= int(anchor) < V):
        out["status"] = "bad_anchor"
        return out
    prev = int(anchor)
    for i in range(n):
        row = markov_bias(d[i:i + 1], [prev], W1, W2)[0]
        out["biased"][i] = row
        if not row_is_valid(row):
            out["status"] = "bad_row"
            return out
        if float(T) == 0.0:
            t = argmax_lowest(row)
            window = [t]
        else:
            _, _, logp = row_stats(row, T)
            t, window = inverse_cdf(np.exp(logp), philox.draft_uniform(seed, step, stream, i))
        out["tokens"].append(t)
        out["windows"].append(window)
        prev = t
    return out
