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
"""

import numpy as np


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
