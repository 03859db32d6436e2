"""Token-wise speculative sampling, block verification and the greedy branch, in float64.

Test infrastructure (see ``oracle/__init__``).

Notation (one stream): N draft slots i = 0..N-1 with draft tokens x_i; slot N is the
target-only bonus slot.  p_i, q_i are the target and draft distributions at slot i (slot i is
the position after i accepted drafts), both softmax(logits / T) with the stream's T.
rho_i = p_i(x_i) / q_i(x_i).

Token-wise rule - P1 "MTP, DSpark and Block Verification, Explained", §4 "Token by token"
(Leviathan et al. 2023): walk i = 0..N-1, accept x_i while u_i <= min(1, rho_i); at the
first rejection j emit Y ~ max(0, p_j - q_j) / sum and stop; if nothing is rejected emit the
bonus Y ~ p_N.  (The log-space form in §4 "Greedy is a different code path" differs only on
a set of measure zero; this restatement uses <=.)

Block verification - P1 §4 "Block verification" (Sun et al. 2024) and Figure 3:
    w_0 = 1,  w_{i+1} = min(1, w_i * rho_i)                       (clipped running product)
    r_i = sum_v max(0, w_i p_i(v) - q_i(v))                        (weighted residual mass)
    h_i = r_i / (r_i + 1 - w_i)   for 1 <= i <= N-1,   h_N = w_N
    tau = max{ i >= 1 : eta_i <= h_i },  or 0 if there is none
    emit x_0 .. x_{tau-1}, then Y ~ max(0, w_tau p_tau - q_tau) / r_tau  (tau < N)
                                  Y ~ p_N                               (tau = N)
Readings where the page is terse (each is pinned by exact enumeration in the tests):
  (a) the running product is clipped at 1 (the page's exp(cumulative_log_p) read unclipped
      gives h outside [0, 1]);
  (b) the residual is weighted by w_i (the unweighted form is not lossless);
  (c) 0/0 (r_i = 0 with w_i = 1) reads as h_i = 1;
  (d) eta_i is the acceptance uniform of draft slot i-1 (the same number the token-wise
      rule uses as u_{i-1}).

Greedy branch - P1 §4 "Greedy is a different code path": at T = 0 accept while
argmax p_i == x_i, emit argmax p_tau; this branch comes before the block branch, so the
block flag has no effect at T = 0.  argmax takes the lowest index on ties.

Residual / bonus draw: Y = the smallest v with C(v) >= U * R, C the ascending-index
cumulative sum of the non-negative weights and R their total (inverse CDF; never picks a
zero-weight token since U > 0).

Which rows a rule reads (this decides which invalid rows raise a status):
  T > 0: all 2N+1 rows of the stream (draft rows 0..N-1, target rows 0..N);
  T = 0: the N+1 target rows only.
Offsets: cu[0] = 0 and every draft count N_b = cu[b+1] - cu[b] in [0, kmax]; from the first
stream that breaks this on, every stream is BAD_OFFSETS (its rows have no defined position).
Status precedence per stream: BAD_OFFSETS, BAD_TEMPERATURE, BAD_TOKEN (any of the N draft
tokens outside [0, V)), BAD_ROW (a read row with NaN / +inf / no finite entry),
ZERO_DRAFT_PROB (T > 0 and q_i(x_i) = 0 at some slot), NUMERIC (zero residual mass where a
draw is needed).  A stream with a nonzero status emits nothing.

Near ties: the GPU computes in float32/float64 and this oracle in float64, so a decision
whose uniform lies within TIE_REL (relative) of its threshold is flagged; such streams are
counted and excluded from the exact comparison.
"""

import math

import numpy as np

from . import philox
from .softmax import argmax_lowest, row_is_valid, row_stats

STATUS_OK = 0
STATUS_BAD_TEMPERATURE = 1
STATUS_BAD_TOKEN = 2
STATUS_BAD_ROW = 3
STATUS_ZERO_DRAFT_PROB = 4
STATUS_BAD_OFFSETS = 5
STATUS_TIMEOUT = 6
STATUS_NUMERIC = 7

RULE_TOKENWISE = 0
RULE_BLOCK = 1

TIE_REL = 1e-6
FLT_MIN = 2.0 ** -126

# diag columns, one row per target row (stream b, slot i): target row index cu[b] + b + i
DIAG_COLS = 8
D_PX, D_QX, D_W, D_H, D_R, D_LOGZP, D_LOGZQ, D_RHO = range(DIAG_COLS)


# ----------------------------------------------------------------------------------------
# Distribution-level pieces (also driven directly by the exact-enumeration tests)
# ----------------------------------------------------------------------------------------

def running_weights(log_rho):
    """w_0..w_N of block verification from log rho_0..log rho_{N-1} (clipped product)."""
    logw = [0.0]
    for lr in log_rho:
        logw.append(min(0.0, logw[-1] + lr))
    return [math.exp(v) for v in logw]


def residual_weights(w, p, q):
    """Elementwise max(0, w p - q) (float64 vectors)."""
    return np.maximum(0.0, w * np.asarray(p, np.float64) - np.asarray(q, np.float64))


def block_h(w, r):
    """h_1..h_N (index 0 unused, NaN) from w_0..w_N and r_0..r_{N-1}."""
    n = len(w) - 1
    h = [float("nan")] * (n + 1)
    for i in range(1, n):
        den = r[i] + 1.0 - w[i]
        h[i] = 1.0 if den == 0.0 else r[i] / den
    if n >= 1:
        h[n] = w[n]
    return h


def block_tau(eta, h):
    """tau = max{i >= 1: eta_i <= h_i}, else 0 (eta, h indexed 1..N; index 0 unused)."""
    tau = 0
    for i in range(1, len(h)):
        if eta[i] <= h[i]:
            tau = i
    return tau


def inverse_cdf(weights, u):
    """(Y, margin): Y = smallest v with C(v) >= u * R; margin = relative distance of u*R to
    the two thresholds that decide Y, C(Y) and C(Y-1), each relative to the threshold itself
    (a small margin is a near tie)."""
    c = np.cumsum(np.asarray(weights, np.float64))
    total = float(c[-1])
    t = u * total
    y = int(np.searchsorted(c, t, side="left"))
    y = min(y, len(c) - 1)
    hi = float(c[y])
    margin = abs(t - hi) / hi
    if y > 0 and float(c[y - 1]) > 0.0:
        lo = float(c[y - 1])
        margin = min(margin, abs(t - lo) / lo)
    return y, margin


def _near(a, b):
    return abs(a - b) <= TIE_REL * max(abs(a), abs(b))


# ----------------------------------------------------------------------------------------
# One stream, from logits
# ----------------------------------------------------------------------------------------

def _empty_result(n, status):
    return {"status": status, "tau": 0, "emitted": [], "n_emitted": 0, "tie": False,
            "tie_kind": None, "diag": np.full((n + 1, DIAG_COLS), np.nan)}


def temperature_ok(T):
    T = float(T)
    return math.isfinite(T) and (T == 0.0 or T >= FLT_MIN)


def verify_stream(rule, q_rows, p_rows, x, T, seed, step, stream):
    """Verify one stream.

    q_rows: N draft logit rows, p_rows: N+1 target logit rows (any float dtype; widened
    exactly to float64), x: N draft tokens, T: temperature (0 = greedy).
    Returns a dict: status, tau, emitted (list), n_emitted, tie, tie_kind, diag [(N+1), 8].
    """
    n = len(x)
    V = len(p_rows[0])
    T = float(T)
    if not temperature_ok(T):
        return _empty_result(n, STATUS_BAD_TEMPERATURE)
    xs = [int(v) for v in x]
    if any(v < 0 or v >= V for v in xs):
        return _empty_result(n, STATUS_BAD_TOKEN)

    if T == 0.0:
        return _greedy(p_rows, xs)

    qr = [np.asarray(r, np.float64) for r in q_rows]
    pr = [np.asarray(r, np.float64) for r in p_rows]
    if not all(row_is_valid(r) for r in qr + pr):
        return _empty_result(n, STATUS_BAD_ROW)
    if any(qr[i][xs[i]] == -np.inf for i in range(n)):
        return _empty_result(n, STATUS_ZERO_DRAFT_PROB)

    res = _empty_result(n, STATUS_OK)
    diag = res["diag"]
    ps, qs = [], []
    for i in range(n + 1):
        _, lzp, logp = row_stats(pr[i], T)
        ps.append(logp)
        diag[i, D_LOGZP] = lzp
    log_rho = []
    for i in range(n):
        _, lzq, logq = row_stats(qr[i], T)
        qs.append(logq)
        lr = ps[i][xs[i]] - logq[xs[i]]
        log_rho.append(lr)
        diag[i, D_PX] = math.exp(ps[i][xs[i]])
        diag[i, D_QX] = math.exp(logq[xs[i]])
        diag[i, D_LOGZQ] = lzq
        diag[i, D_RHO] = math.exp(lr)

    if rule == RULE_TOKENWISE:
        return _tokenwise(res, ps, qs, xs, log_rho, seed, step, stream)
    return _block(res, ps, qs, xs, log_rho, seed, step, stream)


def _finish(res, tau, xs, weights, u_sample):
    total = float(np.sum(weights))
    if not (total > 0.0 and math.isfinite(total)):
        out = _empty_result(len(xs), STATUS_NUMERIC)
        out["diag"] = res["diag"]
        return out
    y, margin = inverse_cdf(weights, u_sample)
    if margin <= TIE_REL and not res["tie"]:
        res["tie"], res["tie_kind"] = True, "sample"
    res["tau"] = tau
    res["emitted"] = xs[:tau] + [y]
    res["n_emitted"] = tau + 1
    return res


def _tokenwise(res, ps, qs, xs, log_rho, seed, step, stream):
    n = len(xs)
    for i in range(n):
        u, us = philox.slot_uniforms(seed, step, stream, i)
        acc = min(1.0, math.exp(log_rho[i]))
        if _near(u, acc) and not res["tie"]:
            res["tie"], res["tie_kind"] = True, "accept"
        if u <= acc:
            continue
        p = np.exp(ps[i])
        q = np.exp(qs[i])
        wts = residual_weights(1.0, p, q)
        res["diag"][i, D_R] = float(np.sum(wts))
        return _finish(res, i, xs, wts, us)
    _, us = philox.slot_uniforms(seed, step, stream, n)
    return _finish(res, n, xs, np.exp(ps[n]), us)


def _block(res, ps, qs, xs, log_rho, seed, step, stream):
    n = len(xs)
    diag = res["diag"]
    w = running_weights(log_rho)
    for i in range(n + 1):
        diag[i, D_W] = w[i]
    r = [float("nan")] * (n + 1)
    for i in range(0, n):
        r[i] = float(np.sum(residual_weights(w[i], np.exp(ps[i]), np.exp(qs[i]))))
        diag[i, D_R] = r[i]
    h = block_h(w, r)
    for i in range(1, n + 1):
        diag[i, D_H] = h[i]
    eta = [float("nan")] + [philox.slot_uniforms(seed, step, stream, i - 1)[0]
                            for i in range(1, n + 1)]
    tau = block_tau(eta, h)
    # a comparison whose flip would change tau: every i >= tau (all of them when tau = 0)
    for i in range(max(tau, 1), n + 1):
        if _near(eta[i], h[i]) and not res["tie"]:
            res["tie"], res["tie_kind"] = True, "block"
    _, us = philox.slot_uniforms(seed, step, stream, tau)
    if tau == n:
        return _finish(res, tau, xs, np.exp(ps[n]), us)
    wts = residual_weights(w[tau], np.exp(ps[tau]), np.exp(qs[tau]))
    return _finish(res, tau, xs, wts, us)


def _greedy(p_rows, xs):
    n = len(xs)
    pr = [np.asarray(r, np.float64) for r in p_rows]
    if not all(row_is_valid(r) for r in pr):
        return _empty_result(n, STATUS_BAD_ROW)
    res = _empty_result(n, STATUS_OK)
    tau = n
    for i in range(n):
        if argmax_lowest(pr[i]) != xs[i]:
            tau = i
            break
    res["tau"] = tau
    res["emitted"] = xs[:tau] + [argmax_lowest(pr[tau])]
    res["n_emitted"] = tau + 1
    return res


# ----------------------------------------------------------------------------------------
# Batch, in the C-ABI layout
# ----------------------------------------------------------------------------------------

def verify_batch(rule, cu_drafts, draft_logits, target_logits, draft_tokens, temperature,
                 kmax, seed, step, streams=None):
    """Mirror of spec_verify_tokenwise / spec_verify_block.

    cu_drafts [B+1]; draft row of (b, i) = cu[b] + i; target row of (b, i) = cu[b] + b + i.
    draft_logits [cu[B], V], target_logits [cu[B] + B, V] (row-indexable float arrays),
    draft_tokens [cu[B]], temperature [B].  ``streams`` restricts the work to a subset (the
    other streams' outputs are left at their fill values: status -1).
    Returns dict of numpy arrays: accepted_len, out_tokens [B, kmax+1] (-1 padded),
    n_emitted, status, diag [cu[B] + B, 8], tie (bool) and tie_kind (list).
    """
    cu = [int(v) for v in np.asarray(cu_drafts)]
    B = len(cu) - 1
    tokens = np.asarray(draft_tokens)
    temps = np.asarray(temperature, dtype=np.float32).astype(np.float64)
    out = {
        "accepted_len": np.zeros(B, np.int32),
        "out_tokens": np.full((B, kmax + 1), -1, np.int32),
        "n_emitted": np.zeros(B, np.int32),
        "status": np.full(B, -1, np.int32),
        "diag": np.full((max(cu[-1] + B, 0), DIAG_COLS), np.nan),
        "tie": np.zeros(B, bool),
        "tie_kind": [None] * B,
    }
    # Streams are packed from row 0 in order.  The first stream whose draft count lies
    # outside [0, kmax] (or cu[0] != 0) leaves the row positions of every later stream
    # undefined, so from there on every stream is BAD_OFFSETS.
    first_bad = B
    for b in range(B):
        n = cu[b + 1] - cu[b]
        if n < 0 or n > kmax or (b == 0 and cu[0] != 0):
            first_bad = b
            break
    todo = range(B) if streams is None else streams
    for b in todo:
        n = cu[b + 1] - cu[b]
        if b >= first_bad:
            out["status"][b] = STATUS_BAD_OFFSETS
            continue
        q_rows = [draft_logits[cu[b] + i] for i in range(n)]
        p_rows = [target_logits[cu[b] + b + i] for i in range(n + 1)]
        x = tokens[cu[b]:cu[b] + n]
        r = verify_stream(rule, q_rows, p_rows, x, temps[b], seed, step, b)
        out["status"][b] = r["status"]
        out["tie"][b] = r["tie"]
        out["tie_kind"][b] = r["tie_kind"]
        if r["status"] == STATUS_OK:
            out["accepted_len"][b] = r["tau"]
            out["n_emitted"][b] = r["n_emitted"]
            out["out_tokens"][b, :len(r["emitted"])] = r["emitted"]
        if float(temps[b]) > 0.0 and r["status"] in (STATUS_OK, STATUS_NUMERIC):
            out["diag"][cu[b] + b: cu[b] + b + n + 1] = r["diag"]
    return out
