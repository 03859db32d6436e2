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

Near ties: the GPU computes in float32 and double-float, this oracle in float64, so a
decision whose uniform lies within TIE_REL (relative) of its threshold is flagged, and so is a
draw whose target U R lies within TIE_REL (relative) of a CDF value that decides the token.
For such a stream the result also lists every outcome a computation with that much relative
error may reach: each (tau, tokens) pair obtained by flipping any subset of the near
comparisons (and nothing else), with, for that tau, every positive-weight token whose CDF
interval meets the draw's window.  A flagged stream is then checked against that list, not
skipped.
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


def residual_gross(w, p, q):
    """sum_v [w p(v) > q(v)] w p(v): the positive part's gross mass, an upper bound of the
    residual mass.  Float32 per-element arithmetic computes each term of the residual with an
    error proportional to w p(v) + q(v), so where the residual is a small difference of large
    terms its attainable relative accuracy is set by this mass, not by the residual itself."""
    wp = w * np.asarray(p, np.float64)
    return float(np.sum(np.where(wp > np.asarray(q, np.float64), wp, 0.0)))


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


def window_bounds(t, total):
    """The CDF window of a draw with target t = U R: [t (1 - TIE_REL), t (1 + TIE_REL)]."""
    return t * (1.0 - TIE_REL), t * (1.0 + TIE_REL)


def inverse_cdf(weights, u):
    """(Y, window): Y = the smallest v with C(v) >= u * R (C the ascending-index cumulative sum
    of the non-negative weights, R their total).  ``window`` lists, in ascending order, every
    token with positive weight whose CDF interval [C(v-1), C(v)] meets window_bounds(u R): the
    tokens a sampler whose partial sums carry a relative error below TIE_REL may return.  Y is
    always one of them; more than one is a near tie."""
    w = np.asarray(weights, np.float64)
    c = np.cumsum(w)
    total = float(c[-1])
    t = u * total
    y = min(int(np.searchsorted(c, t, side="left")), len(c) - 1)
    lo_t, hi_t = window_bounds(t, total)
    lo = min(int(np.searchsorted(c, lo_t, side="left")), len(c) - 1)
    hi = min(int(np.searchsorted(c, hi_t, side="left")), len(c) - 1)
    window = [v for v in range(lo, hi + 1) if w[v] > 0.0]
    if y not in window:   # only when every weight is zero; the caller rejects that total
        window = sorted(set(window) | {y})
    return y, window


def _near(a, b):
    """A comparison a <= b is a near tie when a lies within TIE_REL (relative) of b."""
    return abs(a - b) <= TIE_REL * max(abs(a), abs(b))


def _flip_outcomes(passed, near, decide, limit=10):
    """Every tau reachable by flipping any subset of the near comparisons (at most ``limit`` of
    them are enumerated), in first-seen order starting with the unflipped tau."""
    idx = [i for i in range(len(passed)) if near[i]][:limit]
    seen = []
    for mask in range(1 << len(idx)):
        flipped = list(passed)
        for j, i in enumerate(idx):
            if (mask >> j) & 1:
                flipped[i] = not flipped[i]
        t = decide(flipped)
        if t not in seen:
            seen.append(t)
    return seen


# ----------------------------------------------------------------------------------------
# One stream, from logits
# ----------------------------------------------------------------------------------------

def _empty_result(n, status):
    return {"status": status, "tau": 0, "emitted": [], "n_emitted": 0, "tie": False,
            "tie_kind": None, "outcomes": [], "diag": np.full((n + 1, DIAG_COLS), np.nan),
            "gross": np.full(n + 1, np.nan)}


def temperature_ok(T):
    T = float(T)
    return math.isfinite(T) and (T == 0.0 or T >= FLT_MIN)


def verify_stream(rule, q_rows, p_rows, x, T, seed, step, stream):
    """Verify one stream.

    q_rows: N draft logit rows, p_rows: N+1 target logit rows (any float dtype; widened
    exactly to float64), x: N draft tokens, T: temperature (0 = greedy).
    Returns a dict: status, tau, emitted (list), n_emitted, tie, tie_kind, outcomes (a list of
    (tau, tokens) pairs: every result a computation within the near-tie window may give, the
    exact one first), diag [(N+1), 8].
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


def _draw_weights_total_ok(weights):
    total = float(np.sum(weights))
    return total > 0.0 and math.isfinite(total)


def _finish(res, taus, xs, weights_at, u_sample_at):
    """Draw at the decided tau (taus[0]) and at every alternative tau; fill the result."""
    tau = taus[0]
    weights = weights_at(tau)
    if not _draw_weights_total_ok(weights):
        out = _empty_result(len(xs), STATUS_NUMERIC)
        out["diag"] = res["diag"]
        out["gross"] = res["gross"]
        return out
    y, window = inverse_cdf(weights, u_sample_at(tau))
    if len(window) > 1 and not res["tie"]:
        res["tie"], res["tie_kind"] = True, "sample"
    outcomes = [(tau, window)]
    for t in taus[1:]:
        wt = weights_at(t)
        if _draw_weights_total_ok(wt):
            outcomes.append((t, inverse_cdf(wt, u_sample_at(t))[1]))
    res["tau"] = tau
    res["emitted"] = xs[:tau] + [y]
    res["n_emitted"] = tau + 1
    res["outcomes"] = outcomes
    return res


def _tokenwise_tau(passed):
    """tau of the token-wise rule: the first rejected slot, N if none."""
    for i, ok in enumerate(passed):
        if not ok:
            return i
    return len(passed)


def _tokenwise(res, ps, qs, xs, log_rho, seed, step, stream):
    n = len(xs)
    uni = [philox.slot_uniforms(seed, step, stream, i) for i in range(n + 1)]
    acc = [min(1.0, math.exp(log_rho[i])) for i in range(n)]
    passed = [uni[i][0] <= acc[i] for i in range(n)]
    near = [_near(uni[i][0], acc[i]) for i in range(n)]
    tau = _tokenwise_tau(passed)
    # the comparisons that were evaluated: slots 0..tau (all of them when tau = N)
    if any(near[i] for i in range(min(tau + 1, n))):
        res["tie"], res["tie_kind"] = True, "accept"
    taus = _flip_outcomes(passed, near, _tokenwise_tau)

    def weights_at(t):
        if t == n:
            return np.exp(ps[n])
        return residual_weights(1.0, np.exp(ps[t]), np.exp(qs[t]))

    if tau < n:
        res["diag"][tau, D_R] = float(np.sum(weights_at(tau)))
        res["gross"][tau] = residual_gross(1.0, np.exp(ps[tau]), np.exp(qs[tau]))
    return _finish(res, taus, xs, weights_at, lambda t: uni[t][1])


def block_tie_range(tau, n):
    """The slots whose comparison eta_i <= h_i decides tau = max{i : eta_i <= h_i}: tau itself
    and every slot above it (all of 1..N when tau = 0).  A near comparison below tau cannot
    change tau on its own."""
    return range(max(tau, 1), n + 1)


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
        res["gross"][i] = residual_gross(w[i], np.exp(ps[i]), np.exp(qs[i]))
    h = block_h(w, r)
    for i in range(1, n + 1):
        diag[i, D_H] = h[i]
    uni = [philox.slot_uniforms(seed, step, stream, i) for i in range(n + 1)]
    eta = [float("nan")] + [uni[i - 1][0] for i in range(1, n + 1)]
    tau = block_tau(eta, h)
    for i in block_tie_range(tau, n):
        if _near(eta[i], h[i]) and not res["tie"]:
            res["tie"], res["tie_kind"] = True, "block"
    # passed / near indexed by slot - 1 (slots 1..N)
    passed = [eta[i] <= h[i] for i in range(1, n + 1)]
    near = [_near(eta[i], h[i]) for i in range(1, n + 1)]

    def decide(flags):
        t = 0
        for j, ok in enumerate(flags):
            if ok:
                t = j + 1
        return t

    taus = _flip_outcomes(passed, near, decide)

    def weights_at(t):
        if t == n:
            return np.exp(ps[n])
        return residual_weights(w[t], np.exp(ps[t]), np.exp(qs[t]))

    return _finish(res, taus, xs, weights_at, lambda t: uni[t][1])


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
    y = argmax_lowest(pr[tau])
    res["tau"] = tau
    res["emitted"] = xs[:tau] + [y]
    res["n_emitted"] = tau + 1
    res["outcomes"] = [(tau, [y])]
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
    n_emitted, status, diag [cu[B] + B, 8], tie (bool), tie_kind (list) and outcomes (list of
    each stream's admissible (tau, tokens) pairs; empty for a stream that was not verified or
    whose status is not OK), gross [cu[B] + B] (residual_gross of each slot where the residual
    was computed, NaN elsewhere).
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
        "outcomes": [[] for _ in range(B)],
        "gross": np.full(max(cu[-1] + B, 0), np.nan),
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
        out["outcomes"][b] = r["outcomes"]
        if r["status"] == STATUS_OK:
            out["accepted_len"][b] = r["tau"]
            out["n_emitted"][b] = r["n_emitted"]
            out["out_tokens"][b, :len(r["emitted"])] = r["emitted"]
        if float(temps[b]) > 0.0 and r["status"] in (STATUS_OK, STATUS_NUMERIC):
            out["diag"][cu[b] + b: cu[b] + b + n + 1] = r["diag"]
            out["gross"][cu[b] + b: cu[b] + b + n + 1] = r["gross"]
    return out


# ----------------------------------------------------------------------------------------
# Reduced draft vocabulary
# ----------------------------------------------------------------------------------------

class ScatteredRows:
    """Draft rows scored over a reduced draft vocabulary, seen in target-vocabulary columns.

    P1 "MTP, DSpark and Block Verification, Explained", §3 "The Markov fix-up": the drafter
    scores a reduced vocabulary and scatters those logits into target-vocabulary columns, so
    the draft distribution puts no mass outside the reduced vocabulary.  Column v of row r
    holds reduced[r, t2d[v]] when 0 <= t2d[v] < K and -inf otherwise (t2d is the inverse of
    the map from draft ids to target columns).  Row-indexable like a [rows, V] array.
    """

    def __init__(self, reduced, t2d):
        self.reduced = reduced
        self.t2d = np.asarray(t2d, np.int64)
        K = np.asarray(reduced[0]).shape[0] if len(reduced) else 0
        self.K = K
        self.inside = (self.t2d >= 0) & (self.t2d < K)
        ids = self.t2d[self.inside]
        # every draft id is referenced by exactly one column: the scatter is a bijection
        # between a reduced row and its columns
        if len(ids) != K or (K and np.bincount(ids, minlength=K).max() != 1):
            raise ValueError("t2d must reference every draft id in [0, K) exactly once")

    def __len__(self):
        return len(self.reduced)

    def __getitem__(self, r):
        row = np.full(self.t2d.shape[0], -np.inf)
        row[self.inside] = np.asarray(self.reduced[r], np.float64)[self.t2d[self.inside]]
        return row


def verify_batch_reduced(rule, cu_drafts, reduced_draft_logits, t2d, target_logits, draft_tokens,
                         temperature, kmax, seed, step, streams=None):
    """Mirror of spec_verify_tokenwise_reduced / spec_verify_block_reduced: the verify of
    draft rows given over a reduced draft vocabulary (reduced_draft_logits [cu[B], K], column
    map t2d [V]), by definition the dense verify of the scattered rows."""
    return verify_batch(rule, cu_drafts, ScatteredRows(reduced_draft_logits, t2d), target_logits,
                        draft_tokens, temperature, kmax, seed, step, streams)

