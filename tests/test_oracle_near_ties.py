"""The oracle's near-tie detector, pinned by constructed cases (CPU only).

The GPU computes in float32 and double-float, so where a uniform lies within TIE_REL = 1e-6
(relative) of its threshold the oracle flags the stream and lists every outcome the GPU may
reach there.  These tests build 2-3 token rows whose threshold is placed exactly at, just
inside (0.5e-6) and just outside (2e-6, relative) the stream's own uniform, for each
threshold the rules compare against:

* min(1, rho) of the token-wise rule (P1 "MTP, DSpark and Block Verification, Explained",
  §4 "Token by token");
* h_N = w_N and h_i (i < N) of block verification (§4 "Block verification"), including a
  near comparison below tau, which cannot change tau and must not flag;
* C(Y) and C(Y - 1) of the inverse-CDF draw.

Each case checks the flag, its kind and the admissible outcomes.  Planted mistakes in the
oracle (an absolute instead of a relative margin, a draw window measured against R instead
of U R, a block tie range that includes slots below tau or leaves tau out) must make these
checks fail.
"""

import math

import numpy as np
import pytest

from oracle import philox
from oracle import verify as ov

INSIDE = (0.0, 0.5e-6, -0.5e-6)
OUTSIDE = (2e-6, -2e-6)


def find_stream(pred, seed=0, step=0, limit=20000):
    """The first stream index whose uniforms satisfy pred(list of (u_acc, u_smp) per slot)."""
    for s in range(limit):
        u = [philox.slot_uniforms(seed, step, s, i) for i in range(4)]
        if pred(u):
            return s, u
    raise AssertionError("no stream found")


def logits_for(probs):
    return np.log(np.asarray(probs, np.float64))


# ---------------------------------------------------------------------------------------
# token-wise: u_0 against min(1, rho_0)
# ---------------------------------------------------------------------------------------
def tokenwise_case(delta, u0, stream):
    """N = 1, V = 2, x_0 = 0, q_0 uniform: rho_0 = 2 p_0(0) = u_0 (1 + delta)."""
    q = [np.zeros(2)]
    p0 = u0 * (1.0 + delta) / 2.0
    p = [logits_for([p0, 1.0 - p0]), np.array([0.4, -0.3])]
    return ov.verify_stream(ov.RULE_TOKENWISE, q, p, [0], 1.0, 0, 0, stream)


def accept_pin_failures():
    s, u = find_stream(lambda u: 0.2 < u[0][0] < 0.45)
    bad = []
    for d in INSIDE:
        r = tokenwise_case(d, u[0][0], s)
        if not (r["tie"] and r["tie_kind"] == "accept"):
            bad.append(("inside not flagged", d))
        if {t for t, _ in r["outcomes"]} != {0, 1}:
            bad.append(("outcomes", d, r["outcomes"]))
    for d in OUTSIDE:
        r = tokenwise_case(d, u[0][0], s)
        if r["tie"]:
            bad.append(("outside flagged", d))
        want = 1 if d > 0 else 0   # rho above u accepts, below rejects
        if r["tau"] != want or len(r["outcomes"]) != 1:
            bad.append(("outside outcome", d, r["tau"], r["outcomes"]))
    return bad


def test_tokenwise_accept_threshold_is_pinned():
    assert accept_pin_failures() == []


def test_planted_absolute_margin_is_caught(monkeypatch):
    """Planted mistake: the margin measured in absolute terms, not relative to the threshold."""
    monkeypatch.setattr(ov, "_near", lambda a, b: abs(a - b) <= ov.TIE_REL)
    assert accept_pin_failures() != []


# ---------------------------------------------------------------------------------------
# block: eta_N against h_N = w_N (N = 1)
# ---------------------------------------------------------------------------------------
def block_last_pin_failures():
    s, u = find_stream(lambda u: 0.2 < u[0][0] < 0.45)
    bad = []
    for d in INSIDE + OUTSIDE:
        q = [np.zeros(2)]
        p0 = u[0][0] * (1.0 + d) / 2.0
        p = [logits_for([p0, 1.0 - p0]), np.array([0.4, -0.3])]
        r = ov.verify_stream(ov.RULE_BLOCK, q, p, [0], 1.0, 0, 0, s)
        inside = d in INSIDE
        if inside and not (r["tie"] and r["tie_kind"] == "block"):
            bad.append(("inside not flagged", d))
        if not inside and r["tie"]:
            bad.append(("outside flagged", d))
        want = {0, 1} if inside else {1 if d > 0 else 0}
        if {t for t, _ in r["outcomes"]} != want:
            bad.append(("outcomes", d, r["outcomes"]))
    return bad


def test_block_last_threshold_is_pinned():
    assert block_last_pin_failures() == []


# ---------------------------------------------------------------------------------------
# block: eta_1 against h_1 = r_1 / (r_1 + 1 - w_1) with N = 2
# ---------------------------------------------------------------------------------------
W1 = 0.6
QA = 0.01


def block_mid_case(delta, eta1, stream, x1):
    """Slot 0: q uniform, p(0) = 0.3 so rho_0 = 0.6 = w_1.  Slot 1: q = (QA, 1 - QA),
    p = (pa, 1 - pa) with w_1 pa - QA = r_1 (the other term is clipped at 0), chosen so that
    h_1 = eta_1 (1 + delta).  x_1 = 0 makes w_2 = 1 (tau = 2 for sure); x_1 = 1 makes w_2
    small, so tau is decided by slot 1's comparison."""
    h1 = eta1 * (1.0 + delta)
    r1 = (1.0 - W1) * h1 / (1.0 - h1)
    pa = (r1 + QA) / W1
    q = [np.zeros(2), logits_for([QA, 1.0 - QA])]
    p = [logits_for([W1 / 2.0, 1.0 - W1 / 2.0]), logits_for([pa, 1.0 - pa]), np.array([0.2, 0.1])]
    return ov.verify_stream(ov.RULE_BLOCK, q, p, [0, x1], 1.0, 0, 0, stream)


def block_mid_pin_failures():
    # eta_1 = u_0 in (0.2, 0.35): h_1 reachable below w_1; eta_2 = u_1 above w_2 when x_1 = 1
    s, u = find_stream(lambda u: 0.2 < u[0][0] < 0.35 and u[1][0] > 0.8)
    eta1 = u[0][0]
    bad = []
    for d in INSIDE + OUTSIDE:
        inside = d in INSIDE
        # x_1 = 0: tau = 2 whatever slot 1 does, a near comparison at slot 1 < tau must not flag
        r = block_mid_case(d, eta1, s, 0)
        if r["tau"] != 2 or r["tie_kind"] == "block":
            bad.append(("below tau", d, r["tau"], r["tie_kind"]))
        # x_1 = 1: slot 1 decides tau (1 if eta_1 <= h_1, else 0)
        r = block_mid_case(d, eta1, s, 1)
        if abs(r["diag"][1, ov.D_H] / (eta1 * (1 + d)) - 1.0) > 1e-12:
            bad.append(("construction", d, r["diag"][1, ov.D_H]))
        if inside and not (r["tie"] and r["tie_kind"] == "block"):
            bad.append(("at tau not flagged", d))
        if not inside and r["tie_kind"] == "block":
            bad.append(("outside flagged", d))
        want = {0, 1} if inside else {1 if d > 0 else 0}
        decided = {0, 1} if d == 0.0 else {1 if d > 0 else 0}   # at d = 0 rounding decides
        if {t for t, _ in r["outcomes"]} != want or r["tau"] not in decided:
            bad.append(("outcomes", d, r["tau"], r["outcomes"]))
    return bad


def test_block_mid_threshold_is_pinned():
    assert block_mid_pin_failures() == []


def test_planted_tie_range_with_slots_below_tau_is_caught(monkeypatch):
    monkeypatch.setattr(ov, "block_tie_range", lambda tau, n: range(1, n + 1))
    assert block_mid_pin_failures() != []


def test_planted_tie_range_without_tau_is_caught(monkeypatch):
    monkeypatch.setattr(ov, "block_tie_range", lambda tau, n: range(tau + 1, n + 1))
    assert block_mid_pin_failures() != [] or block_last_pin_failures() != []


# ---------------------------------------------------------------------------------------
# the draw: U R against C(Y) and C(Y - 1)
# ---------------------------------------------------------------------------------------
def draw_case(delta, us, stream, side):
    """N = 0 (the bonus draw from p_0), V = 3.  side 'hi': C(0) = U (1 + delta), so Y = 0 is
    decided by C(Y); side 'lo': C(0) = U (1 - delta), so Y = 1 is decided by C(Y - 1)."""
    c0 = us * (1.0 + delta) if side == "hi" else us * (1.0 - delta)
    rest = (1.0 - c0) / 2.0
    p = [logits_for([c0, rest, rest])]
    return ov.verify_stream(ov.RULE_BLOCK, [], p, [], 1.0, 0, 0, stream)


def draw_pin_failures():
    # the bonus draw at slot 0 uses word 1 of slot 0; U well below 1/2 so that a window
    # measured against R = 1 instead of U R would be more than twice as wide
    s, u = find_stream(lambda u: 0.15 < u[0][1] < 0.35)
    us = u[0][1]
    bad = []
    for side in ("hi", "lo"):
        for d in INSIDE + OUTSIDE:
            r = draw_case(d, us, s, side)
            inside = d in INSIDE
            if inside and not (r["tie"] and r["tie_kind"] == "sample"):
                bad.append((side, "inside not flagged", d))
            if not inside and r["tie"]:
                bad.append((side, "outside flagged", d))
            toks = r["outcomes"][0][1] if r["outcomes"] else None
            want = [0, 1] if inside else [r["emitted"][-1]]
            if toks != want:
                bad.append((side, "window", d, toks))
    return bad


def test_draw_thresholds_are_pinned():
    assert draw_pin_failures() == []


def test_planted_window_relative_to_total_is_caught(monkeypatch):
    monkeypatch.setattr(ov, "window_bounds",
                        lambda t, total: (t - ov.TIE_REL * total, t + ov.TIE_REL * total))
    assert draw_pin_failures() != []


def test_window_skips_zero_weight_tokens():
    """A zero-weight token next to the boundary is never admissible (U > 0 never selects it)."""
    w = np.array([0.3, 0.0, 0.0, 0.7])
    y, window = ov.inverse_cdf(w, 0.3 / 1.0)
    assert y == 0 and window == [0, 3]
    y, window = ov.inverse_cdf(w, 0.5)
    assert y == 3 and window == [3]


def test_tokenwise_flip_below_tau_reaches_later_slots():
    """A near comparison at slot 0 of a stream rejected at slot 1: flipping it alone leaves
    tau = 1 only if slot 0 was accepted; the listed outcomes follow the flip through."""
    s, u = find_stream(lambda u: 0.2 < u[0][0] < 0.45 and u[1][0] > 0.9)
    p0 = u[0][0] / 2.0          # rho_0 = u_0 exactly: near
    q = [np.zeros(2), np.zeros(2)]
    p = [logits_for([p0, 1.0 - p0]), logits_for([0.05, 0.95]), np.array([0.0, 0.0])]
    r = ov.verify_stream(ov.RULE_TOKENWISE, q, p, [0, 0], 1.0, 0, 0, s)
    # slot 1: rho_1 = 0.1 < u_1, rejected whatever happens at slot 0
    assert r["tie_kind"] == "accept"
    assert {t for t, _ in r["outcomes"]} == {0, 1}
    assert math.isclose(r["diag"][1, ov.D_RHO], 0.1, rel_tol=1e-12)
