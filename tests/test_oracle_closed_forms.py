"""Closed-form and special-case pins of the oracle's verify rules (CPU only)."""

import numpy as np
import pytest

from oracle import verify
from speculative_decoding_block_verify_gb300 import workloads

RULES = (verify.RULE_TOKENWISE, verify.RULE_BLOCK)


@pytest.mark.parametrize("rule", RULES)
def test_identical_draft_and_target_accepts_everything(rule):
    """p = q: rho = 1 at every slot, so both rules accept all N drafts (tau = N)."""
    rng = np.random.default_rng(0)
    N, V = 5, 300
    tgt = (rng.standard_normal((N + 1, V)) * 2).astype(np.float32)
    x = rng.integers(0, V, N)
    for step in range(50):
        r = verify.verify_stream(rule, tgt[:N], tgt, x, 0.8, seed=1, step=step, stream=0)
        assert r["status"] == 0 and r["tau"] == N and r["emitted"][:N] == list(x)
        if rule == verify.RULE_BLOCK:
            assert np.allclose(r["diag"][:, verify.D_W], 1.0)


@pytest.mark.parametrize("rule", RULES)
def test_disjoint_supports_reject_at_first_slot(rule):
    """supp(q) and supp(p) disjoint: rho_0 = 0, so w_1 = 0 and h = 0 (block), and the first
    token-wise test fails; the draw is then from max(0, p_0 - q_0) = p_0."""
    rng = np.random.default_rng(1)
    N, V = 3, 40
    half = V // 2
    q = np.full((N, V), -np.inf)
    q[:, :half] = rng.standard_normal((N, half))
    p = np.full((N + 1, V), -np.inf)
    p[:, half:] = rng.standard_normal((N + 1, V - half))
    x = rng.integers(0, half, N)
    counts = np.zeros(V)
    M = 3000
    for step in range(M):
        r = verify.verify_stream(rule, q, p, x, 1.0, seed=2, step=step, stream=1)
        assert r["status"] == 0 and r["tau"] == 0
        counts[r["emitted"][0]] += 1
    assert counts[:half].sum() == 0
    p0 = np.exp(p[0, half:] - np.logaddexp.reduce(p[0, half:]))
    chi = ((counts[half:] - M * p0) ** 2 / (M * p0)).sum()
    assert chi < 60          # 19 dof; p ~ 1e-6 at 60


def test_small_temperature_reduces_to_greedy():
    """T -> 0: p and q become one-hot, both rules reproduce the greedy branch (this also
    exercises the 0/0 reading h = 1 when p_i = q_i exactly)."""
    rng = np.random.default_rng(2)
    N, V = 5, 200
    for trial in range(20):
        tgt = rng.standard_normal((N + 1, V))
        drf = tgt[:N] + rng.standard_normal((N, V)) * (0.05 if trial % 2 else 1.0)
        x = np.argmax(drf, axis=1)
        g = verify.verify_stream(0, drf, tgt, x, 0.0, seed=0, step=trial, stream=0)
        for rule in RULES:
            r = verify.verify_stream(rule, drf, tgt, x, 1e-4, seed=0, step=trial, stream=0)
            assert (r["tau"], r["emitted"]) == (g["tau"], g["emitted"])


def test_greedy_ignores_draft_rows_and_the_rule():
    tgt = np.array([[0.0, 5.0, 1.0], [2.0, 2.0, 0.0], [1.0, 0.0, 3.0]])
    drf = np.full((2, 3), np.nan)            # never read at T = 0
    for rule in RULES:
        r = verify.verify_stream(rule, drf, tgt, [1, 0], 0.0, seed=0, step=0, stream=0)
        assert r["status"] == 0 and r["tau"] == 2 and r["emitted"] == [1, 0, 2]
        r = verify.verify_stream(rule, drf, tgt, [1, 1], 0.0, seed=0, step=0, stream=0)
        assert r["tau"] == 1 and r["emitted"] == [1, 0]     # tie 2.0/2.0 -> lowest index


def test_zero_drafts_emits_the_bonus_token():
    tgt = np.log(np.array([[0.1, 0.2, 0.7]]))
    for rule in RULES:
        r = verify.verify_stream(rule, np.zeros((0, 3)), tgt, [], 1.0, seed=3, step=0, stream=0)
        assert r["status"] == 0 and r["tau"] == 0 and r["n_emitted"] == 1


def test_status_precedence():
    V = 4
    good = np.zeros((3, V))
    nan_row = good.copy()
    nan_row[1, 2] = np.nan
    qzero = good[:2].copy()
    qzero[1, 3] = -np.inf
    cases = [
        (good[:2], good, [0, 1], -1.0, verify.STATUS_BAD_TEMPERATURE),
        (good[:2], good, [0, 1], float("nan"), verify.STATUS_BAD_TEMPERATURE),
        (good[:2], good, [0, 1], 1e-40, verify.STATUS_BAD_TEMPERATURE),
        (good[:2], good, [0, 4], 1.0, verify.STATUS_BAD_TOKEN),
        (good[:2], good, [-1, 0], 0.0, verify.STATUS_BAD_TOKEN),
        (good[:2], nan_row, [0, 1], 1.0, verify.STATUS_BAD_ROW),
        (good[:2], nan_row, [0, 1], 0.0, verify.STATUS_BAD_ROW),
        (np.full((2, V), -np.inf), good, [0, 1], 1.0, verify.STATUS_BAD_ROW),
        (qzero, good, [0, 3], 1.0, verify.STATUS_ZERO_DRAFT_PROB),
        (qzero, nan_row, [0, 3], 1.0, verify.STATUS_BAD_ROW),
        (qzero, good, [0, 3], 0.0, verify.STATUS_OK),       # greedy does not read q
    ]
    for q, p, x, T, want in cases:
        for rule in RULES:
            r = verify.verify_stream(rule, q, p, x, T, seed=0, step=0, stream=0)
            assert r["status"] == want, (x, T, want, r["status"])
            if want:
                assert r["n_emitted"] == 0 and r["emitted"] == []


def test_batch_layout_and_offsets():
    inp = workloads.make_verify_inputs("tiny", 5, B=3, V=64, k=[2, 0, 3])
    cu = inp["cu_drafts"]
    assert list(cu) == [0, 2, 2, 5]
    assert inp["target_logits"].shape == (8, 64) and inp["draft_logits"].shape == (5, 64)
    out = verify.verify_batch(verify.RULE_BLOCK, cu, inp["draft_logits"], inp["target_logits"],
                              inp["draft_tokens"], inp["temperature"], kmax=5, seed=4, step=9)
    for b in range(3):
        n = cu[b + 1] - cu[b]
        ref = verify.verify_stream(verify.RULE_BLOCK, inp["draft_logits"][cu[b]:cu[b] + n],
                                   inp["target_logits"][cu[b] + b:cu[b] + b + n + 1],
                                   inp["draft_tokens"][cu[b]:cu[b] + n],
                                   inp["temperature"][b], 4, 9, b)
        assert out["accepted_len"][b] == ref["tau"]
        assert list(out["out_tokens"][b, :ref["n_emitted"]]) == ref["emitted"]
        assert (out["out_tokens"][b, ref["n_emitted"]:] == -1).all()
    bad = verify.verify_batch(0, np.array([0, 3, 2]), inp["draft_logits"],
                              inp["target_logits"], inp["draft_tokens"],
                              inp["temperature"][:2], kmax=2, seed=0, step=0)
    assert list(bad["status"]) == [verify.STATUS_BAD_OFFSETS, verify.STATUS_BAD_OFFSETS]
    # a valid-looking stream after a broken one, and a batch that does not start at row 0
    B5 = verify.STATUS_BAD_OFFSETS
    for cu_bad, want in (([0, 2, 1, 6], [0, B5, B5]), ([0, 1, 5, 6], [0, B5, B5]),
                         ([0, 5, 1, 2], [B5, B5, B5]), ([1, 2, 3, 4], [B5, B5, B5])):
        r = verify.verify_batch(0, np.array(cu_bad), np.zeros((8, 4)), np.zeros((12, 4)),
                                np.zeros(8, np.int32), np.ones(3, np.float32), kmax=2, seed=0,
                                step=0)
        assert list(r["status"]) == want, cu_bad


def test_tokenwise_acceptance_rate_is_one_minus_tv():
    """At scale the per-slot token-wise acceptance rate is sum_v min(p, q) = 1 - TV(p, q)
    (the draft token being drawn from q)."""
    rng = np.random.default_rng(5)
    V = 50
    p = np.log(rng.dirichlet(np.ones(V)))
    q = np.log(rng.dirichlet(np.ones(V)))
    pe, qe = np.exp(p), np.exp(q)
    want = np.minimum(pe, qe).sum()
    acc, M = 0, 4000
    for step in range(M):
        x = [int(rng.choice(V, p=qe))]
        r = verify.verify_stream(0, [q], [p, p], x, 1.0, seed=6, step=step, stream=0)
        acc += r["tau"] == 1
    assert abs(acc / M - want) < 4 * np.sqrt(want * (1 - want) / M)


def test_residual_gross_bounds_the_residual():
    """residual_gross is the positive part's w p mass: >= the residual, equal when q = 0 on
    that part, and 0 when w p <= q everywhere."""
    from oracle import verify as v
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.1, 0.6, 0.3])
    g = v.residual_gross(1.0, p, q)
    assert g == 0.5 and float(v.residual_weights(1.0, p, q).sum()) == pytest.approx(0.4)
    assert v.residual_gross(1.0, p, np.array([0.0, 1.0, 1.0])) == 0.5
    assert v.residual_gross(0.1, p, q) == 0.0
