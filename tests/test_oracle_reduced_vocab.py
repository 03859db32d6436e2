"""The oracle's reduced-draft-vocabulary verify pinned on the CPU.

P1 "MTP, DSpark and Block Verification, Explained", §3 "The Markov fix-up": the drafter scores
a reduced vocabulary and scatters those logits into target-vocabulary columns, so q puts no
mass outside it.

* Identity map (K = V, t2d = identity): the same results as the dense oracle, bit for bit.
* Permuted map (K = V, t2d a permutation): the reduced rows are the dense rows gathered at
  d2t; the results equal the dense oracle's on the dense rows.  A transposed map (the
  permutation used the other way round) changes them.
* Residual closed form: r_i = w_i (1 - sum_{v in S} p_i(v)) + sum_{j < K} max(0, w_i p_i(d2t[j])
  - q_i(j)), written out here from the logits; mass outside the draft vocabulary enters with
  weight w_i.
* A draft token outside the draft vocabulary: ZERO_DRAFT_PROB.
* Losslessness (token-wise, one slot): the emitted token follows p over many Philox steps.
* Invalid maps are refused.
"""

import numpy as np
import pytest
from scipy import stats

from oracle import verify as ov
from speculative_decoding_block_verify_gb300 import workloads

KEYS = ("accepted_len", "out_tokens", "n_emitted", "status")


def _same(a, b):
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k
    assert np.allclose(a["diag"], b["diag"], equal_nan=True, rtol=0, atol=0)


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_identity_map_equals_the_dense_oracle(rule):
    d = workloads.make_verify_inputs("batch64", 71, B=6, V=256)
    t2d = np.arange(256, dtype=np.int32)
    r = ov.verify_batch_reduced(rule, d["cu_drafts"], d["draft_logits"], t2d, d["target_logits"],
                                d["draft_tokens"], d["temperature"], 5, 3, 9)
    o = ov.verify_batch(rule, d["cu_drafts"], d["draft_logits"], d["target_logits"], d["draft_tokens"],
                        d["temperature"], 5, 3, 9)
    _same(r, o)


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_permuted_map_gathers_the_dense_rows(rule):
    d = workloads.make_verify_inputs("batch64", 72, B=6, V=256)
    rng = np.random.default_rng(5)
    d2t = rng.permutation(256).astype(np.int32)
    t2d = np.empty(256, np.int32)
    t2d[d2t] = np.arange(256, dtype=np.int32)
    reduced = d["draft_logits"][:, d2t]           # draft id j holds the logit of column d2t[j]
    r = ov.verify_batch_reduced(rule, d["cu_drafts"], reduced, t2d, d["target_logits"], d["draft_tokens"],
                                d["temperature"], 5, 3, 9)
    o = ov.verify_batch(rule, d["cu_drafts"], d["draft_logits"], d["target_logits"], d["draft_tokens"],
                        d["temperature"], 5, 3, 9)
    _same(r, o)
    # the map used the other way round is a different draft distribution
    wrong = ov.verify_batch_reduced(rule, d["cu_drafts"], reduced, d2t, d["target_logits"], d["draft_tokens"],
                                    d["temperature"], 5, 3, 9)
    assert not np.allclose(wrong["diag"][:, ov.D_QX], o["diag"][:, ov.D_QX], equal_nan=True)


def _softmax(l, T):
    z = np.asarray(l, np.float64) / T
    z = z - z[np.isfinite(z)].max()
    e = np.exp(z)
    return e / e.sum()


def test_block_residual_closed_form_with_mass_outside_the_vocabulary():
    d = workloads.make_verify_inputs("batch64_topk", 73, B=8, V=512, K=96)
    t2d, d2t = d["t2d"], d["d2t"]
    r = ov.verify_batch_reduced(ov.RULE_BLOCK, d["cu_drafts"], d["draft_logits"], t2d, d["target_logits"],
                                d["draft_tokens"], d["temperature"], 5, 0, 4)
    cu = d["cu_drafts"]
    checked = 0
    for b in range(8):
        T = float(d["temperature"][b])
        if T == 0.0 or r["status"][b] != ov.STATUS_OK:
            continue
        for i in range(cu[b + 1] - cu[b]):
            row = cu[b] + b + i
            got = r["diag"][row, ov.D_R]
            if not np.isfinite(got):
                continue                          # no residual was needed at this slot
            w = r["diag"][row, ov.D_W]
            p = _softmax(d["target_logits"][row], T)
            q = _softmax(d["draft_logits"][cu[b] + i], T)
            want = w * (1.0 - p[d2t].sum()) + np.maximum(0.0, w * p[d2t] - q).sum()
            assert abs(got - want) <= 1e-12 * max(1.0, want), (b, i, got, want)
            checked += 1
    assert checked >= 3


def test_draft_token_outside_the_vocabulary_is_zero_draft_prob():
    d = workloads.make_verify_inputs("batch64_topk", 74, B=4, V=512, K=96)
    T = np.full(4, 0.8, np.float32)
    x = d["draft_tokens"].copy()
    outside = int(np.flatnonzero(d["t2d"] < 0)[0])
    x[d["cu_drafts"][2] + 1] = outside
    r = ov.verify_batch_reduced(ov.RULE_BLOCK, d["cu_drafts"], d["draft_logits"], d["t2d"], d["target_logits"],
                                x, T, 5, 0, 0)
    assert r["status"][2] == ov.STATUS_ZERO_DRAFT_PROB
    assert r["status"][1] == ov.STATUS_OK and r["n_emitted"][2] == 0


def test_tokenwise_one_slot_is_lossless_over_the_reduced_vocabulary():
    """One stream, one draft slot: the emitted token after the draft is accepted or replaced
    follows p_0 (V = 8, a draft vocabulary of 3 columns)."""
    V, K = 8, 3
    rng = np.random.default_rng(9)
    p_logits = rng.standard_normal((2, V)) * 1.2
    d2t = np.array([1, 4, 6], np.int32)
    t2d = np.full(V, -1, np.int32)
    t2d[d2t] = np.arange(K, dtype=np.int32)
    q_red = rng.standard_normal((1, K)) * 1.2
    q = _softmax(q_red[0], 1.0)
    counts = np.zeros(V)
    steps = 6000
    for st in range(steps):
        j = int(np.searchsorted(np.cumsum(q), rng.random()))   # x ~ q over the draft vocabulary
        r = ov.verify_batch_reduced(ov.RULE_TOKENWISE, [0, 1], q_red, t2d, p_logits, [d2t[min(j, K - 1)]],
                                    [1.0], 1, 7, st)
        counts[r["out_tokens"][0, 0]] += 1
    p = _softmax(p_logits[0], 1.0)
    assert stats.chisquare(counts, p * steps).pvalue > 1e-4


def test_invalid_maps_are_refused():
    red = np.zeros((1, 3))
    with pytest.raises(ValueError):
        ov.ScatteredRows(red, np.array([0, 1, -1, -1]))          # draft id 2 never referenced
    with pytest.raises(ValueError):
        ov.ScatteredRows(red, np.array([0, 1, 2, 2]))            # draft id 2 referenced twice
