"""Statistical checks of the GPU verify path over many draws (not only token parity).

* Token-wise acceptance at slot 0 with the draft token drawn from q afresh for every stream
  and step: the accept rate must equal sum_v min(p(v), q(v)) = 1 - TV(p, q) (P1 "MTP, DSpark
  and Block Verification, Explained", §4 "Token by token") within 4 standard errors.
* With a fixed draft, the first emitted token of the token-wise rule has the exact law
  P(x_0) = min(1, rho_0), P(v) = (1 - min(1, rho_0)) max(0, p_0(v) - q_0(v)) / r_0, and block
  verification with N = 2 (§4 "Block verification") has P(tau = 2) = h_2,
  P(tau = 1) = h_1 (1 - h_2), P(tau = 0) = (1 - h_1)(1 - h_2), with the token at tau drawn
  from the normalised residual max(0, w_tau p_tau - q_tau).  Chi-square tests at V = 64 over
  ~20,000 draws compare the GPU's frequencies with these laws, computed by the float64
  oracle.
"""

import numpy as np
import pytest
from scipy import stats

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from oracle import softmax as osm  # noqa: E402
from oracle import verify as ov  # noqa: E402

pytestmark = pytest.mark.gpu

V = 64
B = 1024


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def _rows(seed, n):
    rng = np.random.default_rng(seed)
    target = (rng.standard_normal((n + 1, V)) * 1.5).astype(np.float32)
    draft = (target[:n] + rng.standard_normal((n, V)) * 1.0).astype(np.float32)
    return draft, target


def _batch(draft, target, x):
    """B identical streams with N = len(draft) drafts each; x [B, N] draft tokens."""
    n = draft.shape[0]
    cu = torch.arange(0, B * n + 1, n, dtype=torch.int32, device="cuda")
    dq = torch.as_tensor(np.tile(draft, (B, 1)), device="cuda")
    dp = torch.as_tensor(np.tile(target, (B, 1)), device="cuda")
    xt = torch.as_tensor(np.asarray(x, np.int32).reshape(-1), device="cuda")
    T = torch.ones(B, dtype=torch.float32, device="cuda")
    return cu, dq, dp, xt, T


def _chi2(counts, probs):
    """Chi-square p-value, categories with expected count < 5 merged into one."""
    counts = np.asarray(counts, np.float64)
    exp = np.asarray(probs, np.float64) * counts.sum()
    big = exp >= 5
    c = np.append(counts[big], counts[~big].sum())
    e = np.append(exp[big], exp[~big].sum())
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    assert counts[exp == 0].sum() == 0, "a token with zero probability was emitted"
    return stats.chisquare(c, e).pvalue


def test_tokenwise_acceptance_rate_is_one_minus_tv():
    draft, target = _rows(1, 1)
    p = osm.probs(target[0], 1.0)
    q = osm.probs(draft[0], 1.0)
    expect = float(np.minimum(p, q).sum())
    rng = np.random.default_rng(2)
    acc = n = 0
    out = None
    for step in range(12):
        x = rng.choice(V, size=(B, 1), p=q / q.sum())
        cu, dq, dp, xt, T = _batch(draft, target, x)
        out = sv.spec_verify_tokenwise(cu, dq, dp, xt, T, 1, 7, step, out=out)
        st = out["status"].cpu().numpy()
        assert (st == 0).all()
        acc += int(out["accepted_len"].cpu().numpy().sum())
        n += B
    rate = acc / n
    se = np.sqrt(expect * (1 - expect) / n)
    assert n >= 10_000
    assert abs(rate - expect) <= 4 * se, (rate, expect, se)


def test_tokenwise_first_token_law():
    draft, target = _rows(3, 1)
    p = osm.probs(target[0], 1.0)
    q = osm.probs(draft[0], 1.0)
    x0 = int(np.argmax(q - p))            # a draft token the target under-weights
    a = min(1.0, p[x0] / q[x0])
    resid = ov.residual_weights(1.0, p, q)
    law = (1.0 - a) * resid / resid.sum()
    law[x0] += a
    cu, dq, dp, xt, T = _batch(draft, target, np.full((B, 1), x0))
    counts = np.zeros(V)
    out = None
    for step in range(20):
        out = sv.spec_verify_tokenwise(cu, dq, dp, xt, T, 1, 11, step, out=out)
        tok = out["out_tokens"][:, 0].cpu().numpy()
        counts += np.bincount(tok, minlength=V)
    assert _chi2(counts, law) > 1e-4


def test_block_tau_and_token_law():
    draft, target = _rows(7, 2)
    p = [osm.probs(target[i], 1.0) for i in range(3)]
    q = [osm.probs(draft[i], 1.0) for i in range(2)]
    x = [int(np.argmax(q[0] * p[0])), int(np.argmax(q[1]))]
    log_rho = [np.log(p[i][x[i]] / q[i][x[i]]) for i in range(2)]
    w = ov.running_weights(log_rho)
    r = [float(ov.residual_weights(w[i], p[i], q[i]).sum()) for i in range(2)]
    h = ov.block_h(w, r)
    p_tau = np.array([(1 - h[1]) * (1 - h[2]), h[1] * (1 - h[2]), h[2]])
    assert p_tau.min() > 0.02, p_tau   # every tau is exercised
    cu, dq, dp, xt, T = _batch(draft, target, np.tile(x, (B, 1)))
    tau_counts = np.zeros(3)
    tok_counts = [np.zeros(V) for _ in range(3)]
    out = None
    for step in range(20):
        out = sv.spec_verify_block(cu, dq, dp, xt, T, 2, 13, step, out=out)
        assert (out["status"].cpu().numpy() == 0).all()
        tau = out["accepted_len"].cpu().numpy()
        toks = out["out_tokens"].cpu().numpy()
        tau_counts += np.bincount(tau, minlength=3)
        for t in range(3):
            sel = tau == t
            tok_counts[t] += np.bincount(toks[sel, t], minlength=V)
    assert _chi2(tau_counts, p_tau) > 1e-4
    for t in range(3):
        law = p[2] if t == 2 else ov.residual_weights(w[t], p[t], q[t])
        assert _chi2(tok_counts[t], law / law.sum()) > 1e-4, t
