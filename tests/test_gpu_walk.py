"""GPU parity of dspark_markov_walk against the oracle's walk, and walk -> verify end to end.

P1 "MTP, DSpark and Block Verification, Explained", §3 "The Markov fix-up" and Figure 2:
slot i is biased by the token sampled at slot i - 1 (slot 0 by the anchor), then t_i is
sampled.  The GPU's tokens must equal the oracle's; at a near-tie draw (the oracle's window
holds more than one token) the GPU's token must be in the window and the later slots, which
then depend on the sampler's choice, are not compared.  Biased rows are compared within the
float32 accumulation bound of the bias, for every slot whose previous token agrees.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from oracle import markov as om  # noqa: E402
from oracle import verify as ov  # noqa: E402
from speculative_decoding_block_verify_gb300 import workloads  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu

EPS32 = 2.0 ** -24
STATUS = {"ok": 0, "bad_temperature": 1, "bad_anchor": 2, "bad_row": 3}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def _bound(row_d, w1, w2, prev):
    R = w2.shape[0]
    mag = np.abs(row_d) + np.abs(w1[prev]) @ np.abs(w2)
    return (R + 2) * EPS32 * mag + 1e-30


def _inputs(name, seed, B, T=None):
    """Per stream: the workload's N draft rows as the drafter's slot logits, an anchor, the
    Markov head's W1, W2; returned as host float arrays and device tensors."""
    inp = workloads.make_verify_inputs(name, seed, B=B)
    bias = workloads.make_bias_inputs(name, seed, rows=B)
    N, V = inp["kmax"], inp["V"]
    d = np.asarray(inp["draft_logits"], np.float32).reshape(B, N, V)
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    temps = np.full(B, 1.0 if T is None else T, np.float32) if T is None or np.isscalar(T) else np.asarray(T, np.float32)
    host = dict(d=d, anchor=bias["prev"][:B].astype(np.int32), w1=bias["W1"], w2=bias["W2"], T=temps)
    dev = dict(d=torch.as_tensor(d).cuda().to(dt), anchor=torch.as_tensor(host["anchor"]).cuda(),
               w1=torch.as_tensor(bias["W1"]).cuda().to(dt), w2=torch.as_tensor(bias["W2"]).cuda().to(dt),
               T=torch.as_tensor(temps).cuda())
    return host, dev


def compare_walk(g, host, b, seed, step, stats):
    """One stream: tokens exact up to the first near tie, biased rows within the bound."""
    r = om.walk(host["d"][b], int(host["anchor"][b]), host["w1"], host["w2"], float(host["T"][b]), seed, step, b)
    assert int(g["status"][b]) == STATUS[r["status"]], (b, g["status"][b], r["status"])
    if r["status"] != "ok":
        return
    prev = int(host["anchor"][b])
    for i, (t, window) in enumerate(zip(r["tokens"], r["windows"])):
        gt = int(g["tokens"][b, i])
        bound = _bound(host["d"][b, i].astype(np.float64), host["w1"], host["w2"], prev)
        err = np.abs(g["logits"][b, i].astype(np.float64) - r["biased"][i])
        assert (err <= bound).all(), (b, i, err.max())
        stats["rows"] += 1
        if len(window) > 1:
            assert gt in window, (b, i, gt, window)
            stats["ties"] += 1
            return
        assert gt == t, (b, i, gt, t)
        stats["tokens"] += 1
        prev = t


@pytest.mark.parametrize("name,steps", [("tiny", 40), ("single_bias", 12)])
def test_walk_matches_the_oracle(name, steps):
    host, dev = _inputs(name, 500, B=1)
    stats = {"rows": 0, "ties": 0, "tokens": 0}
    out = None
    for st in range(steps):
        out = sv.dspark_markov_walk(dev["d"], dev["anchor"], dev["w1"], dev["w2"], dev["T"], 9, st, out=out)
        g = {k: v.cpu().numpy() for k, v in out.items() if k != "workspace"}
        compare_walk(g, host, 0, 9, st, stats)
    assert stats["tokens"] >= 0.7 * steps * host["d"].shape[1], stats


def test_walk_batch_groups_greedy_and_statuses():
    """Six streams (two groups of four): greedy, sampled, a bad anchor, a bad temperature."""
    host, dev = _inputs("tiny", 510, B=6, T=[1.0, 0.0, 0.7, 1.3, 1.0, -1.0])
    host["anchor"][4] = 1024                       # outside [0, V)
    dev["anchor"][4] = 1024
    stats = {"rows": 0, "ties": 0, "tokens": 0}
    out = None
    for st in range(6):
        out = sv.dspark_markov_walk(dev["d"], dev["anchor"], dev["w1"], dev["w2"], dev["T"], 4, st, out=out)
        g = {k: v.cpu().numpy() for k, v in out.items() if k != "workspace"}
        assert list(g["status"]) == [0, 0, 0, 0, 2, 1]
        assert (g["tokens"][4:] == -1).all()
        for b in range(6):
            compare_walk(g, host, b, 4, st, stats)
    assert stats["tokens"] > 0


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_walk_then_verify_is_markov_consistent(rule):
    """The walk's tokens and biased rows feed the verify (the draft distribution q is the one
    the tokens were sampled from); checked against the oracle's walk -> verify."""
    host, dev = _inputs("single_bias", 520, B=1)
    inp = workloads.make_verify_inputs("single_bias", 520)
    dp = torch.as_tensor(np.asarray(inp["target_logits"], np.float32)).cuda().to(torch.bfloat16)
    cu = torch.as_tensor(inp["cu_drafts"]).cuda()
    T = dev["T"]
    fn = sv.spec_verify_block if rule == ov.RULE_BLOCK else sv.spec_verify_tokenwise
    compared = 0
    for st in range(8):
        w = sv.dspark_markov_walk(dev["d"], dev["anchor"], dev["w1"], dev["w2"], T, 2, st)
        r = om.walk(host["d"][0], int(host["anchor"][0]), host["w1"], host["w2"], 1.0, 2, st, 0)
        if any(len(x) > 1 for x in r["windows"]):
            continue                               # a near-tie draft draw: later slots may differ
        assert w["tokens"].cpu().numpy()[0].tolist() == r["tokens"]
        g = parity.to_numpy(fn(cu, w["logits"].view(-1, inp["V"]), dp, w["tokens"].view(-1), T, 5, 2, st))
        o = ov.verify_batch(rule, inp["cu_drafts"], r["biased"], inp["target_logits"], np.array(r["tokens"], np.int32),
                            np.array([1.0], np.float32), 5, 2, st)
        parity.compare_verify(g, o, inp["cu_drafts"], [0], np.array(r["tokens"]), inp["V"], check_diag=False)
        compared += 1
    assert compared >= 5


@pytest.mark.parametrize("name,B", [("single_bias", 1), ("tiny", 9)])
def test_walk_is_reproducible_call_to_call(name, B):
    """Every CTA reduces the same partials and rescans the same drawn slice, with the partials
    alternating between two buffers from slot to slot; the same inputs, seed and step must give
    the same tokens, biased rows and statuses bit for bit, call after call (B = 9: three groups
    of streams, so the buffers also turn over between groups)."""
    host, dev = _inputs(name, 530, B=B, T=None if B == 1 else [1.0, 0.0, 0.7, 1.3, 1.0, 0.5, 1.1, 0.9, 0.0])
    ref = {k: v.clone() for k, v in sv.dspark_markov_walk(dev["d"], dev["anchor"], dev["w1"], dev["w2"], dev["T"],
                                                           3, 7).items() if k != "workspace"}
    out = None
    for _ in range(25):
        out = sv.dspark_markov_walk(dev["d"], dev["anchor"], dev["w1"], dev["w2"], dev["T"], 3, 7, out=out)
        for k, v in ref.items():
            assert torch.equal(out[k].view(torch.int32) if out[k].dtype == torch.float32 else out[k],
                               v.view(torch.int32) if v.dtype == torch.float32 else v), k
