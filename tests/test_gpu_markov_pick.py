"""GPU parity of dspark_markov_bias and adaptive_pick_k against the float64 oracle, and the
end-to-end Markov-bias -> verify pipeline."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from oracle import confidence as oc  # noqa: E402
from oracle import markov as om  # noqa: E402
from oracle import verify as ov  # noqa: E402
from speculative_decoding_block_verify_gb300 import workloads  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu

EPS32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def _t(a, dtype):
    return torch.as_tensor(np.asarray(a, np.float32)).cuda().to(dtype)


def bias_bound(d, w1, w2, prev):
    """Float32 accumulation bound of draft + sum_j W1 W2 (R + 2 roundings of the magnitudes)."""
    R = w2.shape[0]
    mag = np.abs(np.asarray(d, np.float64)) + np.abs(np.asarray(w1, np.float64)[prev]) @ np.abs(
        np.asarray(w2, np.float64))
    return (R + 2) * EPS32 * mag + 1e-30


@pytest.mark.parametrize("case", [("tiny", None, None, None), ("single_bias", None, None, None),
                                  ("tiny", 20, 1001, 24), ("single_bias", 9, 4096, 256),
                                  ("single_bias", 13, 4104, 100), ("tiny", 7, 2056, 3),
                                  ("single_bias", 2, 8200, 40), ("single_bias", 3, 8192, 64)])
def test_markov_bias_parity(case):
    name, rows, V, R = case
    inp = workloads.make_verify_inputs(name, 101, V=V)
    bias = workloads.make_bias_inputs(name, 101, rows=rows, V=V, rank=R)
    rows = len(bias["prev"])
    d = np.resize(inp["draft_logits"], (rows, bias["V"])) if rows != len(inp["draft_logits"]) else inp["draft_logits"]
    dt = torch.bfloat16 if bias["dtype"] == "bf16" else torch.float32
    out = sv.dspark_markov_bias(_t(d, dt), torch.as_tensor(bias["prev"]).cuda(), _t(bias["W1"], dt),
                                _t(bias["W2"], dt)).cpu().numpy()
    ref = om.markov_bias(d, bias["prev"], bias["W1"], bias["W2"])
    bound = bias_bound(d, bias["W1"], bias["W2"], bias["prev"])
    assert (np.abs(out - ref) <= bound).all()


def test_markov_bias_invalid_prev_and_in_place():
    bias = workloads.make_bias_inputs("tiny", 7, rows=4, V=512, rank=16)
    d = np.random.default_rng(0).standard_normal((4, 512)).astype(np.float32)
    prev = bias["prev"].copy()
    prev[1], prev[3] = -1, 512
    dt = torch.float32
    dd = _t(d, dt)
    out = sv.dspark_markov_bias(dd, torch.as_tensor(prev).cuda(), _t(bias["W1"], dt),
                                _t(bias["W2"], dt), out=dd).cpu().numpy()   # in place
    ref = om.markov_bias(d, prev, bias["W1"], bias["W2"])
    assert np.isnan(out[1]).all() and np.isnan(out[3]).all()
    ok = [0, 2]
    assert (np.abs(out[ok] - ref[ok]) <= bias_bound(d, bias["W1"], bias["W2"], np.where(prev < 0, 0, prev) % 512)[ok]).all()


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
@pytest.mark.parametrize("name,n_steps,stride", [("tiny", 300, 1), ("single_bias", 10000, 10)])
def test_bias_then_verify_end_to_end(rule, name, n_steps, stride):
    """Markov bias -> verify on the GPU against float64 bias -> verify in the oracle.  The GPU
    runs every step; the oracle checks every stride-th step (for the single-stream V = 129,280
    workload: the 1,000-step subset 0, 10, 20, ... of 10,000 steps, on the host cores)."""
    inp = workloads.make_verify_inputs(name, 2000)
    bias = workloads.make_bias_inputs(name, 2000)
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    d = parity.verify_to_device(inp, torch)
    biased = sv.dspark_markov_bias(d["dq"], torch.as_tensor(bias["prev"]).cuda(),
                                   _t(bias["W1"], dt), _t(bias["W2"], dt))
    ref_q = om.markov_bias(inp["draft_logits"], bias["prev"], bias["W1"], bias["W2"])
    fn = sv.spec_verify_block if rule == ov.RULE_BLOCK else sv.spec_verify_tokenwise
    taus = []
    gpu = {}
    for step in range(n_steps):
        g = fn(d["cu"], biased, d["dp"], d["x"], d["T"], inp["kmax"], 0, step, diag=(step % stride == 0))
        if step % stride == 0:
            gpu[step] = parity.to_numpy(g)
            taus.append(int(gpu[step]["accepted_len"][0]))
        else:
            taus.append(g["accepted_len"][0])
    taus = [int(t) for t in taus]
    runs = [(rule, 0, st) for st in range(0, n_steps, stride)]
    host = {"cu": inp["cu_drafts"], "dq": ref_q, "dp": np.asarray(inp["target_logits"], np.float64),
            "x": inp["draft_tokens"], "T": inp["temperature"]}
    ref = parity.oracle_runs(host, inp["kmax"], runs, [0], torch, runs_per_task=max(1, len(runs) // 16))
    totals = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0}
    for run in runs:
        # the biased rows differ from the oracle's float64 ones by the float32 bias rounding, so
        # the diag columns are compared by test_markov_bias_parity's bound, not here
        st = parity.compare_verify(gpu[run[2]], ref[run], inp["cu_drafts"], [0], inp["draft_tokens"],
                                   inp["V"], check_diag=False)
        for k in totals:
            totals[k] += st[k]
    assert totals["exact"] + totals["ties"] == len(runs)
    parity.check_tie_totals(totals)
    assert len(taus) == n_steps and min(taus) >= 0 and max(taus) <= 5


def _pick_inputs(seed, B=128, kmax=5, H=7168):
    c = workloads.make_confidence_inputs(seed, B=B, kmax=kmax, H=H)
    return c, _t(c["hidden"], torch.bfloat16), _t(c["w"], torch.bfloat16), torch.as_tensor(c["verify_ms"]).cuda()


def per_stream_tie(a_row, table, kmax, rel=1e-6):
    vals = sorted((oc.expected_tokens(a_row, n) / float(table[n + 1]) for n in range(kmax + 1)),
                  reverse=True)
    return vals[0] - vals[1] <= rel * vals[0]


def batch_tie(a, table, rel=1e-6):
    """Near tie in the batch pick: two a values within rel of each other, or two ratios."""
    B, kmax = a.shape
    flat = np.sort(a.reshape(-1))[::-1]
    if np.any(np.abs(np.diff(flat)) <= rel * flat[1:]):
        return True
    s = np.concatenate([[0.0], np.cumsum(flat)])
    ratios = np.sort((B + s) / table[B:B + len(s)].astype(np.float64))[::-1]
    return ratios[0] - ratios[1] <= rel * ratios[0]


@pytest.mark.parametrize("mode", [0, 1])
def test_pick_k_parity(mode):
    c, h, w, vm = _pick_inputs(5)
    g = sv.adaptive_pick_k(h, w, c["beta"], vm, mode=mode)
    g = {k: v.cpu().numpy() for k, v in g.items()}
    cc = oc.confidence(c["hidden"], c["w"], c["beta"])
    a = oc.prefix_survival(cc)
    assert np.allclose(g["c"], cc, rtol=1e-5, atol=0) and np.allclose(g["a"], a, rtol=1e-5, atol=1e-30)
    if mode == 0:
        k, _ = oc.pick_k_per_stream(a, c["verify_ms"])
        for b in range(len(k)):
            if not per_stream_tie(a[b], c["verify_ms"], 5):
                assert g["k"][b] == k[b], b
    else:
        k, m, v = oc.pick_k_batch(a, c["verify_ms"])
        B = len(k)
        e = sum(oc.expected_tokens(a[b], g["k"][b]) for b in range(B)) / float(c["verify_ms"][B + g["k"].sum()])
        assert abs(e - v) <= 1e-6 * v
        if not batch_tie(a, c["verify_ms"]):
            assert np.array_equal(g["k"], k)
    assert np.array_equal(g["cu"], oc.cu_from_k(g["k"]))


def test_pick_k_worked_example():
    """c = (.95, .90, .85, .40) with verify_ms[n] = 12 + 2.6 n -> verify 3 drafts."""
    cvals = np.array([0.95, 0.90, 0.85, 0.40])
    logits = np.log(cvals / (1 - cvals))
    H = 8
    hidden = np.zeros((1, 4, H), np.float32)
    hidden[0, :, 0] = logits
    w = np.zeros(H, np.float32)
    w[0] = 1.0
    vm = torch.as_tensor((12.0 + 2.6 * np.arange(40)).astype(np.float32)).cuda()
    g = sv.adaptive_pick_k(torch.as_tensor(hidden).cuda(), torch.as_tensor(w).cuda(), 0.0, vm)
    assert int(g["k"][0]) == 3
    assert np.allclose(g["a"].cpu().numpy()[0], [0.95, 0.855, 0.72675, 0.2907], rtol=1e-6)


def test_pick_k_batch_small_brute_force():
    rng = np.random.default_rng(9)
    for trial in range(10):
        B, kmax, H = int(rng.integers(1, 4)), int(rng.integers(1, 4)), 64
        hidden = workloads.round_bf16(rng.standard_normal((B, kmax, H)).astype(np.float32))
        w = workloads.round_bf16((rng.standard_normal(H) * 0.3).astype(np.float32))
        table = (rng.uniform(0.5, 5) + rng.uniform(0.1, 2) * np.arange(B * (kmax + 1) + 1)).astype(np.float32)
        g = sv.adaptive_pick_k(_t(hidden, torch.bfloat16), _t(w, torch.bfloat16), 0.1,
                               torch.as_tensor(table).cuda(), mode=1)
        a = oc.prefix_survival(oc.confidence(hidden, w, 0.1))
        k, m, v = oc.pick_k_batch(a, table)
        gk = g["k"].cpu().numpy()
        e = sum(oc.expected_tokens(a[b], gk[b]) for b in range(B)) / table[B + gk.sum()]
        assert abs(e - v) <= 1e-6 * v


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_adaptive_then_ragged_verify(rule):
    """Per-stream pick over B = 128 (H = 7168), then the ragged verify over V = 129,280 with
    the oracle's k (streams with k = 0 included), every stream checked against the oracle."""
    c, h, w, vm = _pick_inputs(11)
    g = sv.adaptive_pick_k(h, w, c["beta"], vm, mode=0)
    a = oc.prefix_survival(oc.confidence(c["hidden"], c["w"], c["beta"]))
    k, _ = oc.pick_k_per_stream(a, c["verify_ms"])
    gk = g["k"].cpu().numpy()
    for b in range(len(k)):
        if not per_stream_tie(a[b], c["verify_ms"], 5):
            assert gk[b] == k[b], b
    inp = workloads.make_verify_inputs("adaptive128", 12, k=k, backend="torch")
    d = {"cu": inp["cu_drafts"], "dq": inp["draft_logits"], "dp": inp["target_logits"],
         "x": inp["draft_tokens"], "T": inp["temperature"]}
    fn = sv.spec_verify_block if rule == ov.RULE_BLOCK else sv.spec_verify_tokenwise
    runs = [(rule, 0, st) for st in range(2)]
    gpu = {run: parity.to_numpy(fn(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 0, run[2], diag=True))
           for run in runs}
    ref = parity.oracle_runs(d, 5, runs, list(range(128)), torch)
    cu = inp["cu_drafts"].cpu().numpy()
    x = inp["draft_tokens"].cpu().numpy()
    totals = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0}
    for run in runs:
        st = parity.compare_verify(gpu[run], ref[run], cu, range(128), x, inp["V"])
        for key in totals:
            totals[key] += st[key]
    parity.check_tie_totals(totals)
