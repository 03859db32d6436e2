"""GPU parity of the reduced-draft-vocabulary verify calls against the oracle.

P1 "MTP, DSpark and Block Verification, Explained", §3 "The Markov fix-up": draft rows over a
reduced vocabulary scattered into target columns.  The oracle is the dense oracle on the
scattered rows (pinned on the CPU); here the GPU's calls are compared with it:

* small cases (V = 4096, K = 512; ragged counts, greedy streams, both rules, several steps),
  the 16-byte path and the unaligned element path (K not a multiple of 8);
* an identity map (K = V) against the dense call on the same rows, bit for bit;
* a draft token outside the draft vocabulary (ZERO_DRAFT_PROB) and the argument errors;
* dense rows with masked (-inf) columns at twelve temperatures: the exponent of a -inf logit
  must be -inf whatever the sign of the temperature scale's low part;
* the full-size batch64_topk workload (V = 129,280, K = 32,768) in the bench's launch
  configuration, every stream for several steps per rule.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from oracle import verify as ov  # noqa: E402
from speculative_decoding_block_verify_gb300 import workloads  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu

FN = {ov.RULE_TOKENWISE: sv.spec_verify_tokenwise_reduced, ov.RULE_BLOCK: sv.spec_verify_block_reduced}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def _to_device(inp):
    d = parity.verify_to_device(inp, torch)
    d["t2d"] = torch.as_tensor(np.asarray(inp["t2d"], np.int32)).cuda()
    return d


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
@pytest.mark.parametrize("V,K", [(4096, 512), (4093, 509)])
def test_small_cases_match_the_oracle(rule, V, K):
    k = [5, 0, 3, 5, 1, 5, 2, 4, 5, 5, 3, 5]
    inp = workloads.make_verify_inputs("batch64_topk", 81, B=len(k), V=V, K=K, k=k)
    d = _to_device(inp)
    x = np.asarray(inp["draft_tokens"])
    for step in range(6):
        g = parity.to_numpy(FN[rule](d["cu"], d["dq"], d["t2d"], d["dp"], d["x"], d["T"], 5, 11, step, diag=True))
        o = ov.verify_batch_reduced(rule, inp["cu_drafts"], inp["draft_logits"], inp["t2d"], inp["target_logits"], x,
                                    inp["temperature"], 5, 11, step)
        parity.compare_verify(g, o, inp["cu_drafts"], range(len(k)), x, V)


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_identity_map_equals_the_dense_call(rule):
    inp = workloads.make_verify_inputs("batch64", 82, B=16, V=8192)
    d = parity.verify_to_device(inp, torch)
    t2d = torch.arange(8192, dtype=torch.int32, device="cuda")
    dense = sv.spec_verify_block if rule == ov.RULE_BLOCK else sv.spec_verify_tokenwise
    for step in range(4):
        a = dense(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 2, step, diag=True)
        r = FN[rule](d["cu"], d["dq"], t2d, d["dp"], d["x"], d["T"], 5, 2, step, diag=True)
        for key in ("accepted_len", "out_tokens", "n_emitted", "status"):
            assert torch.equal(a[key], r[key]), key
        assert torch.equal(a["diag"].view(torch.int32), r["diag"].view(torch.int32))


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_masked_columns_in_dense_rows_match_the_oracle(rule):
    inp = workloads.make_verify_inputs("batch64", 84, B=12, V=4096)
    rng = np.random.default_rng(84)
    dq = np.asarray(inp["draft_logits"]).copy()
    dp = np.asarray(inp["target_logits"]).copy()
    x = np.asarray(inp["draft_tokens"])
    cu = inp["cu_drafts"]
    for r in range(dq.shape[0]):
        m = rng.random(4096) < 0.3
        m[x[r]] = False                      # keep q(x) > 0
        dq[r, m] = -np.inf
    dp[rng.random(dp.shape) < 0.1] = -np.inf
    inp["draft_logits"], inp["target_logits"] = dq, dp
    inp["temperature"] = np.linspace(0.3, 1.7, 12).astype(np.float32)
    d = parity.verify_to_device(inp, torch)
    dense = sv.spec_verify_block if rule == ov.RULE_BLOCK else sv.spec_verify_tokenwise
    for step in range(4):
        g = parity.to_numpy(dense(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 5, step, diag=True))
        o = ov.verify_batch(rule, cu, dq, dp, x, inp["temperature"], 5, 5, step)
        assert (g["status"] == 0).all(), g["status"]
        parity.compare_verify(g, o, cu, range(12), x, 4096)


def test_token_outside_the_vocabulary_and_argument_errors():
    inp = workloads.make_verify_inputs("batch64_topk", 83, B=4, V=4096, K=512)
    inp["temperature"] = np.full(4, 0.8, np.float32)
    outside = int(np.flatnonzero(np.asarray(inp["t2d"]) < 0)[0])
    inp["draft_tokens"] = np.asarray(inp["draft_tokens"]).copy()
    inp["draft_tokens"][inp["cu_drafts"][2] + 1] = outside
    d = _to_device(inp)
    g = parity.to_numpy(sv.spec_verify_block_reduced(d["cu"], d["dq"], d["t2d"], d["dp"], d["x"], d["T"], 5, 0, 0))
    o = ov.verify_batch_reduced(ov.RULE_BLOCK, inp["cu_drafts"], inp["draft_logits"], inp["t2d"],
                                inp["target_logits"], inp["draft_tokens"], inp["temperature"], 5, 0, 0)
    assert g["status"][2] == ov.STATUS_ZERO_DRAFT_PROB == o["status"][2]
    parity.compare_verify(g, o, inp["cu_drafts"], range(4), inp["draft_tokens"], 4096, check_diag=False)
    L = sv.lib()
    a = sv.VerifyArgs()
    a.B, a.V, a.kmax, a.draft_dtype, a.target_dtype = 0, 4096, 5, 1, 1      # B = 0: no pointer needed
    t2d = d["t2d"].data_ptr()
    assert L.spec_verify_block_reduced(ctypes.byref(a), None, 512, None) == -1    # t2d NULL
    assert L.spec_verify_block_reduced(ctypes.byref(a), t2d, 0, None) == -3       # K outside [1, V]
    assert L.spec_verify_tokenwise_reduced(ctypes.byref(a), t2d, 4097, None) == -3
    assert L.spec_verify_block_reduced(ctypes.byref(a), t2d, 512, None) == 0      # B = 0: nothing to do


def test_batch64_topk_full_size():
    """B = 64, k = 5, V = 129,280 bf16, K = 32,768: four steps per rule, every stream."""
    inp = workloads.make_verify_inputs("batch64_topk", 3000, backend="torch")
    d = {"cu": inp["cu_drafts"], "dq": inp["draft_logits"], "dp": inp["target_logits"], "x": inp["draft_tokens"],
         "T": inp["temperature"], "t2d": inp["t2d"]}
    runs = [(rule, 0, st) for rule in (ov.RULE_TOKENWISE, ov.RULE_BLOCK) for st in range(4)]
    gpu = {run: parity.to_numpy(FN[run[0]](d["cu"], d["dq"], d["t2d"], d["dp"], d["x"], d["T"], 5, 0, run[2],
                                           diag=True)) for run in runs}
    ref = parity.oracle_runs(d, 5, runs, range(64), torch, runs_per_task=2)
    cu = inp["cu_drafts"].cpu().numpy()
    x = inp["draft_tokens"].cpu().numpy()
    totals = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0}
    for run in runs:
        st = parity.compare_verify(gpu[run], ref[run], cu, range(64), x, inp["V"])
        for key in totals:
            totals[key] += st[key]
    parity.check_tie_totals(totals)
    assert totals["streams"] == len(runs) * 64
