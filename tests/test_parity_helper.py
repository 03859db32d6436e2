"""The parity helper's process-pool oracle runner gives exactly what the oracle's own batch
function gives (CPU only; host arrays stand in for device tensors)."""

import numpy as np

from oracle import verify as ov
from speculative_decoding_block_verify_gb300 import workloads
from tests import parity


class _NoTorch:
    bfloat16 = object()


def test_oracle_runs_matches_verify_batch():
    inp = workloads.make_verify_inputs("batch64", 5, B=6, V=512)
    d = {"cu": inp["cu_drafts"], "dq": inp["draft_logits"], "dp": inp["target_logits"],
         "x": inp["draft_tokens"], "T": inp["temperature"]}
    runs = [(ov.RULE_BLOCK, 0, s) for s in range(3)] + [(ov.RULE_TOKENWISE, 1, s) for s in range(3)]
    res = parity.oracle_runs(d, inp["kmax"], runs, range(6), _NoTorch, workers=2, runs_per_task=2)
    assert set(res) == set(runs)
    for (rule, seed, step), o in res.items():
        ref = ov.verify_batch(rule, inp["cu_drafts"], inp["draft_logits"], inp["target_logits"],
                              inp["draft_tokens"], inp["temperature"], inp["kmax"], seed, step)
        for k in ("accepted_len", "out_tokens", "n_emitted", "status", "tie"):
            assert np.array_equal(o[k], ref[k]), k
        assert o["outcomes"] == ref["outcomes"]
        assert np.array_equal(np.isnan(o["diag"]), np.isnan(ref["diag"]))
        assert np.array_equal(np.nan_to_num(o["diag"]), np.nan_to_num(ref["diag"]))
