"""Acceptance counters and the adaptive verify step as one CUDA graph, on the GPU.

* spec_accept_counters: the per-position counts equal a host count of the same results, and
  tokens per step = 1 + sum_p a_p equals the mean emitted tokens tau + 1 of the verified
  streams (P1 "MTP, DSpark and Block Verification, Explained", §6 "The arithmetic you need
  before tuning k").
* SpecPipeline (pick k -> verify each stream's first k_b drafts -> counters -> step + 1):
  every replay equals the eager calls - adaptive_pick_k, then the packed verify of the same
  rows at the same step - bit for bit, and the oracle on the same rows.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from oracle import verify as ov  # noqa: E402
from speculative_decoding_block_verify_gb300 import workloads  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu

RESULTS = ("accepted_len", "out_tokens", "n_emitted", "status")


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def test_accept_counters_match_host_count_and_the_tokens_per_step_identity():
    inp = workloads.make_verify_inputs("batch64", 301, B=24, N=5, V=4096,
                                       k=[5, 5, 3, 0, 5, 2] * 4)
    d = parity.verify_to_device(inp, torch)
    cu = inp["cu_drafts"]
    n = np.diff(cu)
    host = np.zeros(11, np.int64)
    emitted = []
    counts = None
    for step in range(6):
        g = sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 0, step)
        counts = sv.spec_accept_counters(g["accepted_len"], g["status"], d["cu"], 5, counts)
        st = g["status"].cpu().numpy()
        tau = g["accepted_len"].cpu().numpy()
        ok = st == 0
        host[0] += ok.sum()
        for p in range(1, 6):
            host[p] += (ok & (tau >= p)).sum()
            host[5 + p] += (ok & (n >= p)).sum()
        emitted.extend((tau[ok] + 1).tolist())
    assert np.array_equal(counts.cpu().numpy(), host)
    a, marg, tps = sv.acceptance_rates(counts, 5)
    assert abs(tps - np.mean(emitted)) < 1e-12
    assert all(0.0 <= x <= 1.0 for x in a) and all(a[i] >= a[i + 1] for i in range(4))


def _dense(seed, B, kmax, V, H):
    """Dense draft [B, kmax, V] / target [B, kmax + 1, V] rows (the packed layout of uniform
    counts kmax), tokens [B, kmax], and the confidence head's inputs."""
    inp = workloads.make_verify_inputs("batch64", seed, B=B, N=kmax, V=V)
    conf = workloads.make_confidence_inputs(seed, B=B, kmax=kmax, H=H, n_max=64)
    dt = torch.bfloat16
    t = lambda a, dtp: torch.as_tensor(np.asarray(a, np.float32)).cuda().to(dtp)  # noqa: E731
    return dict(
        dq=t(inp["draft_logits"], dt).view(B, kmax, V), dp=t(inp["target_logits"], dt).view(B, kmax + 1, V),
        x=torch.as_tensor(inp["draft_tokens"]).cuda().view(B, kmax),
        T=torch.as_tensor(np.maximum(inp["temperature"], 0.3).astype(np.float32)).cuda(),
        hidden=t(conf["hidden"], dt), w=t(conf["w"], dt),
        vm=torch.as_tensor((2.0 + 0.4 * np.arange(65)).astype(np.float32)).cuda())


@pytest.mark.parametrize("rule", [ov.RULE_TOKENWISE, ov.RULE_BLOCK])
def test_pipeline_graph_equals_eager_calls_and_the_oracle(rule):
    B, kmax, V, H = 16, 5, 4096, 512
    d = _dense(401, B, kmax, V, H)
    pl = sv.SpecPipeline(d["hidden"], d["w"], 0.0, d["vm"], d["dq"], d["dp"], d["x"], d["T"], rule=rule,
                         seed=3, step=7, diag=True)
    fn = sv.spec_verify_block if rule == ov.RULE_BLOCK else sv.spec_verify_tokenwise
    host_counts = np.zeros(2 * kmax + 1, np.int64)
    ks = set()
    for it in range(3):
        out = {k: v.clone() for k, v in pl.launch().items()}
        torch.cuda.synchronize()
        pk = sv.adaptive_pick_k(d["hidden"], d["w"], 0.0, d["vm"])
        assert torch.equal(pk["k"], out["k"]) and torch.equal(pk["cu"], out["cu"])
        k = pk["k"].cpu().numpy()
        ks.update(k.tolist())
        cu = workloads.ragged_cu(k)
        rq = [b * kmax + i for b in range(B) for i in range(k[b])]
        rp = [b * (kmax + 1) + i for b in range(B) for i in range(k[b] + 1)]
        dq = d["dq"].reshape(B * kmax, V)[rq].contiguous()
        dp = d["dp"].reshape(B * (kmax + 1), V)[rp].contiguous()
        x = d["x"].reshape(-1)[rq].contiguous()
        g = fn(torch.as_tensor(cu).cuda(), dq, dp, x, d["T"], kmax, 3, 7 + it, diag=True)
        for key in RESULTS:
            assert torch.equal(g[key], out[key]), (it, key)
        assert torch.equal(g["diag"].view(torch.int32), out["diag"][rp].view(torch.int32))
        o = ov.verify_batch(rule, cu, dq.float().cpu().numpy(), dp.float().cpu().numpy(), x.cpu().numpy(),
                            d["T"].cpu().numpy(), kmax, 3, 7 + it)
        gn = parity.to_numpy(g)
        parity.compare_verify(gn, o, cu, range(B), x.cpu().numpy(), V)
        ok = gn["status"] == 0
        host_counts[0] += ok.sum()
        for p in range(1, kmax + 1):
            host_counts[p] += (ok & (gn["accepted_len"] >= p)).sum()
            host_counts[kmax + p] += (ok & (k >= p)).sum()
    assert int(pl.step.item()) == 10
    assert np.array_equal(pl.counts.cpu().numpy(), host_counts)
    assert len(ks) > 1   # the controller gave the streams different counts
    pl.close()
