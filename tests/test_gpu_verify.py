"""GPU parity of spec_verify_tokenwise / spec_verify_block against the float64 oracle.

Every call goes through the C ABI (ctypes binding).  Accepted lengths, emitted tokens and
status codes must match exactly; where the oracle flags a near tie (a uniform within 1e-6
relative of its threshold) the GPU's (tau, token) must be one of the outcomes the oracle
lists for it.  Diagnostic probabilities, residual masses and log normalisers must agree within
1e-5 relative on every stream.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from oracle import verify as ov  # noqa: E402
from speculative_decoding_block_verify_gb300 import workloads  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu

RULES = {"tokenwise": (ov.RULE_TOKENWISE, sv.spec_verify_tokenwise),
         "block": (ov.RULE_BLOCK, sv.spec_verify_block)}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


class RowView:
    """Row-indexable view of a device tensor for the oracle (rows copied on demand)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, i):
        return self.t[int(i)].float().cpu().numpy()


def run_gpu(rule_name, d, kmax, seed, step, diag=True):
    fn = RULES[rule_name][1]
    return parity.to_numpy(fn(d["cu"], d["dq"], d["dp"], d["x"], d["T"], kmax, seed, step, diag=diag))


def run_oracle(rule_name, inp, seed, step, streams=None, dq=None, dp=None):
    return ov.verify_batch(RULES[rule_name][0], inp["cu_drafts"],
                           inp["draft_logits"] if dq is None else dq,
                           inp["target_logits"] if dp is None else dp,
                           inp["draft_tokens"], inp["temperature"], inp["kmax"], seed, step,
                           streams=streams)


def check(inp, rule_name, seeds_steps, d=None, streams=None, dq=None, dp=None, check_diag=True):
    d = parity.verify_to_device(inp, torch) if d is None else d
    totals = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0}
    B = len(inp["cu_drafts"]) - 1
    streams = range(B) if streams is None else streams
    for seed, step in seeds_steps:
        g = run_gpu(rule_name, d, inp["kmax"], seed, step)
        o = run_oracle(rule_name, inp, seed, step, streams, dq, dp)
        st = parity.compare_verify(g, o, inp["cu_drafts"], streams, np.asarray(inp["draft_tokens"]),
                                   inp["V"], check_diag=check_diag)
        for k in totals:
            totals[k] += st[k]
    parity.check_tie_totals(totals)
    return totals


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_tiny_fp32_many_steps(rule):
    inp = workloads.make_verify_inputs("tiny", 1000)
    check(inp, rule, [(0, s) for s in range(150)])


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
@pytest.mark.parametrize("dtype,V", [("f32", 3000), ("bf16", 4096), ("f32", 4099), ("bf16", 1001)])
def test_small_batches_vector_and_scalar_paths(rule, dtype, V):
    name = "tiny" if dtype == "f32" else "batch64"
    inp = workloads.make_verify_inputs(name, 17 + V, B=12, N=5, V=V)
    check(inp, rule, [(3, s) for s in range(6)])


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_ragged_offsets_and_max_kmax(rule):
    inp = workloads.make_verify_inputs("tiny", 23, B=6, V=2048, k=[0, 1, 32, 3, 0, 7])
    inp["kmax"] = 32
    check(inp, rule, [(5, s) for s in range(8)])


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_greedy_and_sampled_streams_mixed(rule):
    inp = workloads.make_verify_inputs("batch64", 31, B=40, V=4096)
    assert (inp["temperature"] == 0).sum() == 2
    check(inp, rule, [(9, s) for s in range(5)])


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_degenerate_vocab_and_wide_vocab(rule):
    inp = workloads.make_verify_inputs("tiny", 41, B=3, N=4, V=1)
    check(inp, rule, [(0, 0), (0, 1)])
    g = run_gpu(rule, parity.verify_to_device(inp, torch), inp["kmax"], 0, 0)
    assert (g["accepted_len"] == 4).all() and (g["out_tokens"][:, :5] == 0).all()
    big = workloads.make_verify_inputs("tiny", 43, B=1, N=2, V=1 << 24)
    check(big, rule, [(1, 0)])


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_identical_draft_and_target_accept_all(rule):
    inp = workloads.make_verify_inputs("batch64", 47, B=8, N=5, V=2048)
    cu = inp["cu_drafts"]
    for b in range(8):
        for i in range(5):
            inp["draft_logits"][cu[b] + i] = inp["target_logits"][cu[b] + b + i]
    inp["temperature"][:] = 0.9
    g = run_gpu(rule, parity.verify_to_device(inp, torch), 5, 1, 2)
    assert (g["status"] == 0).all() and (g["accepted_len"] == 5).all()


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_status_codes(rule):
    inp = workloads.make_verify_inputs("tiny", 53, B=10, N=3, V=256)
    cu, dq, dp, x, T = (inp[k] for k in ("cu_drafts", "draft_logits", "target_logits",
                                         "draft_tokens", "temperature"))
    dp[cu[0] + 0 + 1, 7] = np.nan                     # stream 0: NaN in a target row
    dq[cu[1] + 2, 100] = np.inf                       # stream 1: +inf in a draft row
    dp[cu[2] + 2 + 3, :] = -np.inf                    # stream 2: bonus row all -inf
    x[cu[3] + 1] = 256                                # stream 3: token out of range
    T[4] = -0.5                                       # stream 4: negative temperature
    T[5] = np.float32(1e-40)                          # stream 5: subnormal temperature
    dq[cu[6] + 1, x[cu[6] + 1]] = -np.inf             # stream 6: q(x) = 0
    T[7] = 0.0                                        # stream 7: greedy, with a NaN draft row
    dq[cu[7], 5] = np.nan
    T[8] = np.nan                                     # stream 8: NaN temperature
    g = run_gpu(rule, parity.verify_to_device(inp, torch), 3, 0, 0)
    o = run_oracle(rule, inp, 0, 0)
    assert list(g["status"]) == list(o["status"])
    assert list(g["status"]) == [3, 3, 3, 2, 1, 1, 4, 0, 1, 0]
    bad = g["status"] != 0
    assert (g["n_emitted"][bad] == 0).all() and (g["out_tokens"][bad] == -1).all()
    assert np.isnan(g["diag"][cu[0]:cu[1] + 1]).all()


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_bad_offsets(rule):
    inp = workloads.make_verify_inputs("tiny", 59, B=3, N=2, V=64)
    d = parity.verify_to_device(inp, torch)
    d["cu"] = torch.tensor([0, 2, 1, 6], dtype=torch.int32, device="cuda")   # N = 2, -1, 5
    g = run_gpu(rule, d, 2, 0, 0, diag=False)
    assert list(g["status"]) == [0, 5, 5]
    assert (g["out_tokens"][1:] == -1).all()
    # a stream with a valid count after a broken one, and a batch not starting at row 0
    for cu, want in (([0, 1, 5, 6], [0, 5, 5]), ([1, 2, 3, 4], [5, 5, 5]), ([0, 1, 3, 4], None)):
        d["cu"] = torch.tensor(cu, dtype=torch.int32, device="cuda")
        g = run_gpu(rule, d, 2, 0, 0, diag=False)
        o = run_oracle(rule, dict(inp, cu_drafts=np.array(cu, np.int32), kmax=2), 0, 0)
        assert list(g["status"]) == list(o["status"])
        assert want is None or list(g["status"]) == want
        ok = (o["status"] == 0) & ~o["tie"]
        assert (g["accepted_len"][ok] == o["accepted_len"][ok]).all()


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_unaligned_rows_take_the_plain_path(rule):
    inp = workloads.make_verify_inputs("tiny", 61, B=4, N=3, V=1024)
    d = parity.verify_to_device(inp, torch)
    for k in ("dq", "dp"):
        t = d[k]
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        buf[1:] = t.reshape(-1)
        d[k] = buf[1:].view(t.shape)                    # data_ptr % 16 != 0
    assert d["dp"].data_ptr() % 16 != 0
    check(inp, rule, [(2, s) for s in range(4)], d=d)


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_mixed_dtypes(rule):
    inp = workloads.make_verify_inputs("batch64", 67, B=6, N=5, V=2048)
    d = parity.verify_to_device(inp, torch)
    d["dq"] = d["dq"].float()                           # draft float32, target bf16
    check(inp, rule, [(4, s) for s in range(4)], d=d)


def test_same_seed_same_bytes():
    inp = workloads.make_verify_inputs("batch64", 71, B=16, N=5, V=8192)
    d = parity.verify_to_device(inp, torch)
    for rule in RULES:
        ref = run_gpu(rule, d, 5, 11, 12)
        for _ in range(30):
            g = run_gpu(rule, d, 5, 11, 12)
            for k in ref:
                if k == "workspace":   # scratch, not an output: unread parts keep old contents
                    continue
                assert np.array_equal(ref[k].view(np.uint8), g[k].view(np.uint8)), k


def test_empty_batch():
    d = {"cu": torch.zeros(1, dtype=torch.int32, device="cuda"),
         "dq": torch.empty((0, 16), dtype=torch.bfloat16, device="cuda"),
         "dp": torch.empty((0, 16), dtype=torch.bfloat16, device="cuda"),
         "x": torch.empty(0, dtype=torch.int32, device="cuda"),
         "T": torch.empty(0, dtype=torch.float32, device="cuda")}
    g = run_gpu("block", d, 5, 0, 0)
    assert g["status"].size == 0


def full_size_parity(name, seeds, rule_names, steps, streams=None, kmax=None):
    """GPU calls of the given rules over `steps` consecutive steps on each seeded full-size
    input set, every listed stream checked against the oracle (run on the host cores)."""
    totals = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0}
    for seed in seeds:
        inp = workloads.make_verify_inputs(name, seed, backend="torch")
        d = {"cu": inp["cu_drafts"], "dq": inp["draft_logits"], "dp": inp["target_logits"],
             "x": inp["draft_tokens"], "T": inp["temperature"]}
        B = inp["B"]
        k = inp["kmax"] if kmax is None else kmax
        ss = list(range(B)) if streams is None else streams
        runs = [(RULES[r][0], 0, st) for r in rule_names for st in range(steps)]
        gpu = {}
        for r in rule_names:
            for st in range(steps):
                gpu[(RULES[r][0], 0, st)] = run_gpu(r, d, k, 0, st)
        ref = parity.oracle_runs(d, k, runs, ss, torch, runs_per_task=max(1, len(runs) // 4))
        cu = inp["cu_drafts"].cpu().numpy()
        x = inp["draft_tokens"].cpu().numpy()
        for run in runs:
            st = parity.compare_verify(gpu[run], ref[run], cu, ss, x, inp["V"])
            for key in totals:
                totals[key] += st[key]
        del d, inp
        torch.cuda.empty_cache()
    parity.check_tie_totals(totals)
    return totals


def test_batch64_full_size():
    """B = 64, k = 5, V = 129,280 bf16, in the launch configuration the bench times: 20 steps
    per rule on each of two input sets, every stream."""
    t = full_size_parity("batch64", [3000, 3017], ["tokenwise", "block"], 20)
    assert t["streams"] == 2 * 2 * 20 * 64


def test_batch256_k9_fp32_full_size():
    """B = 256, k = 9, V = 129,280 fp32, block only: every stream for two steps."""
    t = full_size_parity("batch256_k9", [4000], ["block"], 2)
    assert t["streams"] == 2 * 256


def test_uniforms_bit_exact_against_oracle():
    from oracle import philox
    n_streams, n_slots = 1000, 1000
    for seed, step in [(0, 0), (0x0123456789ABCDEF, 0xFEDCBA9876543210)]:
        g = sv.spec_philox_uniforms(seed, step, n_streams, n_slots).cpu().numpy()
        s, i = np.meshgrid(np.arange(n_streams), np.arange(n_slots), indexing="ij")
        ua, us = philox.slot_uniforms_np(seed, np.full(s.shape, step, np.uint64), s, i)
        assert np.array_equal(g[..., 0], ua) and np.array_equal(g[..., 1], us)


HEADER, ROW = 256, 1536


def _row_counters(ws, rows):
    """The header's tickets (the sweep's ticket and count, the stats tail's eight tickets) and
    the three 32-bit counters at the head of the first `rows`
    1536-byte row blocks of a workspace (all of them zero between calls)."""
    head = ws[:80].contiguous().view(torch.int64).cpu().numpy()
    blocks = ws[HEADER: HEADER + rows * ROW].view(rows, ROW)[:, :12].contiguous().view(torch.int32)
    return np.concatenate([head, blocks.cpu().numpy().reshape(-1)])


@pytest.mark.parametrize("rule", ["tokenwise", "block"])
def test_workspace_reuse_across_batches(rule):
    """One zero-filled workspace serves calls of different B, kmax and stream states (a bad
    token, a greedy stream): the results equal those on fresh workspaces, and after every call
    each row counter is back at zero."""
    fn = RULES[rule][1]
    big = workloads.make_verify_inputs("batch64", 91, B=12, N=5, V=8192)
    small = workloads.make_verify_inputs("batch64", 92, B=5, N=3, V=8192)
    d_big = parity.verify_to_device(big, torch)
    d_small = parity.verify_to_device(small, torch)
    d_bad = dict(d_big)
    d_bad["x"] = d_big["x"].clone()
    d_bad["x"][int(big["cu_drafts"][2])] = 8192          # stream 2: token out of range
    d_bad["T"] = d_big["T"].clone()
    d_bad["T"][4] = 0.0                                  # stream 4: greedy
    cases = [(d_small, 3), (d_big, 5), (d_bad, 5), (d_small, 3), (d_big, 5)]
    ws = torch.zeros(sv.spec_verify_workspace_bytes(12, 5), dtype=torch.uint8, device="cuda")
    for d, kmax in cases:
        B = d["cu"].numel() - 1
        fresh = parity.to_numpy(fn(d["cu"], d["dq"], d["dp"], d["x"], d["T"], kmax, 7, 1))
        o = {"accepted_len": torch.empty(B, dtype=torch.int32, device="cuda"),
             "out_tokens": torch.empty((B, kmax + 1), dtype=torch.int32, device="cuda"),
             "n_emitted": torch.empty(B, dtype=torch.int32, device="cuda"),
             "status": torch.empty(B, dtype=torch.int32, device="cuda"),
             "workspace": ws}
        got = parity.to_numpy(fn(d["cu"], d["dq"], d["dp"], d["x"], d["T"], kmax, 7, 1, out=o))
        for k in ("accepted_len", "out_tokens", "n_emitted", "status"):
            assert np.array_equal(fresh[k], got[k]), k
        assert not _row_counters(ws, 12 * 11).any()
    st = parity.to_numpy(fn(d_bad["cu"], d_bad["dq"], d_bad["dp"], d_bad["x"], d_bad["T"], 5, 7, 1))["status"]
    assert st[2] == 2 and st[4] == 0   # SPEC_ST_BAD_TOKEN, and the greedy stream verifies


def test_bad_row_counter_times_out_and_heals():
    """A row counter that does not match its row's piece count (a workspace that was not
    zero-filled) gives that stream SPEC_ST_TIMEOUT; the other streams are unaffected, the call
    resets the counter, and the next call on the workspace is exact."""
    inp = workloads.make_verify_inputs("batch64", 93, B=6, N=4, V=8192)
    inp["temperature"][:] = np.maximum(inp["temperature"], 0.5)   # every stream samples
    d = parity.verify_to_device(inp, torch)
    fresh = parity.to_numpy(sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 4, 5, 2))
    assert (fresh["status"] == 0).all()
    B = 6
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, 4), dtype=torch.uint8, device="cuda")
    cu = inp["cu_drafts"]
    rho = 2 * int(cu[3]) + 3                              # stream 3's first target row
    ws[HEADER + rho * ROW: HEADER + rho * ROW + 4].view(torch.int32)[0] = 1 << 20
    o = {"accepted_len": torch.empty(B, dtype=torch.int32, device="cuda"),
         "out_tokens": torch.empty((B, 5), dtype=torch.int32, device="cuda"),
         "n_emitted": torch.empty(B, dtype=torch.int32, device="cuda"),
         "status": torch.empty(B, dtype=torch.int32, device="cuda"),
         "workspace": ws}
    got = parity.to_numpy(sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 4, 5, 2, out=o))
    assert got["status"][3] == 6 and got["n_emitted"][3] == 0   # SPEC_ST_TIMEOUT, nothing emitted
    others = [b for b in range(B) if b != 3]
    for k in ("accepted_len", "out_tokens", "n_emitted", "status"):
        assert np.array_equal(fresh[k][others], got[k][others]), k
    assert not _row_counters(ws, B * 9).any()
    again = parity.to_numpy(sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 4, 5, 2, out=o))
    for k in ("accepted_len", "out_tokens", "n_emitted", "status"):
        assert np.array_equal(fresh[k], again[k]), k


def test_garbage_workspace_header_heals():
    """Sweep ticket and work-list count left non-zero in the header (a workspace that was not
    zero-filled): the call resets them before use and its results equal a fresh workspace's."""
    inp = workloads.make_verify_inputs("batch64", 95, B=8, N=5, V=8192)
    d = parity.verify_to_device(inp, torch)
    fresh = parity.to_numpy(sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 3, 4))
    B = 8
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, 5), dtype=torch.uint8, device="cuda")
    ws[0:16].view(torch.int64)[:] = torch.tensor([123456789, 987654321], dtype=torch.int64, device="cuda")
    o = {"accepted_len": torch.empty(B, dtype=torch.int32, device="cuda"),
         "out_tokens": torch.empty((B, 6), dtype=torch.int32, device="cuda"),
         "n_emitted": torch.empty(B, dtype=torch.int32, device="cuda"),
         "status": torch.empty(B, dtype=torch.int32, device="cuda"),
         "workspace": ws}
    got = parity.to_numpy(sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 3, 4, out=o))
    for k in ("accepted_len", "out_tokens", "n_emitted", "status"):
        assert np.array_equal(fresh[k], got[k]), k
    assert not _row_counters(ws, B * 11).any()
