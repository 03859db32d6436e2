"""Helpers for GPU-vs-oracle parity (test helper).

Near ties: a decision whose uniform lies within 1e-6 (relative) of its threshold, or a draw
whose target U R lies within 1e-6 (relative) of a CDF value that decides the token, is flagged
by the oracle.  A flagged stream is not skipped: the oracle lists every (tau, token) outcome
that flipping its near comparisons (and nothing else) and moving the draw inside its window
can give, and the GPU's result must be one of them.  Everything else - the status, the
emitted drafts, the -1 padding and every diagnostic value - is compared as for any stream.
A draw over V tokens has V thresholds, so about 1e-6 * V of the draws are flagged (~13% at
V = 129,280 when every token has mass); MAX_TIE_FRACTION bounds the flagged share per test
and TIE_MATCH_FLOOR asks most flagged streams to still match the oracle's own outcome.

The full-size cases run the oracle on a spawned process pool (safe after CUDA is up) with
each task holding one stream's rows.
"""

import multiprocessing as mp
import os

import numpy as np

REL = 1e-5          # probabilities, residual masses, logZ: relative tolerance
ABS_FLOOR = 1e-30   # below this the comparison is absolute (float32 denormal floor)
# Residual masses are sums of max(0, w p - q) computed per element in float32: each term's
# exponent is rounded to ~2^-24 of |l a - K| <= ~30 and 2^x carries ~2^-22, so a term is off by
# at most ~1.5e-6 (w p + q) and the sum by at most RESID_GROSS * G, G = the positive part's
# gross mass (oracle residual_gross).  Where the residual is a small difference of large terms
# that bound, not 1e-5 of the residual, is what float32 arithmetic attains; h = r / (r + 1 - w)
# inherits the same relative slack.
RESID_GROSS = 3e-6
MAX_TIE_FRACTION = 0.25
TIE_MATCH_FLOOR = 0.5   # of the flagged streams (when there are at least 4)


def verify_to_device(inp, torch, device="cuda"):
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32
    return dict(
        cu=torch.as_tensor(np.asarray(inp["cu_drafts"], np.int32)).to(device),
        dq=torch.as_tensor(np.asarray(inp["draft_logits"], np.float32)).to(device).to(dt),
        dp=torch.as_tensor(np.asarray(inp["target_logits"], np.float32)).to(device).to(dt),
        x=torch.as_tensor(np.asarray(inp["draft_tokens"], np.int32)).to(device),
        T=torch.as_tensor(np.asarray(inp["temperature"], np.float32)).to(device),
    )


def to_numpy(out):
    return {k: v.cpu().numpy() for k, v in out.items()}


def _check_diag(g, o, b, r0, n, rel, stats):
    gd = g["diag"][r0:r0 + n + 1].astype(np.float64)
    od = o["diag"][r0:r0 + n + 1]
    have = ~np.isnan(gd)
    assert not np.isnan(od[have]).any(), (b, gd, od)
    # per-value relative tolerance: rel, widened for r and h by the cancellation bound
    tol = np.full(od.shape, rel)
    if "gross" in o:
        gross = o["gross"][r0:r0 + n + 1]
        r = od[:, 4]
        with np.errstate(divide="ignore", invalid="ignore"):
            extra = np.where(np.isfinite(gross) & (r > 0), RESID_GROSS * gross / r, 0.0)
        tol[:, 4] += extra   # SPEC_DIAG_R
        tol[:, 3] += extra   # SPEC_DIAG_H
    tol = tol[have]
    gv, ov = gd[have], od[have]
    err = np.abs(gv - ov)
    small = np.abs(ov) < ABS_FLOOR
    relerr = np.where(small, err, err / np.maximum(np.abs(ov), ABS_FLOOR))
    bad = relerr > np.where(small, ABS_FLOOR, tol)
    assert not bad.any(), (b, np.argwhere(have)[bad], gv[bad], ov[bad])
    stats["diag_values"] += int(have.sum())
    if relerr.size:
        stats["diag_max_rel"] = max(stats["diag_max_rel"], float(relerr[~small].max(initial=0.0)))


def compare_verify(g, o, cu, streams, x, V, check_diag=True, rel=REL):
    """Exact comparison of tau / tokens / status for every stream; for a stream the oracle
    flags, (tau, token) must be one of the oracle's admissible outcomes.  Diag values within
    ``rel`` for every stream with status OK.  Returns a dict of counts; raises AssertionError
    on a mismatch."""
    stats = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0, "diag_values": 0,
             "diag_max_rel": 0.0}
    x = np.asarray(x)
    for b in streams:
        stats["streams"] += 1
        n = int(cu[b + 1] - cu[b])
        assert g["status"][b] == o["status"][b], (b, g["status"][b], o["status"][b])
        if g["status"][b] != 0:
            assert g["n_emitted"][b] == 0 and (g["out_tokens"][b] == -1).all(), b
            continue
        tau = int(g["accepted_len"][b])
        assert 0 <= tau <= n and g["n_emitted"][b] == tau + 1, (b, tau, g["n_emitted"][b])
        assert list(g["out_tokens"][b, :tau]) == list(x[int(cu[b]):int(cu[b]) + tau]), b
        assert (g["out_tokens"][b, tau + 1:] == -1).all(), b
        same = (tau == o["accepted_len"][b] and np.array_equal(g["out_tokens"][b], o["out_tokens"][b]))
        if o["tie"][b]:
            stats["ties"] += 1
            stats["tie_match"] += int(same)
            tok = int(g["out_tokens"][b, tau])
            ok = any(tau == t and tok in toks for t, toks in o["outcomes"][b])
            assert ok, (b, "near tie: GPU outcome not admissible", tau, tok, o["outcomes"][b])
        else:
            assert same, (b, tau, g["out_tokens"][b], o["accepted_len"][b], o["out_tokens"][b])
            stats["exact"] += 1
        if check_diag and "diag" in g:
            _check_diag(g, o, b, int(cu[b]) + b, n, rel, stats)
    return stats


def check_tie_totals(totals):
    """The flagged share stays bounded and most flagged streams still match exactly."""
    assert totals["ties"] <= max(2, MAX_TIE_FRACTION * totals["streams"]), totals
    if totals["ties"] >= 4:
        assert totals["tie_match"] >= TIE_MATCH_FLOOR * totals["ties"], totals


# ---------------------------------------------------------------------------------------
# the oracle over many streams and steps on the host cores
# ---------------------------------------------------------------------------------------
def _widen(rows, kind):
    if kind == "bf16":
        return (rows.astype(np.uint32) << 16).view(np.float32)
    return rows


def _stream_task(args):
    runs, q_rows, kq, p_rows, kp, x, T, b, t2d = args
    from oracle import verify as ov
    q = _widen(q_rows, kq)
    if t2d is not None:   # draft rows over a reduced draft vocabulary, scattered into target columns
        sc = ov.ScatteredRows(q, t2d)
        q = [sc[i] for i in range(len(q))]
    p = _widen(p_rows, kp)
    return [ov.verify_stream(rule, q, p, x, T, seed, step, b) for rule, seed, step in runs]


def device_rows(t, r0, r1, torch):
    """Rows [r0, r1) of a device logit tensor as host data: bf16 bit patterns (uint16) or
    float32 (halves the transfer to the workers for bf16); a host (numpy) array is sliced as
    it is (float64 stays float64)."""
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t[r0:r1]), "host"
    if r1 <= r0:
        return np.zeros((0, t.shape[1]), np.float32), "f32"
    if t.dtype == torch.bfloat16:
        return t[r0:r1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16"
    return t[r0:r1].float().cpu().numpy(), "f32"


def _host(a):
    return a if isinstance(a, np.ndarray) else a.cpu().numpy()


def oracle_runs(d, kmax, runs, streams, torch, workers=None, runs_per_task=None):
    """Run the oracle for every (rule, seed, step) in ``runs`` over ``streams`` of the inputs
    d = {cu, dq, dp, x, T} (device tensors; dq / dp may also be host arrays; an optional
    ``t2d`` marks dq as rows over a reduced draft vocabulary); returns
    {(rule, seed, step): batch result like oracle.verify.verify_batch (only ``streams``
    filled)}.  A stream's runs are split into tasks of ``runs_per_task``."""
    from oracle import verify as ov
    cu = _host(d["cu"])
    x = _host(d["x"])
    T = _host(d["T"])
    t2d = _host(d["t2d"]) if d.get("t2d") is not None else None
    B = len(cu) - 1
    first_bad = B
    for b in range(B):
        n = cu[b + 1] - cu[b]
        if n < 0 or n > kmax or (b == 0 and cu[0] != 0):
            first_bad = b
            break
    assert first_bad == B, "oracle_runs takes valid offsets only"
    runs = list(runs)
    per = runs_per_task or len(runs)
    tasks, where = [], []
    for b in streams:
        n = int(cu[b + 1] - cu[b])
        q, kq = device_rows(d["dq"], int(cu[b]), int(cu[b]) + n, torch)
        p, kp = device_rows(d["dp"], int(cu[b]) + b, int(cu[b]) + b + n + 1, torch)
        for k0 in range(0, len(runs), per):
            tasks.append((runs[k0:k0 + per], q, kq, p, kp, x[cu[b]:cu[b] + n], float(T[b]), b, t2d))
            where.append((b, k0))
    workers = workers or max(1, min(len(tasks), len(os.sched_getaffinity(0))))
    with mp.get_context("spawn").Pool(workers) as pool:
        chunks = pool.map(_stream_task, tasks, chunksize=1)
    by_stream = {}
    for (b, k0), c in zip(where, chunks):
        by_stream.setdefault(b, {})[k0] = c
    res = [sum((by_stream[b][k0] for k0 in sorted(by_stream[b])), []) for b in streams]
    out = {}
    for k, run in enumerate(runs):
        o = {"accepted_len": np.zeros(B, np.int32), "out_tokens": np.full((B, kmax + 1), -1, np.int32),
             "n_emitted": np.zeros(B, np.int32), "status": np.full(B, -1, np.int32),
             "diag": np.full((int(cu[-1]) + B, ov.DIAG_COLS), np.nan), "tie": np.zeros(B, bool),
             "tie_kind": [None] * B, "outcomes": [[] for _ in range(B)],
             "gross": np.full(int(cu[-1]) + B, np.nan)}
        for j, b in enumerate(streams):
            r = res[j][k]
            n = int(cu[b + 1] - cu[b])
            o["status"][b] = r["status"]
            o["tie"][b] = r["tie"]
            o["tie_kind"][b] = r["tie_kind"]
            o["outcomes"][b] = r["outcomes"]
            if r["status"] == ov.STATUS_OK:
                o["accepted_len"][b] = r["tau"]
                o["n_emitted"][b] = r["n_emitted"]
                o["out_tokens"][b, :len(r["emitted"])] = r["emitted"]
            if float(T[b]) > 0.0 and r["status"] in (ov.STATUS_OK, ov.STATUS_NUMERIC):
                o["diag"][cu[b] + b: cu[b] + b + n + 1] = r["diag"]
                o["gross"][cu[b] + b: cu[b] + b + n + 1] = r["gross"]
        out[run] = o
    return out
