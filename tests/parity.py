"""Helpers for GPU-vs-oracle parity (test helper).

Near ties: a decision whose uniform lies within 1e-6 (relative) of its threshold is flagged
by the oracle and that stream is only checked for validity.  A draw over V tokens has V
thresholds, so about 1e-6 * V of the draws are flagged (~13% at V = 129,280 when every
token has mass); MAX_TIE_FRACTION bounds the flagged share per test.
"""

import numpy as np

REL = 1e-5          # probabilities, residual masses, logZ: relative tolerance
ABS_FLOOR = 1e-30   # below this the comparison is absolute (float32 denormal floor)
MAX_TIE_FRACTION = 0.25


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


def compare_verify(g, o, cu, streams, x, V, check_diag=True, rel=REL):
    """Exact comparison of tau / tokens / status outside oracle-flagged near ties, diag
    values within ``rel``.  Returns a dict of counts; raises AssertionError on a mismatch."""
    stats = {"streams": 0, "ties": 0, "exact": 0, "tie_match": 0, "diag_values": 0,
             "diag_max_rel": 0.0}
    for b in streams:
        stats["streams"] += 1
        n = int(cu[b + 1] - cu[b])
        assert g["status"][b] == o["status"][b], (b, g["status"][b], o["status"][b])
        if o["tie"][b]:
            stats["ties"] += 1
            stats["tie_match"] += int(g["accepted_len"][b] == o["accepted_len"][b] and
                                      np.array_equal(g["out_tokens"][b], o["out_tokens"][b]))
            if g["status"][b] == 0:
                tau = int(g["accepted_len"][b])
                assert 0 <= tau <= n and g["n_emitted"][b] == tau + 1
                assert list(g["out_tokens"][b, :tau]) == list(x[int(cu[b]):int(cu[b]) + tau])
                assert 0 <= g["out_tokens"][b, tau] < V
            continue
        assert g["accepted_len"][b] == o["accepted_len"][b], (b, g["accepted_len"][b], o["accepted_len"][b])
        assert g["n_emitted"][b] == o["n_emitted"][b]
        assert np.array_equal(g["out_tokens"][b], o["out_tokens"][b]), (b, g["out_tokens"][b], o["out_tokens"][b])
        stats["exact"] += 1
        if check_diag and "diag" in g:
            r0 = int(cu[b]) + b
            gd = g["diag"][r0:r0 + n + 1].astype(np.float64)
            od = o["diag"][r0:r0 + n + 1]
            have = ~np.isnan(gd)
            assert not np.isnan(od[have]).any(), (b, gd, od)
            gv, ov = gd[have], od[have]
            err = np.abs(gv - ov)
            small = np.abs(ov) < ABS_FLOOR
            relerr = np.where(small, err, err / np.maximum(np.abs(ov), ABS_FLOOR))
            bad = relerr > np.where(small, ABS_FLOOR, rel)
            assert not bad.any(), (b, np.argwhere(have)[bad], gv[bad], ov[bad])
            stats["diag_values"] += int(have.sum())
            if relerr.size:
                stats["diag_max_rel"] = max(stats["diag_max_rel"], float(relerr[~small].max(initial=0.0)))
    return stats
