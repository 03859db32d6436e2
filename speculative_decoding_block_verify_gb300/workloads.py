"""Seeded synthetic inputs for the verify sampler.

This module only draws random numbers and lays them out in the library's input layout; it
holds none of the verify method's arithmetic (no softmax, no ratio, no residual, no decision,
no bias product).  It is the one module that both the oracle-side tests and the GPU side
read, so both see the same bytes.

Workloads (shapes from the pages' serving lane: V = 129,280, the trained block k = 5, the
k = 9 stress setting, a batch-64 decode; values are synthetic and stand in for the pages'
private transcripts):

* ``tiny``         B=1, k=5, V=1024, fp32.  target ~ N(0, 2^2); draft = target + N(0, 0.5^2);
                   T=1; Markov W1 [V,16], W2 [16,V] fp32 ~ N(0, 0.02^2); prev ~ U[0, V).
* ``single_bias``  B=1, k=5, V=129,280, bf16.  target ~ N(0, 2.5^2); draft = target +
                   N(0, 0.7^2); W1 [V,256], W2 [256,V] bf16 ~ N(0, 0.02^2); prev ~ U[0, V); T=1.
* ``batch64``      B=64, k=5, V=129,280, bf16.  target ~ N(0, 2.5^2); per-stream draft noise
                   sigma_b ~ U[0.2, 2.0]; T_b ~ U[0.3, 1.0]; round(0.05 * 64) = 3 greedy
                   (T = 0) streams chosen by a seeded permutation.
* ``batch256_k9``  B=256, k=9, V=129,280, fp32.  target ~ N(0, 2.5^2); draft noise sigma grows
                   linearly with the slot, 0.3 + 2.2 * i / 8 for i = 0..8; T = 0.7.
* ``adaptive128``  B=128, kmax=5, H=7168 bf16 hidden ~ N(0, 1); head w ~ N(0, 0.02^2) bf16,
                   beta = 0; verify_ms[n] = 12 + 2.6 n for n = 1..768; ragged verify logits
                   with the batch64 statistics at T = 1 for a given per-stream k.
* ``batch64_topk`` the batch64 workload with a reduced draft vocabulary of K = 32,768 target
                   columns (a seeded random subset, in ascending order: d2t [K], and its
                   inverse t2d [V], -1 outside): the draft rows are [cu[B], K] (the batch64
                   draft noise on the target logits at those columns), the draft tokens are
                   target ids sampled over the reduced vocabulary, and the target logits at
                   the reduced columns are raised by 3 (so that, as for a reduced vocabulary
                   of frequent tokens, most of the target mass lies inside it).

Draft tokens: for T > 0, x_i is drawn from softmax(draft_i / T) with the Gumbel-max trick
(argmax of draft_i / T + Gumbel noise) on the *unbiased* draft logits; for T = 0 it is the
draft row's argmax.  bf16 values are float32 rounded to nearest-even; all arrays are returned
as float32 holding exactly the bytes the GPU sees.

Two back-ends: ``numpy`` (PCG64, identical on every machine; used by the CPU tests and the
small cases) and ``torch`` (a seeded torch generator on the given device; used for the large
cases on the GPU, where the oracle then reads the generated tensors back).
"""

import numpy as np

V_FULL = 129280

WORKLOADS = {
    "tiny": dict(B=1, N=5, V=1024, dtype="f32", target_std=2.0, noise=("const", 0.5),
                 temp=("const", 1.0), greedy_frac=0.0, rank=16),
    "single_bias": dict(B=1, N=5, V=V_FULL, dtype="bf16", target_std=2.5, noise=("const", 0.7),
                        temp=("const", 1.0), greedy_frac=0.0, rank=256),
    "batch64": dict(B=64, N=5, V=V_FULL, dtype="bf16", target_std=2.5,
                    noise=("stream_uniform", 0.2, 2.0), temp=("stream_uniform", 0.3, 1.0),
                    greedy_frac=0.05, rank=0),
    "batch256_k9": dict(B=256, N=9, V=V_FULL, dtype="f32", target_std=2.5,
                        noise=("slot_linear", 0.3, 2.5), temp=("const", 0.7), greedy_frac=0.0,
                        rank=0),
    "adaptive128": dict(B=128, N=5, V=V_FULL, dtype="bf16", target_std=2.5,
                        noise=("stream_uniform", 0.2, 2.0), temp=("const", 1.0), greedy_frac=0.0,
                        rank=0, H=7168),
    "batch64_topk": dict(B=64, N=5, V=V_FULL, dtype="bf16", target_std=2.5,
                         noise=("stream_uniform", 0.2, 2.0), temp=("stream_uniform", 0.3, 1.0),
                         greedy_frac=0.05, rank=0, draft_vocab=32768, vocab_boost=3.0),
}


def make_draft_vocab(seed, V, K):
    """A reduced draft vocabulary: d2t [K] (ascending target columns, a seeded random subset)
    and its inverse t2d [V] (-1 for columns outside it).  Pure layout."""
    rng = np.random.Generator(np.random.PCG64(seed + 31337))
    d2t = np.sort(rng.permutation(V)[:K]).astype(np.int32)
    t2d = np.full(V, -1, np.int32)
    t2d[d2t] = np.arange(K, dtype=np.int32)
    return d2t, t2d


def round_bf16(a):
    """float32 -> nearest-even bfloat16, returned as float32 (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + (((u >> 16) & 1) + 0x7FFF)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _as_dtype(a, dtype):
    return round_bf16(a) if dtype == "bf16" else np.asarray(a, np.float32)


def _noise_std(spec, B, N, rng_uniform):
    kind = spec[0]
    if kind == "const":
        return np.full((B, N), spec[1])
    if kind == "stream_uniform":
        s = rng_uniform(spec[1], spec[2], B)
        return np.repeat(s[:, None], N, axis=1)
    if kind == "slot_linear":
        lo, hi = spec[1], spec[2]
        per_slot = lo + (hi - lo) * np.arange(N) / max(N - 1, 1)
        return np.repeat(per_slot[None, :], B, axis=0)
    raise ValueError(kind)


def _temps(spec, B, rng_uniform):
    if spec[0] == "const":
        return np.full(B, spec[1], np.float32)
    return rng_uniform(spec[1], spec[2], B).astype(np.float32)


def ragged_cu(k):
    """cu_drafts [B+1] (exclusive prefix sum of per-stream draft counts) - pure layout."""
    k = np.asarray(k, np.int64)
    return np.concatenate([[0], np.cumsum(k)]).astype(np.int32)


def make_verify_inputs(name, seed, *, B=None, N=None, V=None, k=None, K=None, backend="numpy",
                       device=None):
    """Synthetic verify inputs for workload ``name``.

    Optional overrides B, N (uniform k) or k (ragged per-stream draft counts), V.
    Returns a dict with numpy arrays (``numpy`` back-end) or torch tensors on ``device``
    (``torch`` back-end): cu_drafts [B+1] int32, draft_logits [cu[B], V] float32,
    target_logits [cu[B]+B, V] float32, draft_tokens [cu[B]] int32, temperature [B]
    float32, plus B, V, kmax, dtype, name.  A workload with a reduced draft vocabulary (size
    K, overridable) returns draft_logits [cu[B], K] instead, plus d2t [K], t2d [V] and K.
    """
    spec = dict(WORKLOADS[name])
    if "draft_vocab" in spec and K is not None:
        spec["draft_vocab"] = K
    B = spec["B"] if B is None else B
    V = spec["V"] if V is None else V
    if k is None:
        n = spec["N"] if N is None else N
        k = np.full(B, n, np.int32)
    k = np.asarray(k, np.int32)
    assert len(k) == B
    cu = ragged_cu(k)
    kmax = int(max(spec["N"], k.max() if B else 0))
    if backend == "numpy":
        return _make_numpy(spec, name, seed, B, V, k, cu, kmax)
    return _make_torch(spec, name, seed, B, V, k, cu, kmax, device)


def _layout_noise(spec, B, k, rng_uniform):
    kmax_local = int(k.max()) if B else 0
    std = _noise_std(spec["noise"], B, max(kmax_local, 1), rng_uniform)
    return std


def _make_numpy(spec, name, seed, B, V, k, cu, kmax):
    rng = np.random.Generator(np.random.PCG64(seed))
    n_draft = int(cu[-1])
    n_target = n_draft + B
    target = (rng.standard_normal((n_target, V), dtype=np.float32) * spec["target_std"])
    reduced = "draft_vocab" in spec
    if reduced:
        d2t, t2d = make_draft_vocab(seed, V, spec["draft_vocab"])
        target[:, d2t] += np.float32(spec["vocab_boost"])
    cols = d2t if reduced else slice(None)
    width = len(d2t) if reduced else V
    target = _as_dtype(target, spec["dtype"])
    std = _layout_noise(spec, B, k, lambda lo, hi, n: rng.uniform(lo, hi, n))
    temps = _temps(spec["temp"], B, lambda lo, hi, n: rng.uniform(lo, hi, n))
    greedy = np.zeros(B, bool)
    n_greedy = int(round(spec["greedy_frac"] * B))
    if n_greedy:
        greedy[rng.permutation(B)[:n_greedy]] = True
        temps[greedy] = 0.0
    draft = np.empty((n_draft, width), np.float32)
    tokens = np.empty(n_draft, np.int32)
    for b in range(B):
        for i in range(int(k[b])):
            row = cu[b] + i
            noise = rng.standard_normal(width, dtype=np.float32) * np.float32(std[b, i])
            d = _as_dtype(target[cu[b] + b + i][cols] + noise, spec["dtype"])
            draft[row] = d
            if greedy[b]:
                j = int(np.argmax(d))
            else:
                g = -np.log(-np.log(rng.random(width)))
                j = int(np.argmax(d.astype(np.float64) / float(temps[b]) + g))
            tokens[row] = int(d2t[j]) if reduced else j
    out = dict(name=name, B=B, V=V, kmax=kmax, dtype=spec["dtype"], cu_drafts=cu,
               draft_logits=draft, target_logits=target, draft_tokens=tokens,
               temperature=temps.astype(np.float32))
    if reduced:
        out.update(d2t=d2t, t2d=t2d, K=len(d2t))
    return out


def _make_torch(spec, name, seed, B, V, k, cu, kmax, device):
    import torch
    dev = torch.device(device if device is not None else "cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    host = np.random.Generator(np.random.PCG64(seed))
    n_draft = int(cu[-1])
    n_target = n_draft + B
    tdt = torch.bfloat16 if spec["dtype"] == "bf16" else torch.float32
    target = torch.randn((n_target, V), generator=g, device=dev) * spec["target_std"]
    reduced = "draft_vocab" in spec
    if reduced:
        d2t, t2d = make_draft_vocab(seed, V, spec["draft_vocab"])
        d2t_dev = torch.as_tensor(d2t.astype(np.int64), device=dev)
        target[:, d2t_dev] += spec["vocab_boost"]
    width = len(d2t) if reduced else V
    target = target.to(tdt)
    std = _layout_noise(spec, B, k, lambda lo, hi, n: host.uniform(lo, hi, n))
    temps = _temps(spec["temp"], B, lambda lo, hi, n: host.uniform(lo, hi, n))
    greedy = np.zeros(B, bool)
    n_greedy = int(round(spec["greedy_frac"] * B))
    if n_greedy:
        greedy[host.permutation(B)[:n_greedy]] = True
        temps[greedy] = 0.0
    # row -> (stream, slot) maps for the draft rows
    row_b = np.repeat(np.arange(B), k)
    row_i = np.concatenate([np.arange(int(n)) for n in k]) if n_draft else np.zeros(0, int)
    trow = torch.as_tensor((cu[row_b] + row_b + row_i).astype(np.int64), device=dev)
    row_std = torch.as_tensor(std[row_b, row_i].astype(np.float32), device=dev)
    draft = torch.empty((n_draft, width), dtype=tdt, device=dev)
    tokens = torch.empty(n_draft, dtype=torch.int32, device=dev)
    row_t = torch.as_tensor(temps[row_b].astype(np.float32), device=dev)
    row_g = torch.as_tensor(greedy[row_b], device=dev)
    chunk = 64
    for r0 in range(0, n_draft, chunk):
        r1 = min(n_draft, r0 + chunk)
        noise = torch.randn((r1 - r0, width), generator=g, device=dev) * row_std[r0:r1, None]
        base = target[trow[r0:r1]].float()
        if reduced:
            base = base[:, d2t_dev]
        d = (base + noise).to(tdt)
        draft[r0:r1] = d
        u = torch.rand((r1 - r0, width), generator=g, device=dev, dtype=torch.float64)
        gum = -torch.log(-torch.log(u))
        t = row_t[r0:r1, None].double().clamp_min(1e-30)
        sampled = torch.argmax(d.double() / t + gum, dim=1)
        greedy_pick = torch.argmax(d.float(), dim=1)
        pick = torch.where(row_g[r0:r1], greedy_pick, sampled)
        if reduced:
            pick = d2t_dev[pick]
        tokens[r0:r1] = pick.to(torch.int32)
    out = dict(name=name, B=B, V=V, kmax=kmax, dtype=spec["dtype"],
               cu_drafts=torch.as_tensor(cu, device=dev),
               draft_logits=draft, target_logits=target, draft_tokens=tokens,
               temperature=torch.as_tensor(temps.astype(np.float32), device=dev))
    if reduced:
        out.update(d2t=torch.as_tensor(d2t, device=dev), t2d=torch.as_tensor(t2d, device=dev), K=len(d2t))
    return out


def make_bias_inputs(name, seed, *, rows=None, V=None, rank=None):
    """Markov-bias inputs (numpy back-end): W1 [V, R], W2 [R, V], prev [rows] int32.

    Values are N(0, 0.02^2) in the workload's dtype (returned as float32 holding exact
    values); prev is uniform in [0, V).
    """
    spec = WORKLOADS[name]
    V = spec["V"] if V is None else V
    R = spec["rank"] if rank is None else rank
    rows = spec["B"] * spec["N"] if rows is None else rows
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    w1 = _as_dtype(rng.standard_normal((V, R), dtype=np.float32) * 0.02, spec["dtype"])
    w2 = _as_dtype(rng.standard_normal((R, V), dtype=np.float32) * 0.02, spec["dtype"])
    prev = rng.integers(0, V, rows).astype(np.int32)
    return dict(W1=w1, W2=w2, prev=prev, rank=R, V=V, dtype=spec["dtype"])


def make_confidence_inputs(seed, *, B=128, kmax=5, H=7168, n_max=768):
    """Confidence-head inputs (numpy back-end): hidden [B, kmax, H] and w [H] as bf16 values
    in float32, beta = 0, verify_ms [n_max + 1] float32 with verify_ms[n] = 12 + 2.6 n
    (index 0 is unused and holds 12)."""
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    hidden = round_bf16(rng.standard_normal((B, kmax, H), dtype=np.float32))
    w = round_bf16(rng.standard_normal(H, dtype=np.float32) * 0.02)
    verify_ms = (12.0 + 2.6 * np.arange(n_max + 1)).astype(np.float32)
    return dict(hidden=hidden, w=w, beta=0.0, verify_ms=verify_ms, B=B, kmax=kmax, H=H,
                n_max=n_max)
