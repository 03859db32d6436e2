"""GB300-native speculative-decoding verify sampler: Python binding of libspecverify.so.

The binding only marshals arguments: it checks tensor devices, dtypes and shapes, passes raw
device pointers and the current CUDA stream to the C ABI (``include/specverify.h``) and
raises on a nonzero return code.  Every step of the method runs in the library's CUDA
kernels; there is no fallback.  PyTorch supplies device memory and streams.

Entry points (same names as the C ABI):

* ``dspark_markov_bias``     - Markov head's low-rank previous-token logit bias
* ``dspark_markov_walk``     - the bias with the draft tokens sampled slot by slot
* ``spec_verify_tokenwise``  - token-by-token speculative sampling
* ``spec_verify_block``      - block verification
* ``spec_verify_*_reduced``  - the same over a reduced draft vocabulary (top-k draft columns)
* ``adaptive_pick_k``        - confidence head + pick how many drafts to verify
* ``spec_accept_counters``   - per-position acceptance counts (a_p, tokens per step)
* ``SpecPipeline``           - pick k -> ragged verify -> counters as one CUDA graph
* ``CostCurve``              - the online verify-cost table adaptive_pick_k reads
* ``spec_philox_uniforms``   - the verify calls' uniforms (for checking)

Build the library first: ``python -m speculative_decoding_block_verify_gb300.build`` (or
``__graft_entry__.build()``).
"""

import ctypes
import os

__all__ = [
    "dspark_markov_bias", "dspark_markov_walk", "spec_verify_tokenwise", "spec_verify_block",
    "spec_verify_tokenwise_reduced", "spec_verify_block_reduced",
    "adaptive_pick_k", "spec_accept_counters", "acceptance_rates", "SpecPipeline", "CostCurve",
    "spec_philox_uniforms", "spec_verify_launch_info",
    "spec_verify_workspace_bytes", "spec_verify_block_static", "lib", "lib_path", "SpecError",
    "DTYPE_F32", "DTYPE_BF16", "STATUS_NAMES", "DIAG_COLS",
]

DTYPE_F32 = 0
DTYPE_BF16 = 1
DIAG_COLS = 8
STATUS_NAMES = {0: "OK", 1: "BAD_TEMPERATURE", 2: "BAD_TOKEN", 3: "BAD_ROW",
                4: "ZERO_DRAFT_PROB", 5: "BAD_OFFSETS", 6: "TIMEOUT", 7: "NUMERIC"}
EXPORTED = ["dspark_markov_bias", "dspark_markov_walk", "dspark_markov_walk_workspace_bytes",
            "spec_verify_tokenwise", "spec_verify_block",
            "spec_verify_tokenwise_reduced", "spec_verify_block_reduced",
            "adaptive_pick_k", "spec_philox_uniforms", "spec_verify_launch_info",
            "spec_verify_workspace_bytes", "spec_verify_block_static",
            "spec_accept_counters", "spec_pipeline_create", "spec_pipeline_launch",
            "spec_pipeline_destroy", "spec_cost_curve_create", "spec_cost_curve_begin",
            "spec_cost_curve_end", "spec_cost_curve_poll", "spec_cost_curve_observe",
            "spec_cost_curve_table", "spec_cost_curve_upload", "spec_cost_curve_destroy",
            "spec_last_error", "spec_version"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


class SpecError(RuntimeError):
    """A nonzero return code from the C ABI."""

    def __init__(self, code, msg):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class VerifyArgs(ctypes.Structure):
    """Mirror of spec_verify_args."""
    _fields_ = [
        ("B", ctypes.c_int32), ("V", ctypes.c_int32), ("kmax", ctypes.c_int32),
        ("cu_drafts", ctypes.c_void_p),
        ("draft_logits", ctypes.c_void_p), ("draft_dtype", ctypes.c_int32),
        ("target_logits", ctypes.c_void_p), ("target_dtype", ctypes.c_int32),
        ("draft_tokens", ctypes.c_void_p), ("temperature", ctypes.c_void_p),
        ("seed", ctypes.c_uint64), ("step", ctypes.c_uint64),
        ("accepted_len", ctypes.c_void_p), ("out_tokens", ctypes.c_void_p),
        ("n_emitted", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("diag", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class PipelineArgs(ctypes.Structure):
    """Mirror of spec_pipeline_args."""
    _fields_ = [
        ("hidden", ctypes.c_void_p), ("w", ctypes.c_void_p), ("head_dtype", ctypes.c_int32),
        ("bias", ctypes.c_float), ("H", ctypes.c_int32), ("verify_ms", ctypes.c_void_p),
        ("n_max", ctypes.c_int32), ("mode", ctypes.c_int32),
        ("rule", ctypes.c_int32), ("B", ctypes.c_int32), ("V", ctypes.c_int32), ("kmax", ctypes.c_int32),
        ("draft_logits", ctypes.c_void_p), ("draft_dtype", ctypes.c_int32),
        ("target_logits", ctypes.c_void_p), ("target_dtype", ctypes.c_int32),
        ("draft_tokens", ctypes.c_void_p), ("temperature", ctypes.c_void_p),
        ("seed", ctypes.c_uint64), ("step", ctypes.c_void_p),
        ("c_out", ctypes.c_void_p), ("a_out", ctypes.c_void_p), ("k_out", ctypes.c_void_p),
        ("cu_drafts_out", ctypes.c_void_p), ("accepted_len", ctypes.c_void_p),
        ("out_tokens", ctypes.c_void_p), ("n_emitted", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("diag", ctypes.c_void_p), ("accept_counts", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


def lib_path():
    return os.path.join(_HERE, "_build", "libspecverify.so")


def lib():
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m speculative_decoding_block_verify_gb300.build`")
    L = ctypes.CDLL(path)
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64
    L.dspark_markov_bias.argtypes = [vp, i32, i32, i32, vp, vp, vp, i32, i32, vp, vp]
    L.dspark_markov_walk.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, i32, i32, vp, u64, u64, vp, vp, vp, vp,
                                     ctypes.c_size_t, vp]
    L.dspark_markov_walk_workspace_bytes.argtypes = [i32]
    L.dspark_markov_walk_workspace_bytes.restype = ctypes.c_size_t
    L.spec_verify_tokenwise.argtypes = [ctypes.POINTER(VerifyArgs), vp]
    L.spec_verify_block.argtypes = [ctypes.POINTER(VerifyArgs), vp]
    L.spec_verify_block_static.argtypes = [ctypes.POINTER(VerifyArgs), vp]
    L.spec_verify_tokenwise_reduced.argtypes = [ctypes.POINTER(VerifyArgs), vp, i32, vp]
    L.spec_verify_block_reduced.argtypes = [ctypes.POINTER(VerifyArgs), vp, i32, vp]
    L.adaptive_pick_k.argtypes = [vp, vp, i32, ctypes.c_float, i32, i32, i32, vp, i32, i32,
                                  vp, vp, vp, vp, vp]
    L.spec_philox_uniforms.argtypes = [u64, u64, i32, i32, vp, vp]
    L.spec_verify_launch_info.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.POINTER(i32),
                                          ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.spec_accept_counters.argtypes = [vp, vp, vp, i32, i32, vp, vp]
    L.spec_pipeline_create.argtypes = [ctypes.POINTER(PipelineArgs), ctypes.POINTER(vp)]
    L.spec_pipeline_launch.argtypes = [vp, vp]
    L.spec_pipeline_destroy.argtypes = [vp]
    L.spec_cost_curve_create.argtypes = [vp, i32, i32, i32, i32]
    L.spec_cost_curve_create.restype = vp
    L.spec_cost_curve_begin.argtypes = [vp, vp]
    L.spec_cost_curve_end.argtypes = [vp, i32, vp, vp]
    L.spec_cost_curve_poll.argtypes = [vp]
    L.spec_cost_curve_observe.argtypes = [vp, i32, ctypes.c_float]
    L.spec_cost_curve_table.argtypes = [vp, vp, vp]
    L.spec_cost_curve_upload.argtypes = [vp, vp, vp]
    L.spec_cost_curve_destroy.argtypes = [vp]
    L.spec_cost_curve_destroy.restype = None
    L.spec_verify_workspace_bytes.argtypes = [i32, i32]
    L.spec_verify_workspace_bytes.restype = ctypes.c_size_t
    L.spec_last_error.restype = ctypes.c_char_p
    L.spec_version.restype = ctypes.c_int32
    for name in ("dspark_markov_bias", "dspark_markov_walk", "spec_verify_tokenwise", "spec_verify_block", "spec_verify_block_static",
                 "spec_verify_tokenwise_reduced", "spec_verify_block_reduced",
                 "adaptive_pick_k", "spec_philox_uniforms", "spec_verify_launch_info",
                 "spec_accept_counters", "spec_pipeline_create", "spec_pipeline_launch",
                 "spec_pipeline_destroy", "spec_cost_curve_begin", "spec_cost_curve_end",
                 "spec_cost_curve_poll", "spec_cost_curve_observe", "spec_cost_curve_table",
                 "spec_cost_curve_upload"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(rc):
    if rc != 0:
        raise SpecError(rc, lib().spec_last_error().decode())


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def dspark_markov_bias(draft_logits, prev_tokens, W1, W2, out=None, stream=None):
    """out[r, v] = draft[r, v] + sum_j W1[prev[r], j] W2[j, v] (float32 output).

    draft_logits [rows, V] float32/bf16, prev_tokens [rows] int32, W1 [V, R], W2 [R, V]
    (same dtype).  ``out`` may be ``draft_logits`` itself when that is float32.
    """
    torch = _torch()
    _dev(draft_logits, "draft_logits")
    _dev(prev_tokens, "prev_tokens", torch.int32)
    _dev(W1, "W1")
    _dev(W2, "W2")
    rows, V = draft_logits.shape
    R = W2.shape[0]
    if W1.dtype != W2.dtype or tuple(W1.shape) != (V, R) or tuple(W2.shape) != (R, V):
        raise ValueError("W1 must be [V, R] and W2 [R, V] with one dtype")
    if prev_tokens.shape != (rows,):
        raise ValueError("prev_tokens must be [rows]")
    if out is None:
        out = torch.empty((rows, V), dtype=torch.float32, device=draft_logits.device)
    _dev(out, "out", torch.float32)
    _check(lib().dspark_markov_bias(_ptr(draft_logits), _dtype_code(draft_logits), rows, V,
                                    _ptr(prev_tokens), _ptr(W1), _ptr(W2), _dtype_code(W1), R,
                                    _ptr(out), _stream(stream)))
    return out


def dspark_markov_walk(draft_logits, anchor, W1, W2, temperature, seed, step, out=None, stream=None):
    """The Markov walk: draft_logits [B, N, V] (float32/bf16), anchor [B] int32, W1 [V, R], W2
    [R, V] (one dtype), temperature [B] float32.  Returns (and reuses) ``out`` with tokens
    [B, N] int32, logits [B, N, V] float32 (the biased rows), status [B] int32, workspace."""
    torch = _torch()
    _dev(draft_logits, "draft_logits")
    _dev(anchor, "anchor", torch.int32)
    _dev(W1, "W1")
    _dev(W2, "W2")
    _dev(temperature, "temperature", torch.float32)
    B, N, V = draft_logits.shape
    R = W2.shape[0]
    if W1.dtype != W2.dtype or tuple(W1.shape) != (V, R) or tuple(W2.shape) != (R, V):
        raise ValueError("W1 must be [V, R] and W2 [R, V] with one dtype")
    if anchor.shape != (B,) or temperature.shape != (B,):
        raise ValueError("anchor and temperature must be [B]")
    dev = draft_logits.device
    if out is None:
        out = {"tokens": torch.empty((B, N), dtype=torch.int32, device=dev),
               "logits": torch.empty((B, N, V), dtype=torch.float32, device=dev),
               "status": torch.empty(B, dtype=torch.int32, device=dev),
               "workspace": torch.empty(max(int(lib().dspark_markov_walk_workspace_bytes(B)), 16),
                                        dtype=torch.uint8, device=dev)}
    _check(lib().dspark_markov_walk(_ptr(draft_logits), _dtype_code(draft_logits), B, N, V, _ptr(anchor),
                                    _ptr(W1), _ptr(W2), _dtype_code(W1), R, _ptr(temperature),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF,
                                    _ptr(out["tokens"]), _ptr(out["logits"]), _ptr(out["status"]),
                                    _ptr(out["workspace"]), out["workspace"].numel(), _stream(stream)))
    return out


def _verify(fn, cu_drafts, draft_logits, target_logits, draft_tokens, temperature, kmax, seed,
            step, out=None, diag=False, stream=None, workspace=True, t2d=None):
    """Marshals one verify call.  ``out`` (returned, and reusable by later calls of the same B
    and kmax on the same stream) holds the four result tensors and the device workspace; a
    workspace the caller puts in ``out["workspace"]`` must have been zero-filled before its
    first use (the one allocated here is), since the kernels keep per-row counters there that
    every call leaves at zero."""
    torch = _torch()
    _dev(cu_drafts, "cu_drafts", torch.int32)
    _dev(target_logits, "target_logits")
    _dev(draft_logits, "draft_logits")
    _dev(draft_tokens, "draft_tokens", torch.int32)
    _dev(temperature, "temperature", torch.float32)
    B = cu_drafts.numel() - 1
    V = target_logits.shape[1]
    if t2d is not None:
        _dev(t2d, "t2d", torch.int32)
        if t2d.numel() != V:
            raise ValueError("t2d must be [V]")
        if draft_logits.dim() != 2:
            raise ValueError("draft_logits must be [rows, K]")
    elif draft_logits.dim() != 2 or (draft_logits.shape[0] > 0 and draft_logits.shape[1] != V):
        raise ValueError("draft_logits must be [rows, V]")
    if temperature.numel() != B:
        raise ValueError("temperature must be [B]")
    dev = target_logits.device
    if out is None:
        out = {
            "accepted_len": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, kmax + 1), dtype=torch.int32, device=dev),
            "n_emitted": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
        if diag:
            out["diag"] = torch.empty((target_logits.shape[0], DIAG_COLS), dtype=torch.float32,
                                      device=dev)
    ws = None
    if workspace:
        need = spec_verify_workspace_bytes(B, kmax)
        ws = out.get("workspace")
        if ws is None or ws.numel() < need:
            # zero-filled once: every call leaves the row counters it used at zero
            ws = out["workspace"] = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
    a = VerifyArgs()
    a.B, a.V, a.kmax = B, V, kmax
    a.cu_drafts = cu_drafts.data_ptr()
    a.draft_logits = draft_logits.data_ptr() if draft_logits.numel() else None
    a.draft_dtype = _dtype_code(draft_logits)
    a.target_logits = target_logits.data_ptr()
    a.target_dtype = _dtype_code(target_logits)
    a.draft_tokens = draft_tokens.data_ptr() if draft_tokens.numel() else None
    a.temperature = temperature.data_ptr()
    a.seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    a.step = int(step) & 0xFFFFFFFFFFFFFFFF
    a.accepted_len = out["accepted_len"].data_ptr()
    a.out_tokens = out["out_tokens"].data_ptr()
    a.n_emitted = out["n_emitted"].data_ptr()
    a.status = out["status"].data_ptr()
    a.diag = out["diag"].data_ptr() if out.get("diag") is not None else None
    a.workspace = ws.data_ptr() if ws is not None else None
    a.workspace_bytes = ws.numel() if ws is not None else 0
    if t2d is not None:
        _check(fn(ctypes.byref(a), _ptr(t2d), int(draft_logits.shape[1]), _stream(stream)))
    else:
        _check(fn(ctypes.byref(a), _stream(stream)))
    return out


def spec_verify_tokenwise(cu_drafts, draft_logits, target_logits, draft_tokens, temperature,
                          kmax, seed, step, out=None, diag=False, stream=None):
    """Token-by-token speculative sampling (see include/specverify.h)."""
    return _verify(lib().spec_verify_tokenwise, cu_drafts, draft_logits, target_logits,
                   draft_tokens, temperature, kmax, seed, step, out, diag, stream)


def spec_verify_block(cu_drafts, draft_logits, target_logits, draft_tokens, temperature, kmax,
                      seed, step, out=None, diag=False, stream=None):
    """Block verification (see include/specverify.h)."""
    return _verify(lib().spec_verify_block, cu_drafts, draft_logits, target_logits,
                   draft_tokens, temperature, kmax, seed, step, out, diag, stream)


def spec_verify_tokenwise_reduced(cu_drafts, draft_logits, t2d, target_logits, draft_tokens, temperature,
                                  kmax, seed, step, out=None, diag=False, stream=None):
    """Token-wise verify with draft rows over a reduced draft vocabulary: draft_logits [rows, K],
    t2d [V] int32 (the draft id of each target column, -1 outside the draft vocabulary)."""
    return _verify(lib().spec_verify_tokenwise_reduced, cu_drafts, draft_logits, target_logits,
                   draft_tokens, temperature, kmax, seed, step, out, diag, stream, t2d=t2d)


def spec_verify_block_reduced(cu_drafts, draft_logits, t2d, target_logits, draft_tokens, temperature, kmax,
                              seed, step, out=None, diag=False, stream=None):
    """Block verification with draft rows over a reduced draft vocabulary (see
    spec_verify_tokenwise_reduced)."""
    return _verify(lib().spec_verify_block_reduced, cu_drafts, draft_logits, target_logits,
                   draft_tokens, temperature, kmax, seed, step, out, diag, stream, t2d=t2d)


def spec_verify_block_static(cu_drafts, draft_logits, target_logits, draft_tokens, temperature,
                             kmax, seed, step, out=None, diag=False, stream=None):
    """Block verification on the library's fixed device workspace: no workspace is allocated
    or passed (see include/specverify.h for its capacity and ordering rule)."""
    return _verify(lib().spec_verify_block_static, cu_drafts, draft_logits, target_logits,
                   draft_tokens, temperature, kmax, seed, step, out, diag, stream, workspace=False)


def adaptive_pick_k(hidden, w, bias, verify_ms, mode=0, out=None, stream=None):
    """Confidence head + pick k.  hidden [B, kmax, H], w [H] (float32/bf16, same dtype),
    verify_ms [n_max + 1] float32.  Returns dict c [B, kmax], a [B, kmax], k [B], cu [B+1]."""
    torch = _torch()
    _dev(hidden, "hidden")
    _dev(w, "w")
    _dev(verify_ms, "verify_ms", torch.float32)
    if w.dtype != hidden.dtype:
        raise TypeError("hidden and w must share a dtype")
    B, kmax, H = hidden.shape
    if w.shape != (H,):
        raise ValueError("w must be [H]")
    dev = hidden.device
    if out is None:
        out = {"c": torch.empty((B, kmax), dtype=torch.float32, device=dev),
               "a": torch.empty((B, kmax), dtype=torch.float32, device=dev),
               "k": torch.empty(B, dtype=torch.int32, device=dev),
               "cu": torch.empty(B + 1, dtype=torch.int32, device=dev)}
    _check(lib().adaptive_pick_k(_ptr(hidden), _ptr(w), _dtype_code(hidden), float(bias), B, kmax,
                                 H, _ptr(verify_ms), verify_ms.numel() - 1, int(mode),
                                 _ptr(out["c"]), _ptr(out["a"]), _ptr(out["k"]), _ptr(out["cu"]),
                                 _stream(stream)))
    return out


def spec_accept_counters(accepted_len, status, cu_drafts, kmax, counts=None, stream=None):
    """Adds one batch's per-position acceptance counts to ``counts`` [2 kmax + 1] (uint64 as
    int64, device; allocated zeroed when None) and returns it: counts[0] = verified streams,
    counts[p] = accepted at position p, counts[kmax + p] = offered at position p."""
    torch = _torch()
    _dev(accepted_len, "accepted_len", torch.int32)
    _dev(status, "status", torch.int32)
    _dev(cu_drafts, "cu_drafts", torch.int32)
    B = status.numel()
    if counts is None:
        counts = torch.zeros(2 * kmax + 1, dtype=torch.int64, device=status.device)
    _dev(counts, "counts", torch.int64)
    if counts.numel() != 2 * kmax + 1:
        raise ValueError("counts must have 2 kmax + 1 entries")
    _check(lib().spec_accept_counters(_ptr(accepted_len), _ptr(status), _ptr(cu_drafts), B, kmax,
                                      _ptr(counts), _stream(stream)))
    return counts


def acceptance_rates(counts, kmax):
    """(a_p for p = 1..kmax, marginal a_p / a_{p-1}, tokens per step = 1 + sum a_p) from the
    accumulated counts (P1 §6 "The arithmetic you need before tuning k")."""
    c = [int(v) for v in counts.cpu().tolist()]
    steps = max(c[0], 1)
    a = [c[p] / steps for p in range(1, kmax + 1)]
    marg = [a[0]] + [(a[p] / a[p - 1]) if a[p - 1] > 0 else 0.0 for p in range(1, kmax)]
    return a, marg, 1.0 + sum(a)


class SpecPipeline:
    """pick k -> verify each stream's first k_b drafts -> acceptance counters -> step + 1, as
    one CUDA graph (spec_pipeline_create / launch / destroy).  Inputs are the dense layout:
    draft_logits [B, kmax, V], target_logits [B, kmax + 1, V], draft_tokens [B, kmax]; the
    confidence head's hidden [B, kmax, H], w [H] and verify_ms [n_max + 1].  ``step`` is the
    first launch's Philox step; each launch adds 1.  The outputs (``out`` dict) and the
    counters are device tensors that every launch overwrites (counters accumulate)."""

    def __init__(self, hidden, w, bias, verify_ms, draft_logits, target_logits, draft_tokens,
                 temperature, rule=1, mode=0, seed=0, step=0, diag=False, counters=True):
        torch = _torch()
        for t, n in ((hidden, "hidden"), (w, "w"), (draft_logits, "draft_logits"),
                     (target_logits, "target_logits")):
            _dev(t, n)
        _dev(verify_ms, "verify_ms", torch.float32)
        _dev(draft_tokens, "draft_tokens", torch.int32)
        _dev(temperature, "temperature", torch.float32)
        B, kmax, V = draft_logits.shape
        if tuple(target_logits.shape) != (B, kmax + 1, V) or tuple(draft_tokens.shape) != (B, kmax):
            raise ValueError("target_logits must be [B, kmax + 1, V] and draft_tokens [B, kmax]")
        if hidden.shape[:2] != (B, kmax) or w.shape != (hidden.shape[2],) or w.dtype != hidden.dtype:
            raise ValueError("hidden must be [B, kmax, H] and w [H] of hidden's dtype")
        dev = draft_logits.device
        self.kmax = kmax
        self.out = {
            "c": torch.empty((B, kmax), dtype=torch.float32, device=dev),
            "a": torch.empty((B, kmax), dtype=torch.float32, device=dev),
            "k": torch.empty(B, dtype=torch.int32, device=dev),
            "cu": torch.empty(B + 1, dtype=torch.int32, device=dev),
            "accepted_len": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, kmax + 1), dtype=torch.int32, device=dev),
            "n_emitted": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
        if diag:
            self.out["diag"] = torch.empty((B * (kmax + 1), DIAG_COLS), dtype=torch.float32, device=dev)
        self.counts = torch.zeros(2 * kmax + 1, dtype=torch.int64, device=dev) if counters else None
        self.step = torch.tensor([int(step)], dtype=torch.int64, device=dev)
        self.workspace = torch.zeros(max(spec_verify_workspace_bytes(B, kmax), 16), dtype=torch.uint8,
                                     device=dev)
        self._keep = (hidden, w, verify_ms, draft_logits, target_logits, draft_tokens, temperature)
        a = PipelineArgs()
        a.hidden, a.w, a.head_dtype = hidden.data_ptr(), w.data_ptr(), _dtype_code(hidden)
        a.bias, a.H, a.verify_ms, a.n_max, a.mode = float(bias), hidden.shape[2], verify_ms.data_ptr(), \
            verify_ms.numel() - 1, int(mode)
        a.rule, a.B, a.V, a.kmax = int(rule), B, V, kmax
        a.draft_logits, a.draft_dtype = draft_logits.data_ptr(), _dtype_code(draft_logits)
        a.target_logits, a.target_dtype = target_logits.data_ptr(), _dtype_code(target_logits)
        a.draft_tokens, a.temperature = draft_tokens.data_ptr(), temperature.data_ptr()
        a.seed, a.step = int(seed) & 0xFFFFFFFFFFFFFFFF, self.step.data_ptr()
        o = self.out
        a.c_out, a.a_out, a.k_out, a.cu_drafts_out = (o[k].data_ptr() for k in ("c", "a", "k", "cu"))
        a.accepted_len, a.out_tokens, a.n_emitted, a.status = (
            o[k].data_ptr() for k in ("accepted_len", "out_tokens", "n_emitted", "status"))
        a.diag = o["diag"].data_ptr() if diag else None
        a.accept_counts = self.counts.data_ptr() if counters else None
        a.workspace, a.workspace_bytes = self.workspace.data_ptr(), self.workspace.numel()
        self._handle = ctypes.c_void_p()
        _check(lib().spec_pipeline_create(ctypes.byref(a), ctypes.byref(self._handle)))

    def launch(self, stream=None):
        """One verify step (one graph launch on the current or given stream)."""
        _check(lib().spec_pipeline_launch(self._handle, _stream(stream)))
        return self.out

    def close(self):
        if self._handle:
            _check(lib().spec_pipeline_destroy(self._handle))
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CostCurve:
    """The online verify-cost curve (P3 "Teaching the Speculator What a Draft Costs", "What we
    changed" and "Reproduce"): CUDA-event pairs around real verify steps, read without waiting,
    rolling medians per token count laid over the boot curve every ``rebuild_every``
    observations.  ``boot_ms`` is a host sequence of n_max + 1 floats (index = token count).

    ``begin()`` / ``end(num_tokens, device_count=None)`` bracket one verify step on the current
    (or given) stream; a ``device_count`` int32 CUDA tensor (one element) adds its value to the
    count after the step.  ``poll()`` folds in finished steps, ``table()`` returns the current
    table (a list) and ``upload(device_table)`` queues its copy into a float32 CUDA tensor."""

    def __init__(self, boot_ms, window=32, min_samples=3, rebuild_every=32):
        boot = (ctypes.c_float * len(boot_ms))(*[float(v) for v in boot_ms])
        self.n_max = len(boot_ms) - 1
        self._handle = lib().spec_cost_curve_create(boot, self.n_max, int(window), int(min_samples),
                                                     int(rebuild_every))
        if not self._handle:
            raise SpecError(-1, lib().spec_last_error().decode())

    def begin(self, stream=None):
        _check(lib().spec_cost_curve_begin(self._handle, _stream(stream)))

    def end(self, num_tokens=0, device_count=None, stream=None):
        if device_count is not None:
            _dev(device_count, "device_count", _torch().int32)
        _check(lib().spec_cost_curve_end(self._handle, int(num_tokens), _ptr(device_count), _stream(stream)))

    def poll(self):
        _check(lib().spec_cost_curve_poll(self._handle))

    def observe(self, num_tokens, ms):
        _check(lib().spec_cost_curve_observe(self._handle, int(num_tokens), float(ms)))

    def table(self):
        """(table as a list of n_max + 1 floats, {observations, rebuilds, dropped, pending})."""
        out = (ctypes.c_float * (self.n_max + 1))()
        cnt = (ctypes.c_int64 * 4)()
        _check(lib().spec_cost_curve_table(self._handle, out, cnt))
        return list(out), dict(zip(("observations", "rebuilds", "dropped", "pending"), list(cnt)))

    def upload(self, device_table, stream=None):
        _dev(device_table, "device_table", _torch().float32)
        if device_table.numel() != self.n_max + 1:
            raise ValueError("device_table must hold n_max + 1 floats")
        _check(lib().spec_cost_curve_upload(self._handle, _ptr(device_table), _stream(stream)))

    def close(self):
        if self._handle:
            lib().spec_cost_curve_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spec_verify_workspace_bytes(B, kmax):
    """Device workspace bytes a verify call over B streams with up to kmax drafts needs."""
    return int(lib().spec_verify_workspace_bytes(int(B), int(kmax)))


def spec_verify_launch_info(B, V, kmax, draft_dtype=DTYPE_BF16, target_dtype=DTYPE_BF16,
                            aligned=True):
    """(cluster_size, resident_clusters, elems_per_load) a verify call of this shape uses."""
    a = VerifyArgs()
    a.B, a.V, a.kmax = B, V, kmax
    a.draft_dtype, a.target_dtype = draft_dtype, target_dtype
    a.draft_logits = a.target_logits = 0 if aligned else 2
    c, r, e = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().spec_verify_launch_info(ctypes.byref(a), ctypes.byref(c), ctypes.byref(r),
                                         ctypes.byref(e)))
    return c.value, r.value, e.value


def spec_philox_uniforms(seed, step, n_streams, n_slots, device="cuda", stream=None):
    """[n_streams, n_slots, 2] float64: (acceptance, sampling) uniforms of every (stream, slot)."""
    torch = _torch()
    out = torch.empty((n_streams, n_slots, 2), dtype=torch.float64, device=device)
    _check(lib().spec_philox_uniforms(int(seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF,
                                      n_streams, n_slots, _ptr(out), _stream(stream)))
    return out
