"""spec_verify_block_static: block verification on the library's fixed device workspace.

It must give byte-identical results to spec_verify_block (which runs on a caller workspace)
on consecutive calls, refuse batches above its capacity before touching the GPU, and run
after any other test (the file is named to be collected last; the fixed workspace keeps no
state between calls that could make the order matter).
"""

import ctypes

import numpy as np
import pytest

import speculative_decoding_block_verify_gb300 as sv

SPEC_ERR_WORKSPACE = -6


def _fake_args(B, kmax):
    a = sv.VerifyArgs()
    a.B, a.V, a.kmax = B, 64, kmax
    for f in ("cu_drafts", "draft_logits", "target_logits", "draft_tokens", "temperature",
              "accepted_len", "out_tokens", "n_emitted", "status"):
        setattr(a, f, 4096)   # never dereferenced: the capacity check comes first
    return a


def test_static_workspace_capacity_is_checked_on_the_host():
    L = sv.lib()
    # 512 streams x (2 * 16 + 1) rows need 35 MB > the 16 MiB array: refused, nothing launched
    assert sv.spec_verify_workspace_bytes(512, 16) > 16 << 20
    assert L.spec_verify_block_static(ctypes.byref(_fake_args(512, 16)), None) == SPEC_ERR_WORKSPACE
    assert b"static workspace" in L.spec_last_error()
    # an oversized batch with a bad dtype or V gets spec_verify_block's code for it: the
    # argument checks come before the capacity check
    a = _fake_args(512, 16)
    a.draft_dtype = 7
    assert L.spec_verify_block_static(ctypes.byref(a), None) == -2
    a = _fake_args(512, 16)
    a.V = 0
    assert L.spec_verify_block_static(ctypes.byref(a), None) == -3
    # shape errors and empty batches take the common path's answers
    assert L.spec_verify_block_static(ctypes.byref(_fake_args(4, 33)), None) == -3
    assert L.spec_verify_block_static(ctypes.byref(_fake_args(0, 5)), None) == 0
    assert L.spec_verify_block_static(None, None) == -1


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["batch64_small", "capacity"])
def test_static_matches_caller_workspace_on_consecutive_calls(case):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_block_verify_gb300 import workloads
    from tests import parity
    if case == "batch64_small":
        inp = workloads.make_verify_inputs("batch64", 8100, B=24, V=8192)
    else:   # 208 streams x 31 rows: 15.9 MiB of workspace, just under the 16 MiB array
        inp = workloads.make_verify_inputs("batch64", 8200, B=208, N=15, V=1024)
        assert 15 << 20 < sv.spec_verify_workspace_bytes(208, 15) <= 16 << 20
    d = parity.verify_to_device(inp, torch)
    kmax = inp["kmax"]
    for step in (0, 1):   # two consecutive calls on the same fixed workspace
        ref = sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], kmax, 5, step, diag=True)
        got = sv.spec_verify_block_static(d["cu"], d["dq"], d["dp"], d["x"], d["T"], kmax, 5, step,
                                          diag=True)
        torch.cuda.synchronize()
        for k in ("accepted_len", "out_tokens", "n_emitted", "status", "diag"):
            a = ref[k].cpu().numpy()
            b = got[k].cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (case, step, k)
        assert (ref["status"].cpu().numpy() == 0).all()
        assert "workspace" not in got
