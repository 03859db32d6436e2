"""The C-ABI library builds, loads and exports every symbol include/*.h declares; host-side
argument checks return their codes before any CUDA call (CPU only, no GPU needed)."""

import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_block_verify_gb300 as sv
from speculative_decoding_block_verify_gb300 import build as svbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    svbuild.build()
    return sv.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dspark_markov_bias", "spec_verify_tokenwise", "spec_verify_block",
              "adaptive_pick_k", "spec_philox_uniforms", "spec_last_error", "spec_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    assert set(sv.EXPORTED) <= declared_functions()
    assert L.spec_version() == 1


def test_host_argument_errors_before_any_launch(L):
    vp = ctypes.c_void_p
    assert L.spec_verify_block(None, None) == -1
    assert b"NULL" in L.spec_last_error()
    a = sv.VerifyArgs()
    a.B, a.V, a.kmax = 2, 0, 5
    assert L.spec_verify_tokenwise(ctypes.byref(a), None) == -3
    a.V, a.kmax = 16, 33
    assert L.spec_verify_block(ctypes.byref(a), None) == -3
    a.kmax, a.draft_dtype = 5, 7
    assert L.spec_verify_block(ctypes.byref(a), None) == -2
    a.draft_dtype = 1
    assert L.spec_verify_block(ctypes.byref(a), None) == -1      # NULL pointers
    a.B = 0
    assert L.spec_verify_block(ctypes.byref(a), None) == 0       # nothing to do
    assert L.spec_last_error() == b""
    assert L.dspark_markov_bias(vp(0), 1, 0, 16, vp(0), vp(0), vp(0), 1, 8, vp(0), vp(0)) == 0
    assert L.dspark_markov_bias(vp(0), 1, 4, 16, vp(0), vp(0), vp(0), 1, 2000, vp(0), vp(0)) == -3
    assert L.dspark_markov_bias(vp(0), 3, 4, 16, vp(0), vp(0), vp(0), 1, 8, vp(0), vp(0)) == -2
    assert L.dspark_markov_bias(vp(0), 1, 4, 16, vp(0), vp(0), vp(0), 1, 8, vp(0), vp(0)) == -1
    assert L.adaptive_pick_k(vp(0), vp(0), 1, ctypes.c_float(0), 4, 5, 64, vp(0), 768, 2,
                             vp(0), vp(0), vp(0), vp(0), vp(0)) == -1
    assert L.adaptive_pick_k(vp(0), vp(0), 1, ctypes.c_float(0), 4, 5, 64, vp(0), 5, 0,
                             vp(0), vp(0), vp(0), vp(0), vp(0)) == -3
    assert L.adaptive_pick_k(vp(0), vp(0), 1, ctypes.c_float(0), 2000, 5, 64, vp(0), 20000, 1,
                             vp(0), vp(0), vp(0), vp(0), vp(0)) == -3
    assert L.spec_philox_uniforms(0, 0, -1, 4, vp(0), vp(0)) == -3
    assert L.spec_philox_uniforms(0, 0, 0, 4, vp(0), vp(0)) == 0


def test_verify_args_layout_matches_the_header():
    # field order and natural alignment of spec_verify_args on an LP64 ABI
    offs = {f[0]: getattr(sv.VerifyArgs, f[0]).offset for f in sv.VerifyArgs._fields_}
    assert offs["cu_drafts"] == 16 and offs["draft_logits"] == 24 and offs["draft_dtype"] == 32
    assert offs["target_logits"] == 40 and offs["seed"] == 72 and offs["diag"] == 120
    assert offs["workspace"] == 128 and offs["workspace_bytes"] == 136
    assert ctypes.sizeof(sv.VerifyArgs) == 144


def test_workspace_size_and_check(L):
    # one 16-byte partial per (row, stats segment <= 64); a stream has <= 2 kmax + 1 rows
    # one block per row: a 16-byte counter slot and 64 partials of 16 bytes
    # a 256-byte header, a 1536-byte block per stats row (at the same offset for every B and
    # kmax), then the residual sweep's work list: 32 bytes per claim, one claim per segment
    # (64 per slot)
    assert sv.spec_verify_workspace_bytes(64, 5) == 256 + 64 * 11 * 1536 + 64 * 6 * 64 * 32
    for B, kmax in ((1, 0), (7, 3), (256, 15), (3, 32)):
        assert sv.spec_verify_workspace_bytes(B, kmax) == 256 + B * (2 * kmax + 1) * 1536 + B * (kmax + 1) * 2048
    assert sv.spec_verify_workspace_bytes(0, 5) == 0
    assert sv.spec_verify_workspace_bytes(-1, 5) == 0
    assert sv.spec_verify_workspace_bytes(4, 33) == 0
    a = sv.VerifyArgs()
    a.B, a.V, a.kmax = 2, 16, 3
    for f in ("cu_drafts", "draft_logits", "target_logits", "draft_tokens", "temperature",
              "accepted_len", "out_tokens", "n_emitted", "status"):
        setattr(a, f, 4096)                     # never dereferenced: the check comes first
    assert L.spec_verify_block(ctypes.byref(a), None) == -6
    assert b"workspace" in L.spec_last_error()
    a.workspace, a.workspace_bytes = 4096, sv.spec_verify_workspace_bytes(2, 3) - 1
    assert L.spec_verify_tokenwise(ctypes.byref(a), None) == -6
    a.workspace, a.workspace_bytes = 4104, 1 << 20   # not 16-byte aligned
    assert L.spec_verify_block(ctypes.byref(a), None) == -6


def test_walk_workspace_size_and_check(L):
    # the barrier counter and timeout flag (256 bytes), then every CTA's 16-byte partial per
    # stream (up to 2048 CTAs) in two buffers that alternate from slot to slot
    for B in (1, 4, 33):
        assert L.dspark_markov_walk_workspace_bytes(B) == 256 + 2 * B * 2048 * 16
    assert L.dspark_markov_walk_workspace_bytes(-1) == 0
    vp = ctypes.c_void_p
    p = vp(4096)   # never dereferenced: the workspace check comes before any launch
    need = L.dspark_markov_walk_workspace_bytes(2)
    args = (p, 1, 2, 5, 1024, p, p, p, 1, 256, p, 0, 0, p, p, p)
    assert L.dspark_markov_walk(*args, vp(4096), need - 1, vp(0)) == -6
    assert b"workspace" in L.spec_last_error()
    assert L.dspark_markov_walk(*args, vp(4104), need, vp(0)) == -6   # not 16-byte aligned
    assert L.dspark_markov_walk(*args, None, need, vp(0)) == -6
