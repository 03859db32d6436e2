"""Pins of the oracle's Philox4x32-10 and its uniforms (CPU only)."""

import json
import os

import numpy as np

from oracle import philox


def _kat(golden_dir):
    with open(os.path.join(golden_dir, "philox_kat.json")) as f:
        return json.load(f)["vectors"]


def test_known_answer_vectors_pure_python(golden_dir):
    for v in _kat(golden_dir):
        ctr = [int(w, 16) for w in v["counter"]]
        key = [int(w, 16) for w in v["key"]]
        out = philox.philox4x32_10(ctr, key)
        assert [f"{w:08x}" for w in out] == v["output"]


def test_known_answer_vectors_numpy(golden_dir):
    vs = _kat(golden_dir)
    cols = [np.array([int(v["counter"][i], 16) for v in vs], np.uint64) for i in range(4)]
    keys = [np.array([int(v["key"][i], 16) for v in vs], np.uint64) for i in range(2)]
    out = philox.philox4x32_10_np(*cols, *keys)
    for j, v in enumerate(vs):
        assert [f"{int(out[i][j]):08x}" for i in range(4)] == v["output"]


def test_numpy_matches_pure_python_on_random_counters():
    rng = np.random.default_rng(3)
    c = rng.integers(0, 2 ** 32, size=(4, 200), dtype=np.uint64)
    k = rng.integers(0, 2 ** 32, size=(2, 200), dtype=np.uint64)
    out = philox.philox4x32_10_np(*c, *k)
    for j in range(200):
        ref = philox.philox4x32_10([int(c[i, j]) for i in range(4)], [int(k[i, j]) for i in range(2)])
        assert tuple(int(out[i][j]) for i in range(4)) == ref


def test_uniform_range_and_exactness():
    assert philox.uniform24(0) == 2.0 ** -25
    assert philox.uniform24(0xFFFFFFFF) == 1.0 - 2.0 ** -25
    for w in (0, 1, 255, 256, 0x12345678, 0xFFFFFF00, 0xFFFFFFFF):
        u = philox.uniform24(w)
        assert 0.0 < u < 1.0
        scaled = u * 2.0 ** 25
        assert scaled == int(scaled) and int(scaled) % 2 == 1   # exact odd multiple of 2^-25
    words = np.array([0, 1, 0xFFFFFFFF, 0x80000000], np.uint32)
    assert np.array_equal(philox.uniform24(words), [philox.uniform24(int(w)) for w in words])


def test_slot_uniform_layout():
    seed, step, stream, slot = 0x0123456789ABCDEF, 0x1122334455667788, 17, 3
    out = philox.philox4x32_10([slot, stream, step & 0xFFFFFFFF, step >> 32],
                               [seed & 0xFFFFFFFF, seed >> 32])
    ua, us = philox.slot_uniforms(seed, step, stream, slot)
    assert ua == philox.uniform24(out[0]) and us == philox.uniform24(out[1])
    va, vs = philox.slot_uniforms_np(seed, np.array([step], np.uint64), np.array([stream]),
                                     np.array([slot]))
    assert va[0] == ua and vs[0] == us


def test_uniforms_look_uniform():
    # 2^16 acceptance uniforms of consecutive slots: mean, variance and a coarse histogram
    slots = np.arange(1 << 16)
    u, s = philox.slot_uniforms_np(0, 0, 0, slots)
    for x in (u, s):
        assert abs(x.mean() - 0.5) < 0.01
        assert abs(x.var() - 1 / 12) < 0.005
        hist = np.histogram(x, bins=16, range=(0, 1))[0]
        assert hist.min() > 0.9 * len(x) / 16 and hist.max() < 1.1 * len(x) / 16
