"""Philox4x32-10 counter-based generator and the uniforms the verify sampler draws.

Test infrastructure (see ``oracle/__init__``).

Definition (Salmon, Moraes, Dror, Shaw, SC'11, "Parallel random numbers: as easy as 1, 2, 3"):
a 4 x 32-bit counter and a 2 x 32-bit key; each of the 10 rounds multiplies counter words 0
and 2 by the two round multipliers, takes the 64-bit products apart into high and low halves,
and rebuilds the counter as (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key is bumped by the
two Weyl constants between rounds.

How the verify sampler uses it (the pages only say the sampler is "seeded", P1 §5 "What we
measured"; the layout below is this library's reading):

* key     = (seed & 0xffffffff, seed >> 32)
* counter = (slot, stream, step & 0xffffffff, step >> 32)
* output word 0 -> the acceptance uniform of draft slot ``slot``: u_slot for the token-wise
  rule, and eta_{slot+1} for block verification (the same number, so the two rules are
  coupled draw for draw);
* output word 1 -> the sampling uniform used when the step ends at ``slot`` (the correction
  token at a rejection, or the bonus token at slot N);
* output word 2 -> the draft-side uniform of slot ``slot``: the Markov walk samples the draft
  token t_slot with it (a word the verify does not use, so the two draws are independent).
* U(x) = ((x >> 8) + 0.5) * 2**-24: 24 random bits, strictly inside (0, 1), exact in float64.
"""

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF
ROUNDS = 10


def philox4x32_10(counter, key):
    """Pure-Python Philox4x32-10 of one counter (4 words) under one key (2 words)."""
    c0, c1, c2, c3 = (int(v) & MASK32 for v in counter)
    k0, k1 = (int(v) & MASK32 for v in key)
    for _ in range(ROUNDS):
        p0 = M0 * c0
        p1 = M1 * c2
        hi0, lo0 = p0 >> 32, p0 & MASK32
        hi1, lo1 = p1 >> 32, p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + W0) & MASK32
        k1 = (k1 + W1) & MASK32
    return (c0, c1, c2, c3)


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """The same function on numpy arrays (elementwise), using uint64 products.

    Every argument is broadcast to a common shape; the result is four uint32 arrays.
    """
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(
        *(np.asarray(v, dtype=np.uint64) & np.uint64(MASK32) for v in (c0, c1, c2, c3, k0, k1)))
    c0, c1, c2, c3 = c0.copy(), c1.copy(), c2.copy(), c3.copy()
    k0, k1 = k0.copy(), k1.copy()
    m32 = np.uint64(MASK32)
    sh = np.uint64(32)
    for _ in range(ROUNDS):
        p0 = np.uint64(M0) * c0
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> sh, p0 & m32
        hi1, lo1 = p1 >> sh, p1 & m32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + np.uint64(W0)) & m32
        k1 = (k1 + np.uint64(W1)) & m32
    return tuple(v.astype(np.uint32) for v in (c0, c1, c2, c3))


def uniform24(word):
    """U(x) = ((x >> 8) + 0.5) * 2^-24 in float64 (exact); works on ints and arrays."""
    if isinstance(word, np.ndarray):
        return ((word.astype(np.uint64) >> np.uint64(8)).astype(np.float64) + 0.5) * 2.0 ** -24
    return ((int(word) >> 8) + 0.5) * 2.0 ** -24


def _key(seed):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return (seed & MASK32, seed >> 32)


def _counter(step, stream, slot):
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    return (int(slot), int(stream), step & MASK32, step >> 32)


def slot_uniforms(seed, step, stream, slot):
    """(acceptance uniform, sampling uniform) of one (stream, slot) in one verify step."""
    w = philox4x32_10(_counter(step, stream, slot), _key(seed))
    return uniform24(w[0]), uniform24(w[1])


def draft_uniform(seed, step, stream, slot):
    """The draft-side uniform (word 2) of one (stream, slot) in one step."""
    return uniform24(philox4x32_10(_counter(step, stream, slot), _key(seed))[2])


def slot_uniforms_np(seed, step, stream, slot):
    """Vectorised ``slot_uniforms``: stream/slot/step may be arrays (broadcast)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    step = np.asarray(step, dtype=np.uint64)
    k0, k1 = seed & MASK32, seed >> 32
    w = philox4x32_10_np(slot, stream, step & np.uint64(MASK32), step >> np.uint64(32), k0, k1)
    return uniform24(w[0]), uniform24(w[1])
