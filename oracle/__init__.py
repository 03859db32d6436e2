"""Oracle: a plain, slow, float64 CPU restatement of the speculative-decoding verify sampler.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The product path
(the CUDA library and its Python binding) never imports, links or executes anything here, and
nothing here imports the product package.  The two share no code: the only common module is
the seeded input generator, which holds none of the method's arithmetic.

Sources (the pages are cited by title and section):

* "MTP, DSpark and Block Verification, Explained: Six Tokens per Step" (al-engr.com),
  §3 "DSpark: draft a block, then fix it" (Markov fix-up), §4 "Verification: the guarantee"
  (token-by-token rule, block verification, greedy code path), §6 "Why five beat nine"
  (tokens/step = 1 + sum of per-position accept rates).
* "MTP Heads and Confidence Heads: Linking Three Self-Drafting Routes into One Chain"
  (naphjohn.github.io), §6 (Markov head B = W1 @ W2, rank 256), §7-§9 (confidence head,
  prefix survival), figure text after §9 (scheduler adds candidates in descending a_j).
* "Teaching the Speculator What a Draft Costs" (al-engr.com), "The controller, and the table
  it reads from" (expected tokens per millisecond, verify_ms[num_tokens]).
* Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
  SC'11 (round function, multipliers and Weyl key increments).

Modules:

* ``philox``     - counter-based uniforms (pinned by published known-answer vectors).
* ``softmax``    - temperature softmax statistics of one logit row.
* ``verify``     - token-wise rule, block verification, greedy branch, residual sampling,
                   and the batch function that mirrors the C-ABI layout.
* ``markov``     - the Markov head's low-rank previous-token bias.
* ``confidence`` - confidence head, prefix survival, expected tokens, pick-k controller.

Every function is pinned by a ``-m "not gpu"`` test against something other than itself
(exact enumeration, closed forms, the pages' worked numbers, brute force); none is
"parity unpinned".
"""

from . import philox, softmax, verify, markov, confidence  # noqa: F401
from .verify import (  # noqa: F401
    STATUS_OK, STATUS_BAD_TEMPERATURE, STATUS_BAD_TOKEN, STATUS_BAD_ROW,
    STATUS_ZERO_DRAFT_PROB, STATUS_BAD_OFFSETS, STATUS_NUMERIC,
    RULE_TOKENWISE, RULE_BLOCK, TIE_REL, DIAG_COLS,
)
