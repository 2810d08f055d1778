"""Oracle for the target-verify step of draft-tree speculative decoding.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. This package is a plain, slow,
obviously-correct CPU statement (NumPy, fp64 for floating point) of what the
verify step computes. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. The CUDA library never calls
it, and it shares no code with the CUDA path: its only common ground is the
seeded input generator, which holds none of the method's arithmetic.

Sources (web pages, cited by title and section):

* [TS]  "Draft-tree speculation" (tokenspeed design notes).
* [AK]  "EAGLE Tree Attention candidate layout, positions and visibility"
        (DeepSeek-V4 tree-attention source analysis), sections one to six.
* [MI]  "Medusa, EAGLE-1/2/3, MTP, and tree attention" (ML interview notes,
        chapter 6.4).
* [DD]  "From Greedy to Sampling: The Architecture of Choice in DDTree
        Speculative Decoding", Step 2.

Every function here is pinned by a ``-m "not gpu"`` test against values the
pages print, closed forms, invariants or brute force (tests/test_oracle_*.py).

Modules: ``tree`` (validation, ancestor mask, positions, links), ``rope``,
``attention`` (per-path literal attention), ``walk`` (greedy verification),
``compact`` (KV-row / hidden-row / position compaction), ``merge`` (the
log-sum-exp combine rule), ``argmax`` (the target's argmax per verify row and
the walk fed by it), ``sampling`` (Gumbel-max draws keyed by position and the
walk over them).
"""
from . import tree, rope, attention, walk, compact, merge, argmax, sampling, fp8  # noqa: F401
