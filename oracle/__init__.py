"""CPU oracle for the CSA2 hot path (compressor + FP4 quant, hierarchical indexer,
sparse attention over FP4 Main KV + FP8 SWA).

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the method computes, in float64 numpy wherever the sources do
not fix a precision.  Only the test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
CUDA library and its Python binding never import it, and it imports nothing from
them: the two sides share no code.  The only module both sides see is the seeded
input generator, which holds none of the method's arithmetic.

Sources (cited by short name throughout):
  [deep-dive]   "DeepSeek-V4.1-Flash deep dive", tanjunchen.github.io, 2026-09-13.
                Sections used: §2 (CED formulas), §3.1 (CSA2 data flow), §3.2 (modes
                and layer schedule), §3.3 (hierarchical sparse indexer), §3.4 (FP4
                Main KV), §6.3 (structural parameters).
  [paper-reading] "DeepSeek-V4.1-Flash paper reading", inkeast MessageDaily,
                2026-09-19, §4.2 (mode table), §4.3 (FP4 KV cache).
  [daily-report] "Daily technical report 2026-09-11: DeepSeek V4.1 Flash pushes KV
                compression into the model architecture", blog.baizx.cool,
                "core mechanism" paragraph (E2M1 + one E4M3 scale per 16 channels).
  [leak-digest] "DeepSeek V4.1 Flash technical report leaked", agihunt.info,
                "confirmed" list (selected entries + windowed KV into one attention).

Every function states which passage it follows.  Readings taken where the sources
are silent are marked READING at the place they are taken.

Parity status per function (pins live in tests/test_oracle_*.py):
  formats.*            pinned (exhaustive / library cross-checks / golden tables)
  compress.*           pinned (closed forms: m=1, constant Z, RoPE identities)
  indexer.*            pinned (counting definition of top-k, pool invariants)
  attention.*          pinned (dense equality, closed forms, permutation)
  The scoring formula, RoPE layout and softmax scale are readings; the oracle is
  pinned to those readings, not to any number the pages print (none exists).
"""
from . import formats, compress, indexer, attention, schedule  # noqa: F401
