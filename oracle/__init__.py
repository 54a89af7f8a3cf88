"""Plain CPU oracle for the greedy DDTree tree-verify step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

The oracle is deliberately slow and obvious. It shares no code, header,
table or helper with the CUDA library; the only thing both sides use is the
seeded input generator in ``tree_verify_attention_gb300.workload``, which
holds none of the method's arithmetic.

Sources (cited by page title and section throughout):

* [P3] "Luce DFlash: Qwen3.6-27B aiming for up to 2x throughput on a single
  RTX 3090" (ai-navigate-news.com, Japanese translation of the announcement),
  feature list: DDTree tree-verify with block size 16, default budget 22,
  greedy verification; Q4_0 as the legacy KV-cache format; sliding-window
  flash attention at decode with a 2048-token default window; results
  paragraph: the target graph is bit-identical to autoregressive mode.
* [P5] "We got 207 tok/s with Qwen3.5-27B on an RTX 3090" (nowletus.com),
  DFlash section: DDTree budget=22; "What we ported and tuned": Q4_0 KV
  cache; "What we built vs what we didn't": DDTree is a tree-structured
  verify.

Module map:

* ``q4_0``      -- Q4_0 block quantise / dequantise (fp32 rule, exact).
* ``f16``       -- the binary16 (F16) cache format.
* ``tree``      -- depth and ancestor sets of a draft tree.
* ``attention`` -- tree-masked softmax attention, fp64, straight from the
                   definition (no flash / split-K restructuring).
* ``accept``    -- per-node argmax and the greedy tree walk.
* ``commit``    -- commit of the accepted rows into the cache (Q4_0 or F16).
* ``step``      -- the whole verify step composed from the above.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms, invariants or library routines. Parity
with the pages' own implementation is unpinned: the pages print no worked
example and no kernel output.
"""

from . import q4_0, f16, tree, attention, accept, commit, step  # noqa: F401
