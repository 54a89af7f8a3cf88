"""KV commit / rollback, oracle side (test infrastructure only).

[P3] feature list: the verify step runs over a Q4_0 KV cache ([P5] "What we
ported and tuned": Q4_0 KV cache). After greedy acceptance the accepted
nodes' K/V rows are kept and the rejected ones dropped. The adopted reading:

* accepted row ``k`` (path order, root first) of every KV head is
  quantised to Q4_0 and written at cache position ``C + k``;
* the committed length becomes ``C + L``;
* rejected nodes are never written (rollback is "not written"), so cache
  bytes at positions ``>= C + L`` are unchanged;
* if ``C + L`` exceeds the capacity, nothing is written and the length is
  unchanged (the caller sees an error).

Cache layout: ``[Hkv, capacity, D/32, 18]`` bytes (Q4_0 blocks per row).
"""

import numpy as np

from . import q4_0 as _q


class CapacityError(ValueError):
    pass


def kv_commit(k_cache, v_cache, ctx_len, path, k_tree, v_tree):
    """Commit in place; returns the new committed length.

    k_tree / v_tree: float32 values of the tree rows, [N, Hkv, D] (bf16
    values widened exactly to float32).
    """
    cap = k_cache.shape[1]
    L = len(path)
    if ctx_len < 0 or ctx_len + L > cap:
        raise CapacityError(f"ctx {ctx_len} + {L} exceeds capacity {cap}")
    k_rows = np.asarray(k_tree, dtype=np.float32)[np.asarray(path)]  # [L, Hkv, D]
    v_rows = np.asarray(v_tree, dtype=np.float32)[np.asarray(path)]
    k_cache[:, ctx_len:ctx_len + L] = _q.quantize_rows(k_rows).transpose(1, 0, 2, 3)
    v_cache[:, ctx_len:ctx_len + L] = _q.quantize_rows(v_rows).transpose(1, 0, 2, 3)
    return ctx_len + L
