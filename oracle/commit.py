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

Cache layouts: ``[Hkv, capacity, D/32, 18]`` bytes (Q4_0 blocks per row),
or ``[Hkv, capacity, D]`` binary16 values for the F16 format ([P3] results
paragraph: the F16 cache the Q4_0 one is compared against; see ``f16``),
written with round-to-nearest-even.
"""

import numpy as np

from . import q4_0 as _q
from . import f16 as _f16


class CapacityError(ValueError):
    pass


def encode_rows(rows, fmt="q4_0"):
    """Cache rows of float32 values ``rows`` ([..., D]) in format ``fmt``:
    Q4_0 blocks ([..., D/32, 18] bytes) or binary16 values ([..., D])."""
    if fmt == "q4_0":
        return _q.quantize_rows(rows)
    if fmt == "f16":
        return _f16.encode_rows(rows)
    raise ValueError(f"unknown cache format {fmt!r}")


def decode_rows(rows, fmt="q4_0"):
    """Exact float64 values of cache rows in format ``fmt``."""
    if fmt == "q4_0":
        return _q.dequantize_rows(rows)
    if fmt == "f16":
        return _f16.decode_rows(rows)
    raise ValueError(f"unknown cache format {fmt!r}")


def kv_commit(k_cache, v_cache, ctx_len, path, k_tree, v_tree, fmt="q4_0"):
    """Commit in place; returns the new committed length.

    k_tree / v_tree: float32 values of the tree rows, [N, Hkv, D] (bf16
    values widened exactly to float32). ``fmt`` is the cache format: the
    caches are [Hkv, cap, D/32, 18] bytes for "q4_0" and [Hkv, cap, D]
    binary16 bit patterns (uint16) for "f16".
    """
    cap = k_cache.shape[1]
    L = len(path)
    if ctx_len < 0 or ctx_len + L > cap:
        raise CapacityError(f"ctx {ctx_len} + {L} exceeds capacity {cap}")
    k_rows = np.asarray(k_tree, dtype=np.float32)[np.asarray(path)]  # [L, Hkv, D]
    v_rows = np.asarray(v_tree, dtype=np.float32)[np.asarray(path)]
    axes = (1, 0) + tuple(range(2, encode_rows(k_rows[:1], fmt).ndim))
    k_cache[:, ctx_len:ctx_len + L] = encode_rows(k_rows, fmt).transpose(axes)
    v_cache[:, ctx_len:ctx_len + L] = encode_rows(v_rows, fmt).transpose(axes)
    return ctx_len + L
