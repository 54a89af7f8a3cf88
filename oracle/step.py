"""The whole greedy tree-verify step, oracle side (test infrastructure only).

Composition, in the order the step runs it ([P3] feature list: DDTree
tree-verify, greedy verification, Q4_0 KV cache, sliding window):

1. decode the visible committed K/V (exact, float64): Q4_0 by default, or
   the F16 format ([P3] results paragraph);
2. tree-masked softmax attention of the N tree nodes;
3. per-node vocabulary argmax;
4. greedy tree walk;
5. commit of the accepted rows in the cache format, advancing the
   committed length.
"""

import numpy as np

from . import q4_0 as _q
from . import attention as _attn
from . import accept as _acc
from . import commit as _commit


def tree_rows_attended(k_tree, v_tree, fmt="q4_0", tree_as_cache=False):
    """The tree nodes' K/V as the attention sees them. By default (reading
    R3) the unquantised rows; with ``tree_as_cache`` the rows as the commit
    stores them in the cache format (the other reading: tree rows written to
    the cache before attention, rollback by truncation)."""
    if not tree_as_cache:
        return k_tree, v_tree
    return (_commit.decode_rows(_commit.encode_rows(np.asarray(k_tree, np.float32), fmt), fmt),
            _commit.decode_rows(_commit.encode_rows(np.asarray(v_tree, np.float32), fmt), fmt))


def verify_step(k_cache, v_cache, ctx_len, window, q, k_tree, v_tree, parent,
                tokens, logits, scale=None, with_attention=True, fmt="q4_0",
                tree_as_cache=False):
    """Run one step; ``k_cache`` / ``v_cache`` (format ``fmt``: Q4_0 bytes
    [Hkv, cap, D/32, 18] or binary16 bits [Hkv, cap, D]) are updated in
    place. Returns a dict of results."""
    res = {}
    if with_attention:
        lo = 0 if window == 0 else max(0, ctx_len - window + 1)
        d = k_cache.shape[2] * _q.QK if fmt == "q4_0" else k_cache.shape[2]
        k_ctx = np.zeros(k_cache.shape[:2] + (d,))
        v_ctx = np.zeros_like(k_ctx)
        k_ctx[:, lo:ctx_len] = _commit.decode_rows(k_cache[:, lo:ctx_len], fmt)
        v_ctx[:, lo:ctx_len] = _commit.decode_rows(v_cache[:, lo:ctx_len], fmt)
        k_att, v_att = tree_rows_attended(k_tree, v_tree, fmt, tree_as_cache)
        res["out"], res["lse"] = _attn.tree_verify_attention(
            q, k_ctx, v_ctx, k_att, v_att, parent, ctx_len, window, scale)
    res["argmax"] = _acc.node_argmax(logits)
    res["path"], res["out_tokens"] = _acc.greedy_walk(parent, tokens, res["argmax"])
    res["accept_len"] = len(res["path"])
    res["ctx_len"] = _commit.kv_commit(k_cache, v_cache, ctx_len, res["path"],
                                       k_tree, v_tree, fmt)
    return res
