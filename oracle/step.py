"""The whole greedy tree-verify step, oracle side (test infrastructure only).

Composition, in the order the step runs it ([P3] feature list: DDTree
tree-verify, greedy verification, Q4_0 KV cache, sliding window):

1. dequantise the visible committed K/V (exact, float64);
2. tree-masked softmax attention of the N tree nodes;
3. per-node vocabulary argmax;
4. greedy tree walk;
5. Q4_0 commit of the accepted rows, advancing the committed length.
"""

import numpy as np

from . import q4_0 as _q
from . import attention as _attn
from . import accept as _acc
from . import commit as _commit


def verify_step(k_cache, v_cache, ctx_len, window, q, k_tree, v_tree, parent,
                tokens, logits, scale=None, with_attention=True):
    """Run one step; ``k_cache`` / ``v_cache`` ([Hkv, cap, D/32, 18] bytes)
    are updated in place. Returns a dict of results."""
    res = {}
    if with_attention:
        lo = 0 if window == 0 else max(0, ctx_len - window + 1)
        k_ctx = np.zeros(k_cache.shape[:2] + (k_cache.shape[2] * _q.QK,))
        v_ctx = np.zeros_like(k_ctx)
        k_ctx[:, lo:ctx_len] = _q.dequantize_rows(k_cache[:, lo:ctx_len])
        v_ctx[:, lo:ctx_len] = _q.dequantize_rows(v_cache[:, lo:ctx_len])
        res["out"], res["lse"] = _attn.tree_verify_attention(
            q, k_ctx, v_ctx, k_tree, v_tree, parent, ctx_len, window, scale)
    res["argmax"] = _acc.node_argmax(logits)
    res["path"], res["out_tokens"] = _acc.greedy_walk(parent, tokens, res["argmax"])
    res["accept_len"] = len(res["path"])
    res["ctx_len"] = _commit.kv_commit(k_cache, v_cache, ctx_len, res["path"],
                                       k_tree, v_tree)
    return res
