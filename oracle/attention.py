"""Tree-verify attention, oracle side (test infrastructure only).

What the step computes. [P3] feature list: the target verifies a DDTree
draft tree in one forward (tree-verify) and decodes with sliding-window
flash attention (default window 2048). [P5] "What we built vs what we
didn't": DDTree is a tree-structured verify. Flash attention and split-K
are only faster routes to plain softmax attention, so this module writes the
plain definition out, in float64:

* committed key ``j`` (0 <= j < C) sits at position ``j``; tree node ``i``
  sits at position ``C + depth[i]``;
* committed key ``j`` is visible to node ``i`` iff ``j < C`` and either the
  window ``W`` is 0 (none) or ``(C + depth[i]) - j < W``;
* tree node ``t`` is visible to node ``i`` iff ``t`` is ``i`` or one of its
  ancestors (the window limits the committed context only);
* query head ``h`` uses KV head ``h // (Hq // Hkv)`` (grouped-query
  attention in contiguous groups);
* ``s = (q . k) * scale``, ``O = sum softmax(s) v`` over the visible keys,
  ``lse = log sum exp(s)``.

Inputs are the exact values: committed K/V already dequantised (float64),
Q and tree K/V as float64 copies of their bf16 values.
"""

import numpy as np

from . import tree as _tree


def visible_committed(ctx_len, window, depth_i):
    """Half-open range [lo, C) of committed keys node ``i`` sees."""
    if window == 0:
        return 0, ctx_len
    lo = ctx_len + depth_i - window + 1
    return max(0, min(lo, ctx_len)), ctx_len


def tree_verify_attention(q, k_ctx, v_ctx, k_tree, v_tree, parent, ctx_len,
                          window, scale=None):
    """Return ``(out, lse)``.

    q:       [N, Hq, D]    queries of the N tree nodes
    k_ctx:   [Hkv, >=C, D] committed keys (dequantised); v_ctx likewise
    k_tree:  [N, Hkv, D]   keys of the tree nodes; v_tree likewise
    out:     [N, Hq, D] float64, lse: [N, Hq] float64 (natural log)
    """
    q = np.asarray(q, dtype=np.float64)
    k_ctx = np.asarray(k_ctx, dtype=np.float64)
    v_ctx = np.asarray(v_ctx, dtype=np.float64)
    k_tree = np.asarray(k_tree, dtype=np.float64)
    v_tree = np.asarray(v_tree, dtype=np.float64)
    n, hq, d = q.shape
    hkv = k_tree.shape[1]
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    depth = _tree.depths(parent)
    anc = _tree.ancestors_or_self(parent)
    out = np.zeros((n, hq, d), dtype=np.float64)
    lse = np.zeros((n, hq), dtype=np.float64)
    for i in range(n):
        lo, hi = visible_committed(ctx_len, window, int(depth[i]))
        for h in range(hq):
            kv = h // group
            keys = np.concatenate([k_ctx[kv, lo:hi], k_tree[anc[i], kv]], axis=0)
            vals = np.concatenate([v_ctx[kv, lo:hi], v_tree[anc[i], kv]], axis=0)
            s = (keys @ q[i, h]) * scale
            mx = s.max()
            p = np.exp(s - mx)
            den = p.sum()
            out[i, h] = (p @ vals) / den
            lse[i, h] = mx + np.log(den)
    return out, lse


def attention_one(q_ih, k_ctx_kv, v_ctx_kv, k_tree_kv, v_tree_kv, parent,
                  ctx_len, window, node, scale=None):
    """Output row of one (node, query head) pair; used for sampled checks
    at sizes where the full product is too slow. Arrays are the KV head's
    slices: k_ctx_kv [>=C, D], k_tree_kv [N, D]."""
    depth = _tree.depths(parent)
    anc = _tree.ancestors_or_self(parent)[node]
    lo, hi = visible_committed(ctx_len, window, int(depth[node]))
    q_ih = np.asarray(q_ih, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(q_ih.shape[0])
    keys = np.concatenate([np.asarray(k_ctx_kv[lo:hi], np.float64),
                           np.asarray(k_tree_kv, np.float64)[anc]], axis=0)
    vals = np.concatenate([np.asarray(v_ctx_kv[lo:hi], np.float64),
                           np.asarray(v_tree_kv, np.float64)[anc]], axis=0)
    s = (keys @ q_ih) * scale
    mx = s.max()
    p = np.exp(s - mx)
    den = p.sum()
    return (p @ vals) / den, mx + np.log(den)


def tree_verify_attention_by_head(q, k_ctx, v_ctx, k_tree, v_tree, parent, ctx_len,
                                  window, scale=None):
    """The same ``(out, lse)`` as ``tree_verify_attention``, computed one KV
    head at a time with whole-matrix products instead of a loop over (node,
    query head) pairs, so that it finishes in seconds at a context of
    131072. The definition is unchanged: every row of a KV head's group
    scores the committed keys of the union of the visible ranges and the
    tree keys, the keys a row may not see get -inf (window per node depth,
    ancestors-or-self for tree keys), then a max-subtracted softmax in
    float64. ``k_ctx`` / ``v_ctx`` may be callables ``f(kv, lo, hi)``
    returning the KV head's rows [lo, hi) (so that a caller can dequantise
    one head at a time)."""
    q = np.asarray(q, dtype=np.float64)
    k_tree = np.asarray(k_tree, dtype=np.float64)
    v_tree = np.asarray(v_tree, dtype=np.float64)
    n, hq, d = q.shape
    hkv = k_tree.shape[1]
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(float(d))
    depth = _tree.depths(parent)
    anc = _tree.ancestors_or_self(parent)
    ranges = [visible_committed(ctx_len, window, int(depth[i])) for i in range(n)]
    lo_all = min(lo for lo, _ in ranges) if n else 0
    # visibility of each row (node i, query head h within the group), row
    # index i * group + h: committed keys [lo_all, C) then tree keys 0..N-1
    vis_c = np.zeros((n, ctx_len - lo_all), dtype=bool)
    for i, (lo, hi) in enumerate(ranges):
        vis_c[i, lo - lo_all:hi - lo_all] = True
    vis_t = np.zeros((n, n), dtype=bool)
    for i in range(n):
        vis_t[i, anc[i]] = True
    vis = np.repeat(np.concatenate([vis_c, vis_t], axis=1), group, axis=0)

    def rows(src, kv):
        if callable(src):
            return np.asarray(src(kv, lo_all, ctx_len), dtype=np.float64)
        return np.asarray(src[kv, lo_all:ctx_len], dtype=np.float64)

    out = np.zeros((n, hq, d), dtype=np.float64)
    lse = np.zeros((n, hq), dtype=np.float64)
    for kv in range(hkv):
        qg = q[:, kv * group:(kv + 1) * group].reshape(n * group, d)
        keys = np.concatenate([rows(k_ctx, kv), k_tree[:, kv]], axis=0)
        vals = np.concatenate([rows(v_ctx, kv), v_tree[:, kv]], axis=0)
        s = (qg @ keys.T) * scale
        s = np.where(vis, s, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        p = np.exp(s - mx)
        den = p.sum(axis=1, keepdims=True)
        o = (p @ vals) / den
        out[:, kv * group:(kv + 1) * group] = o.reshape(n, group, d)
        lse[:, kv * group:(kv + 1) * group] = (mx + np.log(den)).reshape(n, group)
    return out, lse
