"""Pins of the oracle's tree-verify attention (no GPU).

The oracle is compared with torch's scaled_dot_product_attention (a library
routine) under an explicit visibility matrix built here by brute force, and
with closed forms: a chain tree is causal sliding-window decode, a window
longer than everything is no window, budget 0 is one decode query, equal
keys give the mean of the visible values, Hq == Hkv is plain multi-head
attention.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import tree as T


def _rand_tree(rng, n, max_depth):
    parent = np.full(n, -1)
    depth = np.zeros(n, dtype=int)
    for i in range(1, n):
        cand = [j for j in range(i) if depth[j] < max_depth]
        parent[i] = rng.choice(cand)
        depth[i] = depth[parent[i]] + 1
    return parent


def _is_ancestor_or_self(parent, t, i):
    while True:
        if i == t:
            return True
        if i == 0:
            return False
        i = parent[i]


def _brute_mask(parent, C, W):
    """[N, C + N] visibility by brute force: committed key j at position j,
    node t at position C + depth(t)."""
    n = len(parent)
    depth = [0] * n
    for i in range(1, n):
        d, j = 0, i
        while j != 0:
            j = parent[j]
            d += 1
        depth[i] = d
    mask = np.zeros((n, C + n), dtype=bool)
    for i in range(n):
        pos = C + depth[i]
        for j in range(C):
            mask[i, j] = (W == 0) or (pos - j < W)
        for t in range(n):
            mask[i, C + t] = _is_ancestor_or_self(parent, t, i)
    return mask


def _sdpa(q, k_ctx, v_ctx, k_tree, v_tree, mask, C):
    n, hq, d = q.shape
    hkv = k_tree.shape[1]
    g = hq // hkv
    out = np.zeros((n, hq, d))
    lse = np.zeros((n, hq))
    for h in range(hq):
        kv = h // g
        keys = torch.from_numpy(np.concatenate([k_ctx[kv, :C], k_tree[:, kv]]))
        vals = torch.from_numpy(np.concatenate([v_ctx[kv, :C], v_tree[:, kv]]))
        qq = torch.from_numpy(q[:, h])
        m = torch.from_numpy(mask)
        o = torch.nn.functional.scaled_dot_product_attention(
            qq[None], keys[None], vals[None], attn_mask=m[None], scale=1.0 / np.sqrt(d))[0]
        s = (qq @ keys.T) / np.sqrt(d)
        s = s.masked_fill(~m, float("-inf"))
        out[:, h] = o.numpy()
        lse[:, h] = torch.logsumexp(s, dim=-1).numpy()
    return out, lse


def _inputs(rng, n, hq, hkv, d, C):
    q = rng.standard_normal((n, hq, d))
    k_ctx = rng.standard_normal((hkv, C, d))
    v_ctx = rng.standard_normal((hkv, C, d))
    k_tree = rng.standard_normal((n, hkv, d))
    v_tree = rng.standard_normal((n, hkv, d))
    return q, k_ctx, v_ctx, k_tree, v_tree


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("window", [0, 1, 3, 17, 40])
def test_matches_sdpa_with_brute_force_mask(seed, window):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    C = int(rng.integers(0, 48))
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 3]))
    parent = _rand_tree(rng, n, 4)
    q, kc, vc, kt, vt = _inputs(rng, n, hq, hkv, 16, C)
    out, lse = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, window)
    mask = _brute_mask(parent, C, window)
    ref, ref_lse = _sdpa(q, kc, vc, kt, vt, mask, C)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    # the per-KV-head matrix form, against the same brute-force reference
    out_h, lse_h = A.tree_verify_attention_by_head(q, kc, vc, kt, vt, parent, C, window)
    np.testing.assert_allclose(out_h, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse_h, ref_lse, rtol=1e-12, atol=1e-12)


def test_by_head_takes_row_callables():
    """The per-head form reads committed rows through a callable exactly as
    from arrays (the GPU tests pass one that dequantises a head at a time)."""
    rng = np.random.default_rng(23)
    n, C, W = 9, 40, 17
    parent = _rand_tree(rng, n, 4)
    q, kc, vc, kt, vt = _inputs(rng, n, 6, 2, 16, C)
    calls = []

    def fk(kv, lo, hi):
        calls.append((kv, lo, hi))
        return kc[kv, lo:hi]

    out, lse = A.tree_verify_attention_by_head(q, fk, lambda kv, lo, hi: vc[kv, lo:hi], kt, vt,
                                               parent, C, W)
    ref, ref_lse = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, W)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    assert calls == [(0, C - W + 1, C), (1, C - W + 1, C)]


def test_chain_is_causal_sliding_window_decode():
    """A chain draft is ordinary causal decode of the appended sequence."""
    rng = np.random.default_rng(11)
    n, C, W, d = 7, 30, 12, 32
    parent = np.arange(-1, n - 1)
    q, kc, vc, kt, vt = _inputs(rng, n, 2, 1, d, C)
    out, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, W)
    seq_k = np.concatenate([kc[0], kt[:, 0]])   # positions 0 .. C+n-1
    seq_v = np.concatenate([vc[0], vt[:, 0]])
    for i in range(n):
        pos = C + i
        lo = max(0, pos - W + 1)
        for h in range(2):
            s = seq_k[lo:pos + 1] @ q[i, h] / np.sqrt(d)
            p = np.exp(s - s.max())
            np.testing.assert_allclose(out[i, h], p @ seq_v[lo:pos + 1] / p.sum(), rtol=1e-12, atol=1e-13)


def test_long_window_equals_no_window():
    rng = np.random.default_rng(12)
    n, C = 9, 40
    parent = _rand_tree(rng, n, 4)
    q, kc, vc, kt, vt = _inputs(rng, n, 4, 2, 16, C)
    full, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, 0)
    depth_max = int(T.depths(parent).max())
    for W in (C + depth_max + 1, C + 100):
        out, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, W)
        np.testing.assert_array_equal(out, full)
    short, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, C)
    assert not np.allclose(short, full)


def test_budget_zero_is_one_decode_query():
    rng = np.random.default_rng(13)
    C, W, d = 50, 20, 16
    q, kc, vc, kt, vt = _inputs(rng, 1, 3, 1, d, C)
    out, lse = A.tree_verify_attention(q, kc, vc, kt, vt, np.array([-1]), C, W)
    keys = np.concatenate([kc[0, C - W + 1:], kt[:, 0]])
    vals = np.concatenate([vc[0, C - W + 1:], vt[:, 0]])
    assert keys.shape[0] == W
    for h in range(3):
        s = keys @ q[0, h] / np.sqrt(d)
        w = np.exp(s) / np.exp(s).sum()
        np.testing.assert_allclose(out[0, h], w @ vals, rtol=1e-12)
        np.testing.assert_allclose(lse[0, h], np.log(np.exp(s).sum()), rtol=1e-12)


def test_equal_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(14)
    n, C, W, d = 8, 25, 10, 8
    parent = _rand_tree(rng, n, 3)
    q, kc, vc, kt, vt = _inputs(rng, n, 2, 1, d, C)
    kc[:] = 0.7
    kt[:] = 0.7
    out, lse = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, W)
    depth = T.depths(parent)
    anc = T.ancestors_or_self(parent)
    for i in range(n):
        lo = max(0, C + depth[i] - W + 1)
        vis = np.concatenate([vc[0, lo:C], vt[anc[i], 0]])
        count = (C - lo) + depth[i] + 1
        assert vis.shape[0] == count
        for h in range(2):
            np.testing.assert_allclose(out[i, h], vis.mean(axis=0), rtol=1e-12)
            s = 0.7 * q[i, h].sum() / np.sqrt(d)
            np.testing.assert_allclose(lse[i, h], s + np.log(count), rtol=1e-12)


def test_gqa_group_one_is_multi_head():
    rng = np.random.default_rng(15)
    n, C = 6, 20
    parent = _rand_tree(rng, n, 3)
    q, kc, vc, kt, vt = _inputs(rng, n, 3, 3, 16, C)
    out, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, 9)
    for h in range(3):
        one, _ = A.tree_verify_attention(q[:, h:h + 1], kc[h:h + 1], vc[h:h + 1],
                                         kt[:, h:h + 1], vt[:, h:h + 1], parent, C, 9)
        np.testing.assert_array_equal(out[:, h], one[:, 0])


def test_grouped_heads_use_contiguous_groups():
    """Query head h reads KV head h // g: permuting KV heads permutes the
    output head groups."""
    rng = np.random.default_rng(16)
    n, C = 5, 12
    parent = _rand_tree(rng, n, 2)
    q, kc, vc, kt, vt = _inputs(rng, n, 4, 2, 8, C)
    out, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, 0)
    sw = [1, 0]
    out2, _ = A.tree_verify_attention(q[:, [2, 3, 0, 1]], kc[sw], vc[sw], kt[:, sw], vt[:, sw], parent, C, 0)
    np.testing.assert_array_equal(out2, out[:, [2, 3, 0, 1]])


def test_attention_one_matches_full():
    rng = np.random.default_rng(17)
    n, C, W = 9, 33, 15
    parent = _rand_tree(rng, n, 4)
    q, kc, vc, kt, vt = _inputs(rng, n, 4, 2, 16, C)
    out, lse = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, W)
    for i in range(n):
        for h in range(4):
            o, l = A.attention_one(q[i, h], kc[h // 2], vc[h // 2], kt[:, h // 2], vt[:, h // 2],
                                   parent, C, W, i)
            np.testing.assert_allclose(o, out[i, h], rtol=1e-13)
            np.testing.assert_allclose(l, lse[i, h], rtol=1e-13)


def test_tree_helpers():
    parent = np.array([-1, 0, 0, 1, 3, 2])
    assert T.depths(parent).tolist() == [0, 1, 1, 2, 3, 2]
    assert T.ancestors_or_self(parent)[4] == [0, 1, 3, 4]
    assert T.children(parent)[0] == [1, 2]
    with pytest.raises(ValueError):
        T.validate(np.array([-1, 0, 2]))
