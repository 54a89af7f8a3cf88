"""Pins of the oracle's argmax, greedy walk and commit (no GPU)."""

import itertools

import numpy as np
import pytest

from oracle import accept as AC
from oracle import commit as CM
from oracle import q4_0 as Q
from oracle import step as ST
from tree_verify_attention_gb300 import workload as W


# ---------------------------------------------------------------- argmax

def _argmax_loop(row):
    best, bi = row[0], 0
    for i in range(1, len(row)):
        if row[i] > best:
            best, bi = row[i], i
    return bi


def test_argmax_brute_force_small():
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        row = rng.integers(-3, 4, size=V).astype(np.float32)   # many ties
        assert AC.node_argmax(row[None])[0] == _argmax_loop(row.tolist())


def test_argmax_ties_signed_zero_and_ends():
    V = 151936
    row = np.full(V, -1.0, dtype=np.float32)
    assert AC.node_argmax(row[None])[0] == 0                    # all equal
    row[[5000, 70000, V - 1]] = 3.0
    assert AC.node_argmax(row[None])[0] == 5000                 # lowest of ties
    row = np.full(V, -1.0, dtype=np.float32)
    row[V - 1] = 2.0
    assert AC.node_argmax(row[None])[0] == V - 1
    row = np.full(8, -1.0, dtype=np.float32)
    row[3] = 0.0
    row[2] = -0.0
    assert AC.node_argmax(row[None])[0] == 2                    # -0 == +0
    row = np.full(8, -np.inf, dtype=np.float32)
    assert AC.node_argmax(row[None])[0] == 0


# ---------------------------------------------------------------- walk

def _all_matching_paths(parent, tokens, target):
    n = len(parent)
    kids = [[c for c in range(1, n) if parent[c] == a] for a in range(n)]
    out = []

    def rec(path):
        out.append(list(path))
        for c in kids[path[-1]]:
            if tokens[c] == target[path[-1]]:
                rec(path + [c])
    rec([0])
    return out


@pytest.mark.parametrize("seed", range(40))
def test_walk_is_longest_matching_path(seed):
    """With distinct sibling tokens the greedy walk is the unique longest
    root path whose every token matches its parent's target."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    parent = np.full(n, -1)
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    vocab = 4
    target = rng.integers(0, vocab, size=n)
    tokens = np.zeros(n, dtype=int)
    for a in range(n):
        kids = [c for c in range(1, n) if parent[c] == a]
        for c, t in zip(kids, rng.permutation(max(vocab, len(kids)))):
            tokens[c] = t
    path, out_tokens = AC.greedy_walk(parent, tokens, target)
    paths = _all_matching_paths(parent, tokens, target)
    longest = max(len(p) for p in paths)
    assert [p for p in paths if len(p) == longest] == [path.tolist()]
    assert out_tokens.tolist() == [tokens[c] for c in path[1:]] + [target[path[-1]]]


def test_walk_exhaustive_tiny_trees():
    """All trees of 4 nodes, all token/target assignments over 2 symbols."""
    for parents in itertools.product(*[range(i) for i in range(1, 4)]):
        parent = np.array([-1] + list(parents))
        for tok in itertools.product(range(2), repeat=3):
            tokens = np.array([0] + list(tok))
            for tgt in itertools.product(range(2), repeat=4):
                path, _ = AC.greedy_walk(parent, tokens, np.array(tgt))
                # each step is the lowest-index matching child
                for a, b in zip(path[:-1], path[1:]):
                    assert parent[b] == a and tokens[b] == tgt[a]
                    assert not any(parent[c] == a and tokens[c] == tgt[a] for c in range(1, b))
                last = path[-1]
                assert not any(parent[c] == last and tokens[c] == tgt[last] for c in range(1, 4))


def test_walk_duplicate_sibling_takes_lowest_index():
    # root's children 1 and 2 both carry the root's target; only 2 continues
    parent = np.array([-1, 0, 0, 2])
    tokens = np.array([0, 7, 7, 5])
    target = np.array([7, 9, 5, 1])
    path, out = AC.greedy_walk(parent, tokens, target)
    assert path.tolist() == [0, 1]
    assert out.tolist() == [7, 9]


def test_walk_root_only():
    path, out = AC.greedy_walk(np.array([-1]), np.array([3]), np.array([42]))
    assert path.tolist() == [0] and out.tolist() == [42]


# ---------------------------------------------------------------- commit

def test_commit_positions_and_rollback():
    rng = np.random.default_rng(5)
    hkv, cap, D, C = 2, 40, 64, 17
    kc = rng.integers(0, 256, size=(hkv, cap, D // 32, 18)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(hkv, cap, D // 32, 18)).astype(np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    kt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((6, hkv, D))))
    vt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((6, hkv, D))))
    path = [0, 2, 5]
    newc = CM.kv_commit(kc, vc, C, path, kt, vt)
    assert newc == C + 3
    for k, node in enumerate(path):
        for h in range(hkv):
            assert np.array_equal(kc[h, C + k], Q.quantize_rows(kt[node, h][None])[0])
            assert np.array_equal(vc[h, C + k], Q.quantize_rows(vt[node, h][None])[0])
    assert np.array_equal(kc[:, :C], k0[:, :C]) and np.array_equal(kc[:, C + 3:], k0[:, C + 3:])
    assert np.array_equal(vc[:, :C], v0[:, :C]) and np.array_equal(vc[:, C + 3:], v0[:, C + 3:])
    with pytest.raises(CM.CapacityError):
        CM.kv_commit(kc, vc, cap - 2, path, kt, vt)
    assert np.array_equal(kc[:, cap - 2:], k0[:, cap - 2:])


def test_step_composes_the_parts():
    cfg = W.TINY
    s = W.make_step(cfg)
    kf, vf = W.make_context(cfg)
    cap = cfg.ctx_len + 32
    kc = np.zeros((1, cap, 2, 18), np.uint8)
    vc = np.zeros_like(kc)
    kc[:, :cfg.ctx_len] = Q.quantize_rows(kf)
    vc[:, :cfg.ctx_len] = Q.quantize_rows(vf)
    kt = W.bf16_bits_to_f32(s.k_tree)
    vt = W.bf16_bits_to_f32(s.v_tree)
    res = ST.verify_step(kc, vc, cfg.ctx_len, cfg.window, W.bf16_bits_to_f32(s.q), kt, vt,
                         s.parent, s.tokens, s.logits)
    assert res["ctx_len"] == cfg.ctx_len + res["accept_len"]
    assert res["out"].shape == (9, 4, 64)
    assert np.all(np.isfinite(res["out"]))
