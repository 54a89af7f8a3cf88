"""The seeded generator: determinism, tree shapes, planting, bf16 rounding."""

import numpy as np
import pytest
import torch

from oracle import accept as AC
from oracle import tree as T
from tree_verify_attention_gb300 import workload as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.float32([0.0, -0.0, 1.0, 1.00390625, 1.0078125, 65504.0, 3.0e38])])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_deterministic():
    a = W.make_step(W.TINY, 3)
    b = W.make_step(W.TINY, 3)
    for f in ("parent", "tokens", "q", "k_tree", "v_tree", "logits"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = W.make_step(W.TINY, 4)
    assert not np.array_equal(a.q, c.q)


def test_context_prefix_property():
    k1, v1 = W.make_context(W.TINY, n_rows=100)
    k2, v2 = W.make_context(W.TINY, n_rows=300)
    assert np.array_equal(k1, k2[:, :100]) and np.array_equal(v1, v2[:, :100])
    kh, vh = W.make_context(W.TINY, n_rows=100, head=0)
    assert np.array_equal(kh, k1[0]) and np.array_equal(vh, v1[0])


@pytest.mark.parametrize("cfg", [W.TINY, W.SHORT] + W.sweep_configs()[::37], ids=lambda c: c.name)
def test_tree_shape_and_planting(cfg):
    s = W.make_step(cfg)
    n = cfg.n_nodes
    T.validate(s.parent)
    depth = T.depths(s.parent)
    assert depth.max() <= cfg.max_depth
    # spine is a root path
    assert s.spine[0] == 0
    for a, b in zip(s.spine[:-1], s.spine[1:]):
        assert s.parent[b] == a
    # sibling tokens are distinct
    for a in range(n):
        toks = [int(s.tokens[c]) for c in range(1, n) if s.parent[c] == a]
        assert len(toks) == len(set(toks))
    logits = s.logits if cfg.logits_dtype == "f32" else W.bf16_bits_to_f32(s.logits)
    assert logits.shape == (n, cfg.vocab)
    # every spine parent row holds exactly one planted value
    for a in s.spine[:-1]:
        assert np.count_nonzero(logits[a] == W.BOOST) == 1


def test_planted_acceptance_rate():
    """Over many steps the accepted spine length follows p: the walk takes
    spine edge k with probability p^k (the oracle's walk on generator
    inputs)."""
    cfg = W.TINY
    lens = []
    for step in range(400):
        s = W.make_step(cfg, step)
        target = AC.node_argmax(s.logits)
        path, _ = AC.greedy_walk(s.parent, s.tokens, target)
        lens.append(len(path))
    mean = np.mean(lens)
    P = cfg.planted_depth
    expect = 1 + sum(cfg.p_accept ** k for k in range(1, P + 1))
    assert abs(mean - expect) < 0.25


def test_sweep_covers_the_grid():
    cfgs = W.sweep_configs()
    assert len(cfgs) == 5 * 4 * 3 * 5
    assert {c.n_nodes for c in cfgs} == {1, 9, 23, 49, 65}
    chain64 = [c for c in cfgs if c.tree == "chain" and c.budget == 64][0]
    assert T.depths(W.make_step(chain64).parent).max() == 64
