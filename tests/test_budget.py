"""The budget selector (host logic) and the committed measured table.

The selector must return the (budget, shape) with the most accepted tokens
per second, mean accept length / step time, for any form of acceptance
profile; the committed table must cover the whole sweep, and the accept
lengths it recorded from the kernel must be the oracle's greedy walks of
the same seeded inputs."""

import os

import numpy as np
import pytest

import oracle
from tree_verify_attention_gb300 import budget
from tree_verify_attention_gb300 import workload as W


def _table(us, lens):
    """us: {(budget, shape): us}, lens: {(budget, shape, p): [accept lengths]}."""
    pts = []
    for (b, s, p), ls in lens.items():
        pts.append({"budget": b, "tree": s, "p_accept": p, "seed": 0, "us_per_step": us[(b, s)],
                    "accept_lens": ls})
    return {"meta": {}, "points": pts}


US = {(0, "chain"): 10.0, (8, "chain"): 12.0, (22, "chain"): 20.0, (8, "kary2"): 11.0}
LENS = {(0, "chain", 0.5): [1, 1], (8, "chain", 0.5): [2, 2], (22, "chain", 0.5): [3, 3],
        (8, "kary2", 0.5): [2, 1],
        (0, "chain", 0.9): [1, 1], (8, "chain", 0.9): [3, 3], (22, "chain", 0.9): [7, 7],
        (8, "kary2", 0.9): [3, 2]}


def test_select_measured_p():
    t = _table(US, LENS)
    # p 0.5: 1/10, 2/12, 3/20, 1.5/11 tokens per us -> budget 8 chain
    c = budget.select_budget(0.5, t)
    assert (c.budget, c.shape) == (8, "chain")
    assert c.accept_len == 2.0 and c.us_per_step == 12.0
    assert c.tokens_per_s == pytest.approx(2.0 / 12.0 * 1e6)
    # p 0.9: 7/20 beats 3/12
    c = budget.select_budget(0.9, t)
    assert (c.budget, c.shape) == (22, "chain")


def test_rank_is_sorted_and_complete():
    t = _table(US, LENS)
    r = budget.rank(0.5, t)
    assert len(r) == 4
    tps = [c.tokens_per_s for c in r]
    assert tps == sorted(tps, reverse=True)
    # brute force over the grid
    best = max(US, key=lambda k: np.mean(LENS[(k[0], k[1], 0.5)]) / US[k])
    assert (r[0].budget, r[0].shape) == best


def test_profile_forms_and_filters():
    t = _table(US, LENS)
    by_budget = {0: 1.0, 8: 4.0, 22: 5.0}
    c = budget.select_budget(by_budget, t)
    # 4/11 (kary2 at budget 8, the cheaper shape) beats 4/12 and 5/20
    assert (c.budget, c.shape) == (8, "kary2")
    c = budget.select_budget(lambda b, s: 1.0 + b, t)
    assert c.budget == 22                                   # 23/20 is the best rate
    c = budget.select_budget(lambda b, s: 1.0 + b, t, budgets=[0, 8])
    assert (c.budget, c.shape) == (8, "kary2")
    c = budget.select_budget({(0, "chain"): 1.0}, t)       # candidates without a length are skipped
    assert (c.budget, c.shape) == (0, "chain")
    c = budget.select_budget(0.5, t, shapes=["kary2"])
    assert (c.budget, c.shape) == (8, "kary2")


def test_ties_prefer_the_smaller_budget():
    t = _table({(0, "chain"): 10.0, (8, "chain"): 20.0},
               {(0, "chain", 0.5): [1], (8, "chain", 0.5): [2]})
    assert budget.select_budget(0.5, t).budget == 0


def test_bad_profiles():
    t = _table(US, LENS)
    with pytest.raises(ValueError):
        budget.select_budget(0.7, t)                        # p not measured
    with pytest.raises(ValueError):
        budget.select_budget(lambda b, s: 0.5, t)            # the root is always accepted
    with pytest.raises(TypeError):
        budget.select_budget("fast", t)
    with pytest.raises(ValueError):
        budget.select_budget({99: 3.0}, t)                   # no candidate at all


# ---------------------------------------------------------------- the committed table

needs_table = pytest.mark.skipif(not os.path.exists(budget.TABLE_PATH),
                                 reason="no committed budget table")


@needs_table
def test_committed_table_covers_the_sweep():
    t = budget.load_table()
    keys = {(p["budget"], p["tree"], p["p_accept"], p["seed"]) for p in t["points"]}
    want = {(c.budget, c.tree, c.p_accept, c.seed) for c in W.sweep_configs()}
    assert keys == want and len(t["points"]) == len(want) == 300
    n_in = t["meta"]["inputs_per_point"]
    for p in t["points"]:
        assert p["us_per_step"] > 0
        assert len(p["accept_lens"]) == n_in
        assert all(1 <= L <= p["budget"] + 1 for L in p["accept_lens"])
    assert t["meta"]["clocks"]["samples"] > 0
    assert budget.step_us(t, 64, "chain") > budget.step_us(t, 0, "chain")


@needs_table
def test_committed_accept_lengths_are_the_oracle_walks():
    """A sample of points: the kernel's recorded accept lengths equal the
    oracle's greedy walk of the same seeded inputs."""
    t = budget.load_table()
    cfgs = {(c.budget, c.tree, c.p_accept, c.seed): c for c in W.sweep_configs()}
    rng = np.random.default_rng(0)
    pts = [t["points"][i] for i in rng.choice(len(t["points"]), size=6, replace=False)]
    for p in pts:
        cfg = cfgs[(p["budget"], p["tree"], p["p_accept"], p["seed"])]
        for i, L in enumerate(p["accept_lens"]):
            s = W.make_step(cfg, i)
            am = oracle.accept.node_argmax(W.bf16_bits_to_f32(s.logits))
            path, _ = oracle.accept.greedy_walk(s.parent, s.tokens, am)
            assert len(path) == L, (cfg.name, i)
