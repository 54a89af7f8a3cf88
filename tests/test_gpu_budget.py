"""The budget selector against a fresh measurement on this GPU.

A subset of the sweep (every budget, chain and random trees, p = 0.8, seed
0) is timed again with budget.SweepBench. The kernel's accept lengths must
equal the committed table's, the step times must agree with it, and the
selector must choose, from the fresh times, a (budget, shape) whose rate
under the committed table is within a few percent of the committed
choice's."""

import os

import pytest

from tree_verify_attention_gb300 import budget
from tree_verify_attention_gb300 import workload as W

from _helpers import need_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not os.path.exists(budget.TABLE_PATH),
                                 reason="no committed budget table")]

# step times on the same GPU model, other box and clocks: within this factor
TIME_TOL = 0.25


@pytest.fixture(scope="module")
def fresh():
    need_gpu()
    from tree_verify_attention_gb300 import build
    build.build()
    table = budget.load_table()
    n_in = table["meta"]["inputs_per_point"]
    cfgs = [c for c in W.sweep_configs()
            if c.p_accept == 0.8 and c.seed == 0 and c.tree in ("chain", "random")]
    return table, budget.measure_points(cfgs, inputs_per_point=n_in, steps=64)


def _committed(table, pt):
    for p in table["points"]:
        if all(p[k] == pt[k] for k in ("budget", "tree", "p_accept", "seed")):
            return p
    raise KeyError(pt)


def test_fresh_accept_lengths_match_the_table(fresh):
    table, now = fresh
    for pt in now["points"]:
        assert pt["accept_lens"] == _committed(table, pt)["accept_lens"], pt


def test_fresh_step_times_match_the_table(fresh):
    table, now = fresh
    for pt in now["points"]:
        ref = _committed(table, pt)["us_per_step"]
        assert abs(pt["us_per_step"] - ref) <= TIME_TOL * ref, (pt, ref)


def test_selector_choice_holds_on_fresh_times(fresh):
    table, now = fresh
    cand = {(p["budget"], p["tree"]) for p in now["points"]}
    budgets = sorted({b for b, _ in cand})
    shapes = sorted({s for _, s in cand})
    for p in (0.5, 0.8, 0.95):
        prof = lambda b, s, p=p: budget.measured_accept_len(table, b, s, p)
        old = budget.select_budget(prof, table, budgets=budgets, shapes=shapes)
        new = budget.select_budget(prof, now, budgets=budgets, shapes=shapes)
        if (new.budget, new.shape) != (old.budget, old.shape):
            # a near tie may flip: the fresh choice must then be as good under
            # the committed times
            alt = [c for c in budget.rank(prof, table, budgets=budgets, shapes=shapes)
                   if (c.budget, c.shape) == (new.budget, new.shape)][0]
            assert alt.tokens_per_s >= 0.95 * old.tokens_per_s, (p, old, new)
