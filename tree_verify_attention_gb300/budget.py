"""Tree budget selection from measured step costs.

The verify step's cost grows with the tree budget (the drafted nodes per
step), while the tokens a step accepts grow with it only as far as the
draft model's acceptance allows. "We got 207 tok/s with Qwen3.5-27B on an
RTX 3090" (nowletus), "What we ported and tuned" and the DFlash section,
swept the budget on their GPU and found 22 the best trade-off there. This
module makes that choice for this library on the GPU at hand:

* a table of measured step times per (budget, tree shape) -- the committed
  one (``budget_table_gb300.json``, one GB300, context 32768, window 2048,
  24/4 heads, head_dim 256, vocabulary 151936 bf16, Q4_0 cache) or one
  measured on the caller's GPU with :func:`measure_points`;
* :func:`select_budget`, which returns the (budget, shape) that maximises
  accepted tokens per second, mean accept length / step time, for an
  acceptance profile the caller supplies.

The table also records, per point, the accept lengths the kernel returned
on the synthetic inputs of a planted-acceptance profile (p = 0.5, 0.8,
0.95; seeds 0-4), so a bare p in that set is a usable profile too.
"""

import json
import os
from dataclasses import dataclass

TABLE_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "budget_table_gb300.json")


@dataclass(frozen=True)
class Choice:
    budget: int
    shape: str
    us_per_step: float
    accept_len: float
    tokens_per_s: float


def load_table(path=None):
    """The measured table: {"meta": {...}, "points": [{"budget", "tree",
    "p_accept", "seed", "us_per_step", "accept_lens"}, ...]}."""
    with open(path or TABLE_PATH, encoding="utf-8") as f:
        table = json.load(f)
    if not table.get("points"):
        raise ValueError("budget table has no points")
    return table


def _mean(xs):
    xs = list(xs)
    return sum(xs) / len(xs)


def step_us(table, budget, shape):
    """Measured step time of (budget, shape): the mean over the table's
    points of that budget and shape (every p and seed)."""
    us = [pt["us_per_step"] for pt in table["points"]
          if pt["budget"] == budget and pt["tree"] == shape]
    if not us:
        raise KeyError(f"no measured point for budget {budget}, shape {shape}")
    return _mean(us)


def measured_accept_len(table, budget, shape, p):
    """Mean accept length the kernel returned on the synthetic inputs of
    acceptance profile ``p`` (over every seed and input of the point)."""
    lens = [x for pt in table["points"]
            if pt["budget"] == budget and pt["tree"] == shape and pt["p_accept"] == p
            for x in pt["accept_lens"]]
    if not lens:
        raise KeyError(f"no accept lengths for budget {budget}, shape {shape}, p {p}")
    return _mean(lens)


def grid(table):
    """Sorted (budget, shape) pairs present in the table."""
    return sorted({(pt["budget"], pt["tree"]) for pt in table["points"]})


def _profile_fn(profile, table):
    """Turn an acceptance profile into f(budget, shape) -> mean accept length."""
    if callable(profile):
        return profile
    if isinstance(profile, (int, float)) and not isinstance(profile, bool):
        p = float(profile)
        known = sorted({pt["p_accept"] for pt in table["points"]})
        if p not in known:
            raise ValueError(f"acceptance p {p} was not measured; the table has {known}")
        return lambda b, s: measured_accept_len(table, b, s, p)
    if isinstance(profile, dict):
        def f(b, s):
            if (b, s) in profile:
                return profile[(b, s)]
            if b in profile:
                return profile[b]
            raise KeyError(f"the profile gives no accept length for budget {b}, shape {s}")
        return f
    raise TypeError("profile must be a callable (budget, shape) -> accept length, a dict "
                    "keyed by (budget, shape) or budget, or a measured p")


def rank(profile, table=None, budgets=None, shapes=None):
    """Every candidate (budget, shape) as a Choice, best first. A candidate
    the profile has no accept length for is left out."""
    table = load_table() if table is None else table
    f = _profile_fn(profile, table)
    out = []
    for b, s in grid(table):
        if (budgets is not None and b not in budgets) or (shapes is not None and s not in shapes):
            continue
        try:
            L = float(f(b, s))
        except KeyError:
            continue
        if L < 1.0:
            raise ValueError(f"accept length {L} < 1 for budget {b}, shape {s} (the root "
                             f"is always accepted)")
        us = step_us(table, b, s)
        out.append(Choice(b, s, us, L, L * 1e6 / us))
    # best tokens/s first; ties to the smaller budget, then the shape name
    out.sort(key=lambda c: (-c.tokens_per_s, c.budget, c.shape))
    return out


def select_budget(profile, table=None, budgets=None, shapes=None):
    """The (budget, shape) with the most accepted tokens per second for
    ``profile``, as a Choice.

    profile: a callable (budget, shape) -> expected accept length (accepted
    drafts plus the bonus token, >= 1), a dict keyed by (budget, shape) or
    by budget, or a planted-acceptance p that the table measured."""
    ranked = rank(profile, table, budgets, shapes)
    if not ranked:
        raise ValueError("no candidate (budget, shape) for this profile")
    return ranked[0]


# ---------------------------------------------------------------- measurement

class SweepBench:
    """Times the verify step for many (budget, shape) points on one set of
    KV-cache replicas at a fixed context, on the current GPU.

    Per point: every input runs once eagerly (its replica fresh at the
    context length) and the kernel's accept length is read back; then one
    CUDA graph of ``steps`` strictly serial steps, input i on replica
    i mod ``replicas``, is replayed twice untimed, L2 is flushed, and one
    replay is timed with CUDA events on the launching stream."""

    def __init__(self, base_cfg, replicas=8, steps=64, device="cuda", fmt="q4_0", max_nodes=65):
        import torch
        from . import api
        from . import workload as W
        self._torch, self._api = torch, api
        self.dev = torch.device(device)
        self.cfg, self.R, self.K, self.fmt = base_cfg, replicas, steps, fmt
        C, hkv, D = base_cfg.ctx_len, base_cfg.n_kv_heads, base_cfg.head_dim
        self.cap = C + (-(-steps // replicas) + 2) * max_nodes
        kf, vf = W.make_context(base_cfg)
        base = api.KVCache(hkv, D, self.cap, device=self.dev, fmt=fmt)
        base.fill(torch.from_numpy(kf).to(self.dev), torch.from_numpy(vf).to(self.dev))
        del kf, vf
        self._k = base.k.unsqueeze(0).repeat(replicas, 1, 1, 1)
        self._v = base.v.unsqueeze(0).repeat(replicas, 1, 1, 1)
        self.ctx0 = torch.full((replicas,), C, dtype=torch.int32, device=self.dev)
        self.ctx_all = self.ctx0.clone()
        del base
        self.caches = [_CacheView(self._k[r], self._v[r], self.ctx_all[r:r + 1], hkv, D,
                                  self.cap, fmt) for r in range(replicas)]
        self.stream = torch.cuda.Stream(device=self.dev)
        self._flush = torch.empty(256 << 20, dtype=torch.uint8, device=self.dev)

    def time_point(self, cfg, inputs):
        """(microseconds per step, the kernel's accept length per input)."""
        import numpy as np
        torch, api = self._torch, self._api
        base = self.cfg
        N, hq, hkv, D, Wn, V = (cfg.n_nodes, base.n_q_heads, base.n_kv_heads, base.head_dim,
                                base.window, base.vocab)

        def bf(x):
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(
                torch.bfloat16).to(self.dev)

        ins = [(bf(s.q), bf(s.k_tree), bf(s.v_tree), torch.from_numpy(s.parent).to(self.dev),
                torch.from_numpy(s.tokens).to(self.dev), bf(s.logits)) for s in inputs]
        st = api.VerifyStep(N, hq, hkv, D, Wn, self.cap, V, max_depth=max(cfg.max_depth, 1),
                            device=self.dev)
        s = self.stream
        lens = []
        with torch.cuda.stream(s):
            self.ctx_all.copy_(self.ctx0)
            for i, x in enumerate(ins):
                st.run(self.caches[i % self.R], *x, stream=s)
                lens.append(st.accept_len.clone())
            self.ctx_all.copy_(self.ctx0)
        torch.cuda.synchronize()
        lens = [int(t.item()) for t in lens]
        if int(st.status.item()) != 0:
            raise api.DfvError(f"device status {int(st.status.item()):#x} at {cfg.name}")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(self.K):
                st.run(self.caches[i % self.R], *ins[i % len(ins)], stream=s)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            for _ in range(2):
                self.ctx_all.copy_(self.ctx0)
                g.replay()
            self.ctx_all.copy_(self.ctx0)
            self._flush.zero_()
            e0.record(s)
            g.replay()
            e1.record(s)
            self.ctx_all.copy_(self.ctx0)
        torch.cuda.synchronize()
        if int(st.status.item()) != 0:
            raise api.DfvError(f"device status {int(st.status.item()):#x} at {cfg.name}")
        us = 1000.0 * e0.elapsed_time(e1) / self.K
        del g, st, ins
        return us, lens


class _CacheView:
    """A replica's K / V byte tensors and committed length, shaped like
    api.KVCache."""

    def __init__(self, k, v, ctx_len, n_kv_heads, head_dim, capacity, fmt):
        from . import api
        self.k, self.v, self.ctx_len = k, v, ctx_len
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        self.fmt, self.kv_format = fmt, api._fmt_code(fmt)


def write_table(table, path):
    """Write a table as load_table reads it: the meta block, then one point
    per line."""
    with open(path, "w", encoding="utf-8") as f:
        f.write('{"meta": ' + json.dumps(table["meta"], indent=1) + ',\n "points": [\n')
        f.write(",\n".join("  " + json.dumps(pt) for pt in table["points"]))
        f.write("\n ]}\n")


def point_record(cfg, us, lens):
    return {"budget": cfg.budget, "tree": cfg.tree, "p_accept": cfg.p_accept, "seed": cfg.seed,
            "us_per_step": us, "accept_lens": list(lens)}


def measure_points(cfgs, inputs_per_point=4, steps=64, replicas=8, device="cuda", fmt="q4_0",
                   inputs=None):
    """Measure the sweep points ``cfgs`` (workload configs sharing one
    context) on the current GPU and return a table like load_table's.
    ``inputs(cfg)`` gives a point's step inputs (default: the seeded
    synthetic inputs workload.make_step(cfg, 0 .. inputs_per_point - 1))."""
    from . import workload as W
    cfgs = list(cfgs)
    bench = SweepBench(cfgs[0], replicas=replicas, steps=steps, device=device, fmt=fmt,
                       max_nodes=max(c.n_nodes for c in cfgs))
    points = []
    for c in cfgs:
        xs = inputs(c) if inputs is not None else [W.make_step(c, i) for i in range(inputs_per_point)]
        us, lens = bench.time_point(c, xs)
        points.append(point_record(c, us, lens))
    return {"meta": table_meta(cfgs[0], steps, replicas, fmt), "points": points}


def table_meta(base_cfg, steps, replicas, fmt):
    import torch
    dev = torch.cuda.current_device()
    return {"gpu": torch.cuda.get_device_name(dev), "ctx": base_cfg.ctx_len,
            "window": base_cfg.window, "heads": f"{base_cfg.n_q_heads}/{base_cfg.n_kv_heads}",
            "head_dim": base_cfg.head_dim, "vocab": base_cfg.vocab, "logits": "bf16",
            "kv": fmt, "steps_per_point": steps, "replicas": replicas,
            "timing": "CUDA events over one CUDA graph of strictly serial verify+commit "
                      "steps, after two untimed replays and an L2 flush"}
