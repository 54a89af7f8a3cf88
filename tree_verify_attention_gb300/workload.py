"""Seeded synthetic inputs for the tree-verify step.

This module is shared by the tests, the benchmark and the oracle checks. It
holds none of the step's arithmetic: it draws random numbers, rounds them to
the storage types (bf16 nearest-even), builds draft-tree shapes and plants
acceptance. It never quantises, attends, takes an argmax or walks a tree.

Workload shapes follow the pages' setting ([P3] feature list: DDTree
tree-verify with block size 16 and default budget 22, Q4_0 KV cache,
2048-token sliding window; [P3]/[P5] benchmark paragraphs: 60K- and
128K-context decode) with synthetic values: the pages measure on HumanEval,
GSM8K and Math500 with trained weights, which these shapes stand in for.

Planted acceptance. Along one planted root path ("spine") the parent row of
each spine edge gets one logit raised to 16.0, far above every N(0,1) draw,
so that token is the row's maximum by construction; with probability ``p``
the spine child's draft token is set to it. Sibling tokens are then made
distinct by redrawing non-spine tokens.

bf16 tensors are carried as ``uint16`` bit patterns.
"""

from dataclasses import dataclass, replace

import numpy as np

BOOST = 16.0  # planted logit; exactly representable in bf16


# ---------------------------------------------------------------- storage types

def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (nearest-even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b):
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- configurations

@dataclass(frozen=True)
class Config:
    name: str
    ctx_len: int
    window: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    budget: int
    max_depth: int
    tree: str            # "random", "chain", "kary2", "kary4"
    planted_depth: int
    p_accept: float
    vocab: int
    logits_dtype: str    # "f32" or "bf16"
    seed: int = 0
    steps: int = 1

    @property
    def n_nodes(self):
        return self.budget + 1


TINY = Config("tiny_ctx256_b8", ctx_len=256, window=0, n_q_heads=4, n_kv_heads=1,
              head_dim=64, budget=8, max_depth=4, tree="random", planted_depth=4,
              p_accept=0.8, vocab=1024, logits_dtype="f32")
SHORT = Config("short_ctx4096_w2048_b22", ctx_len=4096, window=2048, n_q_heads=24,
               n_kv_heads=4, head_dim=256, budget=22, max_depth=16, tree="random",
               planted_depth=8, p_accept=0.8, vocab=151936, logits_dtype="bf16")
LONG_WINDOW = replace(SHORT, name="long_ctx61440_w2048_b22", ctx_len=61440, steps=1000)
FULL_LONG = replace(SHORT, name="full_ctx131072_nowindow_b22", ctx_len=131072, window=0)
SWEEP_BASE = replace(SHORT, name="sweep_ctx32768_w2048", ctx_len=32768)

CONFIGS = {c.name: c for c in (TINY, SHORT, LONG_WINDOW, FULL_LONG)}


def sweep_configs():
    """Tree-shape sweep at context 32768: budgets x shapes x p x seeds."""
    out = []
    for budget in (0, 8, 22, 48, 64):
        for shape in ("chain", "kary2", "kary4", "random"):
            for p in (0.5, 0.8, 0.95):
                for seed in range(5):
                    depth_cap = budget if shape == "chain" else 16
                    out.append(replace(
                        SWEEP_BASE,
                        name=f"sweep_b{budget}_{shape}_p{p}_s{seed}",
                        budget=budget, tree=shape, p_accept=p, seed=seed,
                        max_depth=max(depth_cap, 1),
                        planted_depth=min(8, budget)))
    return out


# ---------------------------------------------------------------- trees

def _depth_of(parent):
    depth = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        depth[i] = depth[parent[i]] + 1
    return depth


def make_tree(rng, n_nodes, shape, max_depth, planted_depth):
    """Return ``(parent, spine)``: parent int32[N] (parent[0] = -1) and the
    spine as a list of node indices from the root."""
    parent = np.full(n_nodes, -1, dtype=np.int64)
    if shape == "chain":
        parent[1:] = np.arange(n_nodes - 1)
        return parent.astype(np.int32), list(range(n_nodes))
    if shape.startswith("kary"):
        k = int(shape[4:])
        for i in range(1, n_nodes):
            parent[i] = (i - 1) // k
        depth = _depth_of(parent)
        end = int(np.argmax(depth))       # lowest-index deepest node
        spine = [end]
        while spine[-1] != 0:
            spine.append(int(parent[spine[-1]]))
        return parent.astype(np.int32), spine[::-1]
    if shape != "random":
        raise ValueError(shape)
    depth = np.zeros(n_nodes, dtype=np.int64)
    P = min(planted_depth, n_nodes - 1, max_depth)
    spine_idx = sorted(rng.choice(np.arange(1, n_nodes), size=P, replace=False).tolist()) if P else []
    spine_set = set(spine_idx)
    prev = 0
    for i in range(1, n_nodes):
        if i in spine_set:
            parent[i] = prev
            prev = i
        else:
            cand = np.nonzero(depth[:i] < max_depth)[0]
            parent[i] = int(rng.choice(cand))
        depth[i] = depth[parent[i]] + 1
    return parent.astype(np.int32), [0] + spine_idx


# ---------------------------------------------------------------- step inputs

@dataclass
class StepInputs:
    parent: np.ndarray   # int32 [N]
    spine: list
    tokens: np.ndarray   # int32 [N]
    q: np.ndarray        # uint16 (bf16) [N, Hq, D]
    k_tree: np.ndarray   # uint16 (bf16) [N, Hkv, D]
    v_tree: np.ndarray   # uint16 (bf16) [N, Hkv, D]
    logits: np.ndarray   # float32 [N, V] or uint16 (bf16) [N, V]


def make_step(cfg, step=0, seed=None):
    """Inputs of verify step ``step`` of ``cfg`` (independent per step)."""
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng((seed, 1, step))
    n, V = cfg.n_nodes, cfg.vocab
    parent, spine = make_tree(rng, n, cfg.tree, cfg.max_depth, cfg.planted_depth)
    tokens = rng.integers(0, V, size=n).astype(np.int64)
    logits = rng.standard_normal((n, V), dtype=np.float32)
    boosted = set()
    for a, b in zip(spine[:-1], spine[1:]):
        t = int(rng.integers(0, V))
        logits[a, t] = BOOST
        boosted.add(a)
        if rng.random() < cfg.p_accept:
            tokens[b] = t
    # distinct sibling tokens: redraw non-spine children that collide
    spine_set = set(spine)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[parent[i]].append(i)
    for a in range(n):
        seen = {int(tokens[c]) for c in kids[a] if c in spine_set}
        for c in kids[a]:
            if c in spine_set:
                continue
            while int(tokens[c]) in seen:
                tokens[c] = int(rng.integers(0, V))
            seen.add(int(tokens[c]))
    if cfg.logits_dtype == "bf16":
        logits = f32_to_bf16_bits(logits)
    hq, hkv, D = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    q = f32_to_bf16_bits(rng.standard_normal((n, hq, D), dtype=np.float32))
    k_tree = f32_to_bf16_bits(rng.standard_normal((n, hkv, D), dtype=np.float32))
    v_tree = f32_to_bf16_bits(rng.standard_normal((n, hkv, D), dtype=np.float32))
    return StepInputs(parent=parent, spine=spine, tokens=tokens.astype(np.int32), q=q,
                      k_tree=k_tree, v_tree=v_tree, logits=logits)


def make_context(cfg, n_rows=None, seed=None, head=None):
    """Committed-context K and V values: float32 N(0,1), [Hkv, n_rows, D]
    (or [n_rows, D] for one ``head``). Each head is its own stream, so a
    single head can be drawn without drawing the others."""
    seed = cfg.seed if seed is None else seed
    n_rows = cfg.ctx_len if n_rows is None else n_rows
    heads = range(cfg.n_kv_heads) if head is None else [head]
    ks, vs = [], []
    for h in heads:
        # K and V of each head are separate streams, so a shorter draw is a
        # prefix of a longer one
        ks.append(np.random.default_rng((seed, 2, h)).standard_normal(
            (n_rows, cfg.head_dim), dtype=np.float32))
        vs.append(np.random.default_rng((seed, 3, h)).standard_normal(
            (n_rows, cfg.head_dim), dtype=np.float32))
    if head is not None:
        return ks[0], vs[0]
    return np.stack(ks), np.stack(vs)
