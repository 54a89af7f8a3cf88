"""The pins catch plausible mistakes (no GPU). Each case plants one mistake
in a copy of an oracle module's source (a dropped term, a wrong constant,
sign, index or tie rule), loads the copy as a separate module, and checks
that the pins written for that part fail on it while they pass on the real
module. The oracle itself is never modified."""

import importlib
import inspect
import json
import os
import types

import numpy as np
import pytest

import test_oracle_attention as TA
from tree_verify_attention_gb300 import workload as W

GOLDEN_Q4 = os.path.join(os.path.dirname(__file__), "golden", "q4_0_worked_examples.json")


def mutant(modname, old, new):
    """The module ``modname`` with ``old`` (present exactly once in its
    source) replaced by ``new``, loaded under another name."""
    real = importlib.import_module(modname)
    src = inspect.getsource(real)
    assert src.count(old) == 1, f"{old!r} not found once in {modname}"
    pkg = modname.rpartition(".")[0]
    mod = types.ModuleType(f"{modname}_mutant")
    mod.__package__ = pkg
    mod.__file__ = real.__file__
    exec(compile(src.replace(old, new), f"{real.__file__} (mutant)", "exec"), mod.__dict__)
    return mod


def fails(pin, *mods):
    try:
        pin(*mods)
    except AssertionError:
        return True
    return False


# ---------------------------------------------------------------- pins, parameterised

def pin_q4_golden(Q):
    for case in json.load(open(GOLDEN_Q4))["cases"]:
        x = np.zeros(32, dtype=np.float32)
        for k, v in case["x"].items():
            x[int(k)] = v
        raw = Q.quantize_rows(x[None])[0, 0]
        assert raw.tobytes().hex() == case["bytes"], case["name"]


def pin_attention_sdpa(A):
    for seed in range(4):
        for window in (0, 1, 3, 17):
            rng = np.random.default_rng(seed)
            n = int(rng.integers(2, 10))
            C = int(rng.integers(4, 48))
            parent = TA._rand_tree(rng, n, 4)
            q, kc, vc, kt, vt = TA._inputs(rng, n, 4, 2, 16, C)
            out, lse = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, window)
            ref, ref_lse = TA._sdpa(q, kc, vc, kt, vt, TA._brute_mask(parent, C, window), C)
            assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)
            assert np.allclose(lse, ref_lse, rtol=1e-10, atol=1e-12)


def pin_attention_by_head_sdpa(A):
    for seed in range(4):
        for window in (0, 1, 3, 17):
            rng = np.random.default_rng(seed)
            n = int(rng.integers(2, 10))
            C = int(rng.integers(4, 48))
            parent = TA._rand_tree(rng, n, 4)
            q, kc, vc, kt, vt = TA._inputs(rng, n, 4, 2, 16, C)
            out, lse = A.tree_verify_attention_by_head(q, kc, vc, kt, vt, parent, C, window)
            ref, ref_lse = TA._sdpa(q, kc, vc, kt, vt, TA._brute_mask(parent, C, window), C)
            assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)
            assert np.allclose(lse, ref_lse, rtol=1e-10, atol=1e-12)


def pin_attention_groups(A):
    rng = np.random.default_rng(16)
    n, C = 5, 12
    parent = TA._rand_tree(rng, n, 2)
    q, kc, vc, kt, vt = TA._inputs(rng, n, 4, 2, 8, C)
    out, _ = A.tree_verify_attention(q, kc, vc, kt, vt, parent, C, 0)
    ref, _ = TA._sdpa(q, kc, vc, kt, vt, TA._brute_mask(parent, C, 0), C)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def pin_argmax_ties(AC):
    lg = np.full((3, 9), -1.0)
    lg[0, [2, 5, 8]] = 4.0
    lg[1, [0, 8]] = 2.0
    lg[2, [3, 6]] = [-0.0, 0.0]
    lg[2, [0, 1, 2, 4, 5, 7, 8]] = -3.0
    assert AC.node_argmax(lg).tolist() == [2, 0, 3]


def pin_walk_lowest_child(AC):
    parent = np.array([-1, 0, 0, 2])
    tokens = np.array([0, 7, 7, 5])
    target = np.array([7, 9, 5, 1])
    path, out = AC.greedy_walk(parent, tokens, target)
    assert path.tolist() == [0, 1] and out.tolist() == [7, 9]


def pin_commit_positions(CM, Q):
    rng = np.random.default_rng(5)
    hkv, cap, D, C = 2, 40, 64, 17
    kc = rng.integers(0, 256, size=(hkv, cap, D // 32, 18)).astype(np.uint8)
    vc = kc.copy()
    k0 = kc.copy()
    kt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((6, hkv, D))))
    vt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((6, hkv, D))))
    path = [0, 2, 5]
    assert CM.kv_commit(kc, vc, C, path, kt, vt) == C + 3
    for k, node in enumerate(path):
        for h in range(hkv):
            assert np.array_equal(kc[h, C + k], Q.quantize_rows(kt[node, h][None])[0])
            assert np.array_equal(vc[h, C + k], Q.quantize_rows(vt[node, h][None])[0])
    assert np.array_equal(kc[:, :C], k0[:, :C]) and np.array_equal(kc[:, C + 3:], k0[:, C + 3:])


def pin_f16_golden(F):
    with open(os.path.join(os.path.dirname(__file__), "golden", "f16_worked_examples.json")) as f:
        for ex in json.load(f)["examples"]:
            x = np.array([float(ex["value"])], dtype=np.float32)
            assert int(F.to_f16_bits(x)[0]) == int(ex["bits"], 16), ex["why"]


def pin_tree_as_cache_chain(S, CM):
    """A fully accepted chain with the tree rows attended as cached sees, at
    node i, plain attention over the committed cache rows [0, C + i]."""
    rng = np.random.default_rng(11)
    hkv, hq, D, C, n = 1, 2, 64, 50, 6
    kf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    vf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    kc = np.zeros((hkv, C + n, D // 32, 18), np.uint8)
    vc = np.zeros_like(kc)
    kc[:, :C] = CM.encode_rows(kf)
    vc[:, :C] = CM.encode_rows(vf)
    bf = lambda a: W.bf16_bits_to_f32(W.f32_to_bf16_bits(a.astype(np.float32)))
    q, kt, vt = (bf(rng.standard_normal(sh)) for sh in ((n, hq, D), (n, hkv, D), (n, hkv, D)))
    tokens = np.arange(n, dtype=np.int32)
    logits = np.zeros((n, 8), np.float32)
    for i in range(n - 1):
        logits[i, tokens[i + 1]] = 1.0
    res = S.verify_step(kc, vc, C, 0, q, kt, vt, np.arange(-1, n - 1, dtype=np.int32), tokens,
                        logits, tree_as_cache=True)
    for i in range(n):
        keys = CM.decode_rows(kc[0, :C + i + 1])
        vals = CM.decode_rows(vc[0, :C + i + 1])
        for h in range(hq):
            sc = keys @ q[i, h].astype(np.float64) / np.sqrt(D)
            p = np.exp(sc - sc.max())
            assert np.allclose(res["out"][i, h], p @ vals / p.sum(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- the mistakes

def _real(name):
    return importlib.import_module(name)


CASES = [
    ("q4_0: 8.0 instead of 8.5 before truncation", pin_q4_golden,
     [("oracle.q4_0", "np.float32(8.5)", "np.float32(8.0)")]),
    ("q4_0: last element of largest magnitude", pin_q4_golden,
     [("oracle.q4_0", "idx = np.argmax(np.abs(blocks), axis=-1)",
       "idx = QK - 1 - np.argmax(np.abs(blocks)[..., ::-1], axis=-1)")]),
    ("q4_0: no clamp of q = 16", pin_q4_golden,
     [("oracle.q4_0", "np.minimum(np.trunc(shifted), np.float32(15.0))", "np.trunc(shifted)")]),
    ("q4_0: d = m / 8 (sign dropped)", pin_q4_golden,
     [("oracle.q4_0", "np.divide(m, np.float32(-8.0), dtype=np.float32)",
       "np.divide(m, np.float32(8.0), dtype=np.float32)")]),
    ("attention: window one key too wide", pin_attention_sdpa,
     [("oracle.attention", "lo = ctx_len + depth_i - window + 1", "lo = ctx_len + depth_i - window")]),
    ("attention: window from the root's position", pin_attention_sdpa,
     [("oracle.attention", "lo = ctx_len + depth_i - window + 1", "lo = ctx_len - window + 1")]),
    ("attention: scale 1/D", pin_attention_sdpa,
     [("oracle.attention", "scale = 1.0 / np.sqrt(d)", "scale = 1.0 / d")]),
    ("attention: query head h % g", pin_attention_groups,
     [("oracle.attention", "kv = h // group", "kv = h % hkv")]),
    ("attention: node excluded from its own keys", pin_attention_sdpa,
     [("oracle.attention", "anc = _tree.ancestors_or_self(parent)\n    out = np.zeros",
       "anc = [a[:-1] if len(a) > 1 else a for a in _tree.ancestors_or_self(parent)]\n"
       "    out = np.zeros")]),
    ("attention by head: window range one key late", pin_attention_by_head_sdpa,
     [("oracle.attention", "vis_c[i, lo - lo_all:hi - lo_all] = True",
       "vis_c[i, lo - lo_all + 1:hi - lo_all] = True")]),
    ("attention by head: scale 1/D", pin_attention_by_head_sdpa,
     [("oracle.attention", "scale = 1.0 / np.sqrt(float(d))", "scale = 1.0 / float(d)")]),
    ("attention by head: query heads strided over KV heads", pin_attention_by_head_sdpa,
     [("oracle.attention", "qg = q[:, kv * group:(kv + 1) * group].reshape(n * group, d)",
       "qg = q[:, kv::hkv].reshape(n * group, d)")]),
    ("attention by head: node excluded from its own keys", pin_attention_by_head_sdpa,
     [("oracle.attention", "vis_t[i, anc[i]] = True", "vis_t[i, anc[i][:-1]] = True")]),
    ("argmax: last index of the maximum", pin_argmax_ties,
     [("oracle.accept", "return np.argmax(np.asarray(logits, dtype=np.float64), axis=-1).astype(np.int64)",
       "x = np.asarray(logits, dtype=np.float64)\n"
       "    return (x.shape[-1] - 1 - np.argmax(x[..., ::-1], axis=-1)).astype(np.int64)")]),
    ("walk: highest-index matching child", pin_walk_lowest_child,
     [("oracle.accept", "                nxt = c\n                break\n", "                nxt = c\n")]),
    ("commit: rows one position late", pin_commit_positions,
     [("oracle.commit", "k_cache[:, ctx_len:ctx_len + L]", "k_cache[:, ctx_len + 1:ctx_len + L + 1]")]),
    ("f16: rounding toward zero", pin_f16_golden,
     [("oracle.f16", "return x.astype(np.float16).view(np.uint16)",
       "h = x.astype(np.float16)\n"
       "    h = np.where(np.abs(h.astype(np.float32)) > np.abs(x), "
       "np.nextafter(h, np.float16(0)), h)\n"
       "    return h.astype(np.float16).view(np.uint16)")]),
    ("tree as cache: flag ignored", pin_tree_as_cache_chain,
     [("oracle.step", "    if not tree_as_cache:\n        return k_tree, v_tree",
       "    if True:\n        return k_tree, v_tree")]),
]


@pytest.mark.parametrize("name,pin,edits", CASES, ids=[c[0] for c in CASES])
def test_pin_catches_planted_mistake(name, pin, edits):
    mods = {"pin_q4_golden": ["oracle.q4_0"],
            "pin_attention_sdpa": ["oracle.attention"],
            "pin_attention_by_head_sdpa": ["oracle.attention"],
            "pin_attention_groups": ["oracle.attention"],
            "pin_argmax_ties": ["oracle.accept"],
            "pin_walk_lowest_child": ["oracle.accept"],
            "pin_commit_positions": ["oracle.commit", "oracle.q4_0"],
            "pin_f16_golden": ["oracle.f16"],
            "pin_tree_as_cache_chain": ["oracle.step", "oracle.commit"]}[pin.__name__]
    pin(*[_real(m) for m in mods])                     # the real oracle passes
    planted = {m: mutant(m, old, new) for m, old, new in edits}
    assert fails(pin, *[planted.get(m, _real(m)) for m in mods]), name
