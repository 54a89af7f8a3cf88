"""Pins of the oracle's binary16 (F16) cache format and of the tree-as-cache
reading of the tree rows.

* worked examples derived by hand from the binary16 layout
  (tests/golden/f16_worked_examples.json);
* every bf16 value in the binary16 normal range converts exactly (bf16 has
  8 significant bits, binary16 11);
* bf16 values below the normal range land on the nearest multiple of 2^-24
  with ties to even, checked with exact integer arithmetic;
* commit in the F16 format writes the encoded accepted rows at C..C+L-1
  only;
* with the tree rows attended as the commit stores them, a chain's node i
  sees exactly the keys a decode over the committed cache would see.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tree_verify_attention_gb300 import workload as W

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    with open(os.path.join(HERE, "golden", "f16_worked_examples.json")) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("ex", _golden(), ids=lambda e: e["bits"])
def test_worked_examples(ex):
    x = np.array([float(ex["value"])], dtype=np.float32)
    assert int(oracle.f16.to_f16_bits(x)[0]) == int(ex["bits"], 16), ex["why"]


def _all_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = W.bf16_bits_to_f32(bits)
    return vals[np.isfinite(vals)]


def test_bf16_in_normal_range_is_exact():
    v = _all_bf16()
    a = np.abs(v.astype(np.float64))
    sel = v[(a >= 2.0 ** -14) & (a <= 65504.0)]
    assert sel.size == 30 * 128 * 2          # binades 2^-14 .. 2^15, both signs
    back = oracle.f16.from_f16_bits(oracle.f16.to_f16_bits(sel))
    assert np.array_equal(back, sel.astype(np.float64))


def test_below_normal_range_rounds_half_even_to_2_pow_minus_24():
    v = _all_bf16()
    a = np.abs(v.astype(np.float64))
    sel = v[a < 2.0 ** -14]
    got = oracle.f16.from_f16_bits(oracle.f16.to_f16_bits(sel))
    unit = Fraction(1, 1 << 24)
    for x, g in zip(sel.tolist(), got.tolist()):
        q = Fraction(abs(x)) / unit           # exact multiple count
        k = q.numerator // q.denominator
        rem = q - k
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
            k += 1
        want = float(k * unit) * (1.0 if x >= 0 or (x == 0 and np.signbit(x) == 0) else -1.0)
        assert g == want or (g == 0.0 and want == 0.0), (x, g, want)


def test_decode_is_exact_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.f16.from_f16_bits(bits)
    fin = np.isfinite(vals)
    # re-encoding an exact binary16 value gives the same pattern (up to -0/+0
    # and NaN payloads, which are outside the domain)
    re = oracle.f16.to_f16_bits(vals[fin].astype(np.float32))
    assert np.array_equal(re, bits[fin])


def _f16_cache(hkv, cap, D, rng):
    return rng.integers(0, 1 << 16, size=(hkv, cap, D)).astype(np.uint16)


def test_commit_f16_writes_only_the_accepted_rows():
    rng = np.random.default_rng(3)
    hkv, cap, D, n = 2, 40, 64, 7
    kc, vc = _f16_cache(hkv, cap, D, rng), _f16_cache(hkv, cap, D, rng)
    k0, v0 = kc.copy(), vc.copy()
    kt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32)))
    vt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32)))
    path = [0, 2, 5]
    c = oracle.commit.kv_commit(kc, vc, 30, path, kt, vt, fmt="f16")
    assert c == 33
    for k, node in enumerate(path):
        assert np.array_equal(oracle.f16.from_f16_bits(kc[:, 30 + k]), kt[node].astype(np.float64))
        assert np.array_equal(oracle.f16.from_f16_bits(vc[:, 30 + k]), vt[node].astype(np.float64))
    assert np.array_equal(kc[:, :30], k0[:, :30]) and np.array_equal(kc[:, 33:], k0[:, 33:])
    assert np.array_equal(vc[:, :30], v0[:, :30]) and np.array_equal(vc[:, 33:], v0[:, 33:])
    with pytest.raises(oracle.commit.CapacityError):
        oracle.commit.kv_commit(kc, vc, 38, path, kt, vt, fmt="f16")


@pytest.mark.parametrize("fmt", ["q4_0", "f16"])
@pytest.mark.parametrize("window", [0, 64])
def test_tree_as_cache_chain_is_decode_over_the_committed_cache(fmt, window):
    """A chain whose nodes are all accepted: with the tree rows attended as
    the commit stores them, node i's output is plain softmax attention over
    the committed cache rows [lo, C + i] after the commit."""
    rng = np.random.default_rng(11 + window)
    hkv, hq, D, C, n = 1, 2, 64, 50, 6
    cap = C + n
    kf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    vf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    kc = np.zeros((hkv, cap) + oracle.commit.encode_rows(kf[:, :1], fmt).shape[2:],
                  dtype=oracle.commit.encode_rows(kf[:, :1], fmt).dtype)
    vc = np.zeros_like(kc)
    kc[:, :C] = oracle.commit.encode_rows(kf, fmt)
    vc[:, :C] = oracle.commit.encode_rows(vf, fmt)
    q = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((n, hq, D)).astype(np.float32)))
    kt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32)))
    vt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32)))
    parent = np.arange(-1, n - 1, dtype=np.int32)
    tokens = np.arange(n, dtype=np.int32)
    logits = np.zeros((n, 8), np.float32)
    for i in range(n - 1):
        logits[i, tokens[i + 1]] = 1.0          # every draft accepted
    kcs, vcs = kc.copy(), vc.copy()
    res = oracle.step.verify_step(kcs, vcs, C, window, q, kt, vt, parent, tokens, logits,
                                  fmt=fmt, tree_as_cache=True)
    assert res["accept_len"] == n and res["ctx_len"] == C + n
    scale = 1.0 / np.sqrt(D)
    for i in range(n):
        lo = 0 if window == 0 else max(0, C + i - window + 1)
        keys = oracle.commit.decode_rows(kcs[0, lo:C + i + 1], fmt)
        vals = oracle.commit.decode_rows(vcs[0, lo:C + i + 1], fmt)
        for h in range(hq):
            s = keys @ q[i, h].astype(np.float64) * scale
            p = np.exp(s - s.max())
            want = p @ vals / p.sum()
            assert np.allclose(res["out"][i, h], want, rtol=1e-12, atol=1e-12)


def test_tree_as_cache_f16_equals_default_for_bf16_rows():
    """bf16 tree rows are exact in binary16 (in range), so for the F16 format
    the tree-as-cache reading changes nothing."""
    rng = np.random.default_rng(5)
    kt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((9, 2, 64)).astype(np.float32)))
    vt = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((9, 2, 64)).astype(np.float32)))
    ka, va = oracle.step.tree_rows_attended(kt, vt, "f16", True)
    assert np.array_equal(ka, kt.astype(np.float64)) and np.array_equal(va, vt.astype(np.float64))
