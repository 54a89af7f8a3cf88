"""Pins of the oracle's Q4_0 quantiser against hand-derived worked examples,
closed forms and invariants (no GPU)."""

import json
import os

import numpy as np
import pytest

from oracle import q4_0 as Q
from tree_verify_attention_gb300.workload import bf16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_0_worked_examples.json")


def _block(spec):
    x = np.zeros(32, dtype=np.float32)
    for k, v in spec.items():
        x[int(k)] = v
    return x


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_worked_examples(case):
    x = _block(case["x"])
    raw = Q.quantize_rows(x[None])[0, 0]
    assert raw.tobytes().hex() == case["bytes"]
    d16, q = Q.unpack_blocks(raw[None])
    assert float(d16[0]) == case["d"]
    assert np.signbit(d16[0]) == np.signbit(case["d"])


def test_pack_layout_low_then_high_nibble():
    q = np.arange(32, dtype=np.uint8) % 16
    raw = Q.pack_blocks(np.float16([0.5]), q[None])[0]
    for j in range(16):
        assert raw[2 + j] & 0xF == q[j]
        assert raw[2 + j] >> 4 == q[j + 16]
    d16, q2 = Q.unpack_blocks(raw[None])
    assert np.array_equal(q2[0], q)
    assert d16[0] == np.float16(0.5)


def test_dequantize_is_q_minus_8_times_d():
    rng = np.random.default_rng(1)
    q = rng.integers(0, 16, size=(7, 32)).astype(np.uint8)
    d16 = rng.standard_normal(7).astype(np.float16)
    v = Q.dequantize_blocks(d16, q)
    for b in range(7):
        for k in range(32):
            assert v[b * 32 + k] == (int(q[b, k]) - 8) * float(d16[b])


def _all_bf16_in_domain():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bf16_bits_to_f32(bits)
    a = np.abs(vals.astype(np.float64))
    keep = np.isfinite(vals) & (a >= 2.0 ** -120) & (a <= 8 * 65504.0)
    return vals[keep]


def test_exhaustive_single_position_blocks():
    """Every in-domain bf16 value alone in a block, at every position: the
    value maps to code 0, the other 31 positions to 8, and the scale is the
    fp16 rounding of -v/8."""
    vals = _all_bf16_in_domain()
    n = vals.shape[0]
    pos = np.arange(n) % 32
    x = np.zeros((n, 32), dtype=np.float32)
    x[np.arange(n), pos] = vals
    d16, q = Q.quantize_blocks(x)
    d16 = d16[:, 0]
    q = q[:, 0]
    assert np.array_equal(q[np.arange(n), pos], np.zeros(n, dtype=np.uint8))
    mask = np.ones((n, 32), dtype=bool)
    mask[np.arange(n), pos] = False
    assert np.all(q[mask] == 8)
    expect = (vals.astype(np.float64) / -8.0).astype(np.float16)  # exact /8, one fp16 rounding
    assert np.array_equal(d16.view(np.uint16), expect.view(np.uint16))


def test_random_block_invariants():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((4096, 64)) * rng.choice([1e-3, 1.0, 50.0], size=(4096, 1))).astype(np.float32)
    d16, q = Q.quantize_blocks(x)
    blocks = x.reshape(4096, 2, 32)
    assert q.max() <= 15
    # the first element of largest magnitude gets code 0; the scale has the
    # opposite sign of that element
    first = np.argmax(np.abs(blocks), axis=-1)
    assert np.all(np.take_along_axis(q, first[..., None], -1) == 0)
    m = np.take_along_axis(blocks, first[..., None], -1)[..., 0]
    assert np.all(np.sign(d16.astype(np.float64)) == -np.sign(m))
    # reconstruction error: half a step, plus the scale's fp16 rounding
    # (at most 8 * |d| * 2^-11); the clamped code 16 -> 15 loses one step
    xhat = Q.dequantize_blocks(d16, q).reshape(4096, 2, 32)
    d = np.abs(d16.astype(np.float64))[..., None]
    err = np.abs(xhat - blocks)
    clamped = (q == 15) & (blocks * np.sign(m)[..., None] < 0)
    bound = d * 0.5 + 8 * d * 2.0 ** -11 + 1e-30
    assert np.all((err <= bound) | (clamped & (err <= d * 1.5 + 8 * d * 2.0 ** -11)))


def test_idempotent_on_dequantised_values():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2000, 256)).astype(np.float32)
    raw = Q.quantize_rows(x)
    xhat = Q.dequantize_rows(raw).astype(np.float32)   # (q-8)*d is exact in fp32
    assert np.array_equal(Q.quantize_rows(xhat), raw)


def test_zero_block_and_unit_scale():
    raw = Q.quantize_rows(np.zeros((3, 64), dtype=np.float32))
    d16, q = Q.unpack_blocks(raw)
    assert np.all(q == 8) and np.all(d16 == 0)
    assert np.all(Q.dequantize_rows(raw) == 0)
