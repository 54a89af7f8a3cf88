"""IEEE binary16 (F16) KV-cache format, oracle side (test infrastructure only).

[P3] results paragraph compares an F16 KV cache against the Q4_0 one
(acceptance length 8.56 with F16, 8.33 with Q4_0); the pages give no layout.
The adopted reading is the plainest one: an F16 cache row holds the row's D
values as IEEE 754 binary16 numbers, in order, little-endian, so a row of
(head, position) is D * 2 bytes and a cache is ``[Hkv, capacity, D]``
binary16 values.

* Reading a row is exact: every binary16 value is a float64 value.
* Writing a row (commit, prefill) rounds each value to the nearest binary16
  value, ties to the one with an even significand (IEEE roundTiesToEven).

The rounding step uses numpy's float32 -> float16 cast, which is that IEEE
conversion. A bf16 value has 8 significant bits, fewer than binary16's 11,
so every bf16 value in the binary16 normal range [2**-14, 65504] converts
exactly (pinned exhaustively in the tests).

Domain (precondition, not checked): finite inputs of magnitude at most 65504.
"""

import numpy as np


def to_f16_bits(x):
    """binary16 bit patterns (uint16) of float32 values ``x``, rounded to
    nearest, ties to even."""
    x = np.asarray(x, dtype=np.float32)
    return x.astype(np.float16).view(np.uint16)


def from_f16_bits(bits):
    """Exact float64 values of binary16 bit patterns."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def encode_rows(x):
    """Rows of float32 values ([..., D]) as binary16 cache rows (uint16)."""
    return to_f16_bits(x)


def decode_rows(bits):
    """binary16 cache rows ([..., D] uint16) as exact float64 values."""
    return from_f16_bits(bits)
