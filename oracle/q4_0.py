"""Q4_0 block format, oracle side (test infrastructure only).

[P3] feature list and [P5] "What we ported and tuned" name Q4_0 as the KV
cache format but do not spell it out. The format adopted is the GGUF/ggml
Q4_0 block, restated from its definition:

* 32 consecutive values of one row form a block;
* a block stores one fp16 scale ``d`` and 32 unsigned 4-bit codes ``q``;
* a stored block represents the values ``(q_k - 8) * d``.

Quantising a block (the rule is fixed in fp32, and is emulated here with
exact IEEE binary32 numpy operations, each one rounded to nearest-even):

1. ``m`` = the element with the largest magnitude (first one on ties);
2. ``d = m / -8``;
3. ``id = 1 / d`` if ``d != 0`` else ``0``;
4. ``q_k = min(15, trunc((x_k * id) + 8.5))`` -- two separately rounded
   operations, no fused multiply-add;
5. the stored scale is ``d`` rounded to fp16 (nearest-even);
6. byte ``j`` (j = 0..15) holds ``q_j`` in its low nibble and ``q_{j+16}`` in
   its high nibble.

A stored block is 18 bytes: the fp16 scale (little-endian) then the 16 code
bytes. A cache row of ``D`` values is ``D / 32`` consecutive blocks.

Domain (precondition, not checked): finite inputs, every block's largest
magnitude either 0 or at least 2**-120 (so ``1/d`` is finite) and at most
8 * 65504 (so the fp16 scale is finite).
"""

import numpy as np

QK = 32            # values per block
BLOCK_BYTES = 18   # 2-byte fp16 scale + 16 bytes of packed nibbles


def quantize_blocks(x):
    """Quantise ``x`` (float32, last axis a multiple of 32) block by block.

    Returns ``(d16, q)``: ``d16`` float16 of shape ``[..., D/32]`` and ``q``
    uint8 codes in [0, 15] of shape ``[..., D/32, 32]``.
    """
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] % QK:
        raise ValueError("last axis must be a multiple of 32")
    blocks = x.reshape(x.shape[:-1] + (x.shape[-1] // QK, QK))
    # step 1: first element of largest magnitude
    idx = np.argmax(np.abs(blocks), axis=-1)
    m = np.take_along_axis(blocks, idx[..., None], axis=-1)[..., 0]
    # step 2: d = m / -8 (binary32 division)
    d = np.divide(m, np.float32(-8.0), dtype=np.float32)
    # step 3: id = 1/d, 0 for an all-zero block
    inv = np.zeros_like(d)
    nz = d != 0
    inv[nz] = np.divide(np.float32(1.0), d[nz], dtype=np.float32)
    # step 4: two separately rounded binary32 operations, then truncation
    prod = np.multiply(blocks, inv[..., None], dtype=np.float32)
    shifted = np.add(prod, np.float32(8.5), dtype=np.float32)
    q = np.minimum(np.trunc(shifted), np.float32(15.0)).astype(np.uint8)
    # step 5: fp16 scale, nearest-even
    d16 = d.astype(np.float16)
    return d16, q


def pack_blocks(d16, q):
    """Lay out ``(d16, q)`` as 18-byte blocks, shape ``[..., D/32, 18]``."""
    d16 = np.asarray(d16, dtype=np.float16)
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty(d16.shape + (BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = d16.astype("<f2")[..., None].view(np.uint8)
    out[..., 2:] = (q[..., :16] & 0xF) | ((q[..., 16:] & 0xF) << 4)
    return out


def unpack_blocks(raw):
    """Inverse of :func:`pack_blocks`: 18-byte blocks -> ``(d16, q)``."""
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    if raw.shape[-1] != BLOCK_BYTES:
        raise ValueError("blocks must be 18 bytes")
    d16 = raw[..., 0:2].copy().view("<f2")[..., 0].astype(np.float16)
    nib = raw[..., 2:]
    q = np.concatenate([nib & 0xF, nib >> 4], axis=-1).astype(np.uint8)
    return d16, q


def quantize_rows(x):
    """Quantise rows ``x[..., D]`` into packed bytes ``[..., D/32, 18]``."""
    return pack_blocks(*quantize_blocks(x))


def dequantize_blocks(d16, q):
    """Values ``(q - 8) * d`` in float64, shape ``[..., D]``."""
    d = np.asarray(d16, dtype=np.float16).astype(np.float64)
    v = (np.asarray(q, dtype=np.float64) - 8.0) * d[..., None]
    return v.reshape(v.shape[:-2] + (v.shape[-2] * QK,))


def dequantize_rows(raw):
    """Packed bytes ``[..., D/32, 18]`` -> float64 values ``[..., D]``."""
    return dequantize_blocks(*unpack_blocks(raw))
