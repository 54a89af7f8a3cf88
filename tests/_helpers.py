"""Shared helpers of the GPU parity tests: moving generator data to the
device and the attention tolerance (max-abs 1e-2, relative L2 2e-3)."""

import numpy as np
import pytest
import torch

import oracle
from tree_verify_attention_gb300 import workload as W

ATOL_MAX = 1e-2
REL_L2 = 2e-3
LSE_ATOL = 2e-3

DEV = "cuda"


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bf16_dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).to(DEV).view(torch.bfloat16)


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def logits_dev(logits):
    if logits.dtype == np.uint16:
        return bf16_dev(logits)
    return torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(DEV)


def oracle_cache(kf, vf, cap):
    """Oracle-quantised cache bytes [Hkv, cap, D/32, 18] with rows [0, C)
    filled from float rows [Hkv, C, D]."""
    hkv, C, D = kf.shape
    kc = np.zeros((hkv, cap, D // 32, 18), np.uint8)
    vc = np.zeros_like(kc)
    kc[:, :C] = oracle.q4_0.quantize_rows(kf)
    vc[:, :C] = oracle.q4_0.quantize_rows(vf)
    return kc, vc


def dequant_window(kc, vc, C, window):
    lo = 0 if window == 0 else max(0, C - window + 1)
    D = kc.shape[2] * 32
    k = np.zeros((kc.shape[0], C, D))
    v = np.zeros_like(k)
    k[:, lo:C] = oracle.q4_0.dequantize_rows(kc[:, lo:C])
    v[:, lo:C] = oracle.q4_0.dequantize_rows(vc[:, lo:C])
    return k, v


def assert_attn_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref).max()
    rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300)
    assert np.all(np.isfinite(gpu)), what
    assert err <= ATOL_MAX and rel <= REL_L2, f"{what}: max_abs {err:.3e} rel_l2 {rel:.3e}"
    return err, rel


def tree_f32(u16):
    return W.bf16_bits_to_f32(u16)
