"""GPU parity of the F16 cache format and of the tree-as-cache reading of the
tree rows, against the oracle, through the C ABI.

Bit-exact: binary16 cache rows (prefill and commit), argmax, accept length,
path, emitted tokens, committed bytes and length. Attention: max-abs 1e-2
and relative L2 2e-3 against the fp64 oracle.

* F16 format: "Luce DFlash ..." (ai-navigate-news, ja) results paragraph
  compares the Q4_0 KV cache against an F16 one; the cache holds binary16
  values written with round-to-nearest-even.
* Tree as cache: the other reading of which tree K/V the attention sees --
  the rows as the commit stores them (tree rows written to the cache before
  attention, rollback by truncation).
"""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from tree_verify_attention_gb300 import api
from tree_verify_attention_gb300 import workload as W

from _helpers import (DEV, LSE_ATOL, assert_attn_close, bf16_dev, i32_dev, logits_dev, need_gpu,
                      tree_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tree_verify_attention_gb300 import build
    build.build()


def _cache_view(cache, fmt):
    """GPU cache bytes as the oracle's arrays: Q4_0 [Hkv, cap, D/32, 18]
    bytes or binary16 bits [Hkv, cap, D]."""
    k = cache.k.cpu().numpy()
    v = cache.v.cpu().numpy()
    if fmt == "f16":
        return (k.view(np.uint16).reshape(cache.n_kv_heads, cache.capacity, cache.head_dim),
                v.view(np.uint16).reshape(cache.n_kv_heads, cache.capacity, cache.head_dim))
    shp = (cache.n_kv_heads, cache.capacity, cache.head_dim // 32, 18)
    return k.reshape(shp), v.reshape(shp)


def _oracle_cache(kf, vf, cap, fmt):
    enc = oracle.commit.encode_rows(kf[:, :1], fmt)
    kc = np.zeros((kf.shape[0], cap) + enc.shape[2:], dtype=enc.dtype)
    vc = np.zeros_like(kc)
    kc[:, :kf.shape[1]] = oracle.commit.encode_rows(kf, fmt)
    vc[:, :kf.shape[1]] = oracle.commit.encode_rows(vf, fmt)
    return kc, vc


def _decode_window(kc, vc, C, window, fmt, D):
    lo = 0 if window == 0 else max(0, C - window + 1)
    k = np.zeros((kc.shape[0], C, D))
    v = np.zeros_like(k)
    k[:, lo:C] = oracle.commit.decode_rows(kc[:, lo:C], fmt)
    v[:, lo:C] = oracle.commit.decode_rows(vc[:, lo:C], fmt)
    return k, v


# ---------------------------------------------------------------- F16 prefill / commit

@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("src_dtype", ["f32", "bf16"])
def test_f16_prefill_bit_exact(D, src_dtype):
    rng = np.random.default_rng(D + 1)
    hkv, n, cap = 3, 131, 140
    x = rng.standard_normal((hkv, n, D)).astype(np.float32)
    x *= rng.choice([1e-6, 1.0, 300.0], size=(hkv, n, 1)).astype(np.float32)
    x[0, 0, :8] = [1.00048828125, 1.00146484375, 2.9802322387695312e-08, -0.0,
                   65280.0, 8.940696716308594e-08, -1.0009765625, 3.1415927410125732]
    if src_dtype == "bf16":
        bits = W.f32_to_bf16_bits(x)
        x = W.bf16_bits_to_f32(bits)
        src = bf16_dev(bits)
    else:
        src = torch.from_numpy(x).to(DEV)
    cache = api.KVCache(hkv, D, cap, fmt="f16")
    cache.k.fill_(0xAB)
    api.kv_quantize_rows(cache.k, src, 5, hkv, D, cap, head_major=True, fmt="f16")
    got, _ = _cache_view(cache, "f16")
    assert np.array_equal(got[:, 5:5 + n], oracle.f16.to_f16_bits(x))
    raw = cache.k.cpu().numpy()
    assert np.all(raw[:, :5] == 0xAB) and np.all(raw[:, 5 + n:] == 0xAB)


@pytest.mark.parametrize("D,hkv", [(64, 1), (128, 2), (256, 4)])
def test_f16_commit_bit_exact(D, hkv):
    rng = np.random.default_rng(D)
    n, C, cap = 12, 50, 80
    cache = api.KVCache(hkv, D, cap, fmt="f16")
    kc = rng.integers(0, 1 << 16, size=(hkv, cap, D)).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, size=(hkv, cap, D)).astype(np.uint16)
    cache.k.copy_(torch.from_numpy(kc.view(np.uint8).reshape(hkv, cap, -1)))
    cache.v.copy_(torch.from_numpy(vc.view(np.uint8).reshape(hkv, cap, -1)))
    cache.ctx_len.fill_(C)
    kt = W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32))
    vt = W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32))
    path = [0, 3, 4, 9]
    pth = np.full(n, -1, np.int32)
    pth[:len(path)] = path
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.kv_commit(cache, i32_dev([len(path)]), i32_dev(pth), bf16_dev(kt), bf16_dev(vt),
                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    newc = oracle.commit.kv_commit(kc, vc, C, path, tree_f32(kt), tree_f32(vt), fmt="f16")
    assert int(cache.ctx_len.item()) == newc == C + len(path)
    gk, gv = _cache_view(cache, "f16")
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)


# ---------------------------------------------------------------- attention

def _attn_case(cfg, C, window, fmt="q4_0", tree_as_cache=False, seed=0, cap_extra=40):
    rng = np.random.default_rng(seed)
    hkv, hq, D, n = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim, cfg.n_nodes
    kf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    vf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    cap = C + cap_extra
    kc, vc = _oracle_cache(kf, vf, cap, fmt)
    s = W.make_step(cfg, seed)
    cache = api.KVCache(hkv, D, cap, fmt=fmt)
    cache.k.copy_(torch.from_numpy(np.ascontiguousarray(kc).view(np.uint8).reshape(hkv, cap, -1)))
    cache.v.copy_(torch.from_numpy(np.ascontiguousarray(vc).view(np.uint8).reshape(hkv, cap, -1)))
    cache.ctx_len.fill_(C)
    out = torch.full((n, hq, D), float("nan"), device=DEV)
    lse = torch.full((n, hq), float("nan"), device=DEV)
    ws = api.workspace(api.attn_workspace_bytes(n, hq, hkv, D, window, cap))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.tree_verify_attn(cache, bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree),
                         i32_dev(s.parent), window, max(cfg.max_depth, n), out, lse, ws,
                         status=status, tree_as_cache=tree_as_cache)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kd, vd = _decode_window(kc, vc, C, window, fmt, D)
    ka, va = oracle.step.tree_rows_attended(tree_f32(s.k_tree), tree_f32(s.v_tree), fmt,
                                            tree_as_cache)
    ref, ref_lse = oracle.attention.tree_verify_attention(
        tree_f32(s.q), kd, vd, ka, va, s.parent, C, window)
    assert_attn_close(out.cpu().numpy(), ref, f"{cfg.name} {fmt} C={C} W={window} tq={tree_as_cache}")
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_ATOL
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("cfg", [W.TINY, W.SHORT], ids=lambda c: c.name)
def test_f16_attention_configs(cfg):
    _attn_case(cfg, cfg.ctx_len, cfg.window, fmt="f16")


@pytest.mark.parametrize("C", [0, 1, 65, 200, 2100])
@pytest.mark.parametrize("window", [0, 64, 2048])
def test_f16_attention_context_and_window_edges(C, window):
    cfg = replace(W.SHORT, n_q_heads=12, n_kv_heads=2)
    _attn_case(cfg, C, window, fmt="f16", seed=C + window)


@pytest.mark.parametrize("D,hq,hkv", [(64, 16, 4), (128, 16, 4), (256, 8, 2)])
def test_f16_attention_multi_chunk_units(D, hq, hkv):
    """F16 rows through the pipelined chunk loop: units of several 128-key
    chunks each (see test_gpu_kernels.test_attention_multi_chunk_units)."""
    cfg = replace(W.SHORT, n_q_heads=hq, n_kv_heads=hkv, head_dim=D)
    _attn_case(cfg, 16000, 0, fmt="f16", seed=D + 1)


@pytest.mark.parametrize("D,hq,hkv", [(64, 4, 1), (128, 8, 2), (128, 32, 4)])
def test_f16_attention_head_dims(D, hq, hkv):
    cfg = replace(W.TINY, head_dim=D, n_q_heads=hq, n_kv_heads=hkv)
    _attn_case(cfg, 300, 0, fmt="f16", seed=D)


@pytest.mark.parametrize("cfg", [W.TINY, W.SHORT], ids=lambda c: c.name)
def test_tree_as_cache_attention_q4_0(cfg):
    got, ref = _attn_case(cfg, cfg.ctx_len, cfg.window, fmt="q4_0", tree_as_cache=True)
    # the variant is a different computation: tree keys differ after quantisation
    base = _attn_case(cfg, cfg.ctx_len, cfg.window, fmt="q4_0", tree_as_cache=False)[1]
    assert np.abs(ref - base).max() > 0


@pytest.mark.parametrize("D,hq,hkv", [(64, 4, 1), (128, 8, 2)])
def test_tree_as_cache_attention_head_dims(D, hq, hkv):
    cfg = replace(W.TINY, head_dim=D, n_q_heads=hq, n_kv_heads=hkv)
    _attn_case(cfg, 300, 0, fmt="q4_0", tree_as_cache=True, seed=D + 7)


def test_tree_as_cache_f16_matches_default():
    cfg = W.TINY
    a, _ = _attn_case(cfg, cfg.ctx_len, cfg.window, fmt="f16", tree_as_cache=True, seed=3)
    b, _ = _attn_case(cfg, cfg.ctx_len, cfg.window, fmt="f16", tree_as_cache=False, seed=3)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- whole steps

class Run:
    """One sequence on both sides, in cache format ``fmt``: the GPU cache
    (filled by the GPU encoder) and the oracle's (filled by the oracle)."""

    def __init__(self, cfg, capacity, fmt, tree_as_cache=False, check_fill=True):
        self.cfg, self.fmt, self.tq = cfg, fmt, tree_as_cache
        kf, vf = W.make_context(cfg)
        self.kc, self.vc = _oracle_cache(kf, vf, capacity, fmt)
        self.cache = api.KVCache(cfg.n_kv_heads, cfg.head_dim, capacity, fmt=fmt)
        self.cache.fill(torch.from_numpy(kf).to(DEV), torch.from_numpy(vf).to(DEV))
        self.C = cfg.ctx_len
        self.step = api.VerifyStep(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                   cfg.window, capacity, cfg.vocab,
                                   max_depth=max(cfg.max_depth, 1))
        if check_fill:
            self.check_cache()

    def check_cache(self, rows=None):
        sl = slice(None) if rows is None else rows
        k, v = _cache_view(self.cache, self.fmt)
        assert np.array_equal(k[:, sl], self.kc[:, sl])
        assert np.array_equal(v[:, sl], self.vc[:, sl])

    def run(self, s, sample=None, by_head=False):
        """One step on both sides; attention compared in full (with
        ``by_head``: through the oracle's per-KV-head form, for long
        contexts), or on the sampled (node, query head) pairs only."""
        cfg = self.cfg
        self.step.status.zero_()
        self.step.run(self.cache, bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree),
                      i32_dev(s.parent), i32_dev(s.tokens), logits_dev(s.logits),
                      tree_as_cache=self.tq)
        torch.cuda.synchronize()
        C0 = self.C
        lg = W.bf16_bits_to_f32(s.logits) if s.logits.dtype == np.uint16 else s.logits
        if sample is not None:
            self.check_sampled(s, C0, sample)
        if by_head:
            ka, va = oracle.step.tree_rows_attended(tree_f32(s.k_tree), tree_f32(s.v_tree),
                                                    self.fmt, self.tq)
            kc, vc, fmt = self.kc, self.vc, self.fmt
            ref_out, ref_lse = oracle.attention.tree_verify_attention_by_head(
                tree_f32(s.q), lambda kv, lo, hi: oracle.commit.decode_rows(kc[kv, lo:hi], fmt),
                lambda kv, lo, hi: oracle.commit.decode_rows(vc[kv, lo:hi], fmt), ka, va,
                s.parent, C0, cfg.window)
        ref = oracle.step.verify_step(self.kc, self.vc, C0, cfg.window, tree_f32(s.q),
                                      tree_f32(s.k_tree), tree_f32(s.v_tree), s.parent,
                                      s.tokens, lg, fmt=self.fmt, tree_as_cache=self.tq,
                                      with_attention=sample is None and not by_head)
        if by_head:
            ref["out"], ref["lse"] = ref_out, ref_lse
        self.C = ref["ctx_len"]
        st = self.step
        L = ref["accept_len"]
        assert int(st.status.item()) == 0
        assert st.argmax.cpu().numpy().tolist() == ref["argmax"].tolist()
        assert int(st.accept_len.item()) == L
        assert st.path.cpu().numpy()[:L].tolist() == ref["path"].tolist()
        assert st.out_tokens.cpu().numpy()[:L].tolist() == ref["out_tokens"].tolist()
        assert int(self.cache.ctx_len.item()) == self.C
        self.check_cache(slice(C0, self.C))
        if sample is None:
            assert_attn_close(st.out.cpu().numpy(), ref["out"], f"{cfg.name} {self.fmt}")
            assert np.abs(st.lse.cpu().numpy() - ref["lse"]).max() <= LSE_ATOL
        return L

    def check_sampled(self, s, C0, pairs):
        cfg = self.cfg
        g = cfg.n_q_heads // cfg.n_kv_heads
        out = self.step.out.cpu().numpy()
        lse = self.step.lse.cpu().numpy()
        lo = 0 if cfg.window == 0 else max(0, C0 - cfg.window + 1)
        ka, va = oracle.step.tree_rows_attended(tree_f32(s.k_tree), tree_f32(s.v_tree), self.fmt,
                                                self.tq)
        deq = {}
        for node, h in pairs:
            kv = h // g
            if kv not in deq:
                k = np.zeros((C0, cfg.head_dim))
                v = np.zeros_like(k)
                k[lo:] = oracle.commit.decode_rows(self.kc[kv, lo:C0], self.fmt)
                v[lo:] = oracle.commit.decode_rows(self.vc[kv, lo:C0], self.fmt)
                deq[kv] = (k, v)
            k, v = deq[kv]
            o, l = oracle.attention.attention_one(tree_f32(s.q)[node, h], k, v, ka[:, kv], va[:, kv],
                                                  s.parent, C0, cfg.window, node)
            assert_attn_close(out[node, h], o, f"{self.fmt} node {node} head {h}")
            assert abs(lse[node, h] - l) <= LSE_ATOL


@pytest.mark.parametrize("fmt,tq", [("f16", False), ("q4_0", True)])
def test_step_tiny_formats(fmt, tq):
    r = Run(W.TINY, W.TINY.ctx_len + 64, fmt, tq)
    for step in range(4):
        r.run(W.make_step(W.TINY, step))


@pytest.mark.parametrize("fmt,tq", [("f16", False), ("q4_0", True)])
def test_step_short_formats(fmt, tq):
    r = Run(W.SHORT, W.SHORT.ctx_len + 100, fmt, tq)
    lens = [r.run(W.make_step(W.SHORT, step)) for step in range(4)]
    assert max(lens) > 1


def test_step_f16_chained_long_context():
    """The 61440-context workload in the F16 format: 12 chained steps, each
    step's commit preceding the next step's attention."""
    cfg = W.LONG_WINDOW
    r = Run(cfg, cfg.ctx_len + 12 * cfg.n_nodes, "f16")
    for step in range(12):
        r.run(W.make_step(cfg, step))
    assert r.C > cfg.ctx_len + 12


@pytest.mark.parametrize("fmt,tq", [("f16", False), ("q4_0", True)])
def test_step_ctx131072_formats(fmt, tq):
    """Full 131072-token context, no window (each attention unit runs many
    key chunks): every (node, query head) attention row against the oracle,
    the rest bit-exactly."""
    cfg = W.FULL_LONG
    r = Run(cfg, cfg.ctx_len + 64, fmt, tq, check_fill=False)
    r.check_cache(slice(0, 2048))
    r.check_cache(slice(cfg.ctx_len - 2048, cfg.ctx_len))
    r.run(W.make_step(cfg, 0), by_head=True)
