"""GPU parity of the whole verify step (dfv_verify_step) against the oracle:
single steps, the chained 61440-context replay, the 131072-context step
(every attention row) and the tree-shape sweep at context 32768."""

import time
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from tree_verify_attention_gb300 import api
from tree_verify_attention_gb300 import workload as W

from _helpers import (DEV, LSE_ATOL, assert_attn_close, bf16_dev, dequant_window, i32_dev,
                      logits_dev, need_gpu, oracle_cache, tree_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tree_verify_attention_gb300 import build
    build.build()


class Run:
    """One sequence on both sides: the GPU cache (filled by the GPU
    quantiser) and the oracle's cache (filled by the oracle quantiser)."""

    def __init__(self, cfg, capacity, check_fill=True):
        self.cfg = cfg
        kf, vf = W.make_context(cfg)
        self.kc, self.vc = oracle_cache(kf, vf, capacity)
        self.cache = api.Q4Cache(cfg.n_kv_heads, cfg.head_dim, capacity)
        self.cache.fill(torch.from_numpy(kf).to(DEV), torch.from_numpy(vf).to(DEV))
        self.C = cfg.ctx_len
        self.step = api.VerifyStep(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                   cfg.window, capacity, cfg.vocab,
                                   max_depth=max(cfg.max_depth, 1))
        if check_fill:
            self.check_cache()

    def check_cache(self, rows=None):
        sl = slice(None) if rows is None else rows
        k = self.cache.k[:, sl].cpu().numpy()
        v = self.cache.v[:, sl].cpu().numpy()
        assert np.array_equal(k, self.kc[:, sl].reshape(k.shape))
        assert np.array_equal(v, self.vc[:, sl].reshape(v.shape))

    def run(self, s, with_attention=True, sample=None, by_head=False):
        cfg = self.cfg
        self.step.status.zero_()
        self.step.run(self.cache, bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree),
                      i32_dev(s.parent), i32_dev(s.tokens), logits_dev(s.logits))
        torch.cuda.synchronize()
        C0 = self.C
        lg = W.bf16_bits_to_f32(s.logits) if s.logits.dtype == np.uint16 else s.logits
        want_attn = with_attention and sample is None
        if want_attn and by_head:
            # every (node, query head) row, one KV head's rows dequantised at a time
            kc, vc = self.kc, self.vc
            ref_out, ref_lse = oracle.attention.tree_verify_attention_by_head(
                tree_f32(s.q), lambda kv, lo, hi: oracle.q4_0.dequantize_rows(kc[kv, lo:hi]),
                lambda kv, lo, hi: oracle.q4_0.dequantize_rows(vc[kv, lo:hi]),
                tree_f32(s.k_tree), tree_f32(s.v_tree), s.parent, C0, cfg.window)
        elif want_attn:
            kd, vd = dequant_window(self.kc, self.vc, C0, cfg.window)
            ref_out, ref_lse = oracle.attention.tree_verify_attention(
                tree_f32(s.q), kd, vd, tree_f32(s.k_tree), tree_f32(s.v_tree), s.parent, C0,
                cfg.window)
        am = oracle.accept.node_argmax(lg)
        path, toks = oracle.accept.greedy_walk(s.parent, s.tokens, am)
        self.C = oracle.commit.kv_commit(self.kc, self.vc, C0, path, tree_f32(s.k_tree),
                                         tree_f32(s.v_tree))
        st = self.step
        L = len(path)
        assert int(st.status.item()) == 0
        assert st.argmax.cpu().numpy().tolist() == am.tolist()
        assert int(st.accept_len.item()) == L
        assert st.path.cpu().numpy()[:L].tolist() == path.tolist()
        assert st.out_tokens.cpu().numpy()[:L].tolist() == toks.tolist()
        assert int(self.cache.ctx_len.item()) == self.C
        self.check_cache(slice(C0, self.C))
        if want_attn:
            assert_attn_close(st.out.cpu().numpy(), ref_out, cfg.name)
            assert np.abs(st.lse.cpu().numpy() - ref_lse).max() <= LSE_ATOL
        elif with_attention:
            self.check_sampled(s, C0, sample)
        return L

    def check_sampled(self, s, C0, pairs):
        cfg = self.cfg
        g = cfg.n_q_heads // cfg.n_kv_heads
        out = self.step.out.cpu().numpy()
        lse = self.step.lse.cpu().numpy()
        lo = 0 if cfg.window == 0 else max(0, C0 - cfg.window + 1)
        deq = {}
        for node, h in pairs:
            kv = h // g
            if kv not in deq:
                k = np.zeros((C0, cfg.head_dim))
                v = np.zeros_like(k)
                k[lo:] = oracle.q4_0.dequantize_rows(self.kc[kv, lo:C0])
                v[lo:] = oracle.q4_0.dequantize_rows(self.vc[kv, lo:C0])
                deq[kv] = (k, v)
            k, v = deq[kv]
            o, l = oracle.attention.attention_one(
                tree_f32(s.q)[node, h], k, v, tree_f32(s.k_tree)[:, kv], tree_f32(s.v_tree)[:, kv],
                s.parent, C0, cfg.window, node)
            assert_attn_close(out[node, h], o, f"node {node} head {h}")
            assert abs(lse[node, h] - l) <= LSE_ATOL


def test_step_tiny():
    r = Run(W.TINY, W.TINY.ctx_len + 64)
    for step in range(5):
        r.run(W.make_step(W.TINY, step))
    r.check_cache()


def test_step_short():
    r = Run(W.SHORT, W.SHORT.ctx_len + 100)
    lens = [r.run(W.make_step(W.SHORT, step)) for step in range(4)]
    assert max(lens) > 1
    r.check_cache()


@pytest.mark.parametrize("budget", [0, 8, 22, 48, 64])
@pytest.mark.parametrize("shape", ["chain", "kary2", "kary4", "random"])
def test_step_sweep_ctx32768(budget, shape):
    """Tree-shape sweep at context 32768, window 2048 (one seed and p per
    shape here; the accept-only sweep covers every seed and p)."""
    cfg = [c for c in W.sweep_configs()
           if c.budget == budget and c.tree == shape and c.p_accept == 0.8 and c.seed == budget % 5][0]
    r = Run(cfg, cfg.ctx_len + 2 * cfg.n_nodes, check_fill=False)
    r.check_cache(slice(cfg.ctx_len - 2100, cfg.ctx_len))
    for step in range(2):
        r.run(W.make_step(cfg, step))


def test_chained_steps_ctx61440():
    """The 60K-context workload: 1000 chained verify + commit steps on one
    cache, each step appending its accepted rows before the next, every step
    with freshly generated inputs (tree, tokens, queries, tree rows, logits).
    Every step is checked bit-exactly; attention is checked in full every 25
    steps and on the last."""
    cfg = W.LONG_WINDOW
    steps = cfg.steps
    cap = cfg.ctx_len + steps * cfg.n_nodes
    r = Run(cfg, cap)
    t0 = time.time()
    for step in range(steps):
        r.run(W.make_step(cfg, step), with_attention=(step % 25 == 0 or step == steps - 1),
              by_head=True)
    r.check_cache()
    assert r.C > cfg.ctx_len + steps            # the planted paths were accepted
    print(f"1000 chained steps: final ctx {r.C}, {time.time() - t0:.1f}s")


def test_step_ctx131072():
    """Full 131072-token context, no window: every (node, query head) row of
    the attention against the oracle (per KV head), the rest bit-exactly;
    two chained steps."""
    cfg = W.FULL_LONG
    r = Run(cfg, cfg.ctx_len + 64, check_fill=False)
    r.check_cache(slice(0, 4096))
    r.check_cache(slice(cfg.ctx_len - 4096, cfg.ctx_len))
    for step in range(2):
        r.run(W.make_step(cfg, step), by_head=True)


def _edge_logits(logits, bf16):
    """Rows that probe the per-node argmax: ties across the vocabulary (the
    lowest index wins), an all -inf row (index 0), the maximum only at the last
    index, and equal signed zeros as the maximum (the lower index wins)."""
    lg = logits.copy()
    V = lg.shape[1]
    if bf16:
        hi, low, ninf, pz, nz = 0x41F0, 0xC0A0, 0xFF80, 0x0000, 0x8000   # 30, -5, -inf, +0, -0
    else:
        hi, low, ninf, pz, nz = (np.float32(30.0), np.float32(-5.0), np.float32(-np.inf),
                                 np.float32(0.0), np.float32(-0.0))
    lg[0, :] = low
    lg[0, [V // 3, V // 2, V - 1]] = hi
    lg[1, :] = ninf
    lg[2, :] = low
    lg[2, V - 1] = hi
    lg[3, :] = low
    lg[3, ::7] = hi                                         # ties in every slice
    lg[4, :] = low
    lg[4, [V // 5, V // 7]] = [nz, pz]                      # -0 after +0 ... lowest index is V // 7
    lg[5, :] = low
    lg[5, [V // 9, V // 4]] = [nz, pz]                      # -0 first
    return lg


@pytest.mark.parametrize("cfg", [W.SHORT, W.TINY], ids=lambda c: c.name)
def test_step_argmax_edges(cfg):
    r = Run(cfg, cfg.ctx_len + 128, check_fill=False)
    s = W.make_step(cfg, 7)
    s = replace(s, logits=_edge_logits(s.logits, s.logits.dtype == np.uint16))
    r.run(s)
    am = r.step.argmax.cpu().numpy()
    V = cfg.vocab
    assert am[0] == V // 3 and am[1] == 0 and am[2] == V - 1 and am[3] == 0
    assert am[4] == V // 7 and am[5] == V // 9
