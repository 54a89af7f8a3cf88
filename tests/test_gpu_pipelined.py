"""GPU parity of the pipelined dependency mode (DFV_STEP_PIPELINED): chains of
verify steps launched back to back, each overlapping the previous kernel of
the stream and waiting for it only before it reads the committed length and
the cache. Checked against the same chain of plain (cooperative) launches,
which must give the same bits everywhere, and against the oracle."""

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


def _dev_inputs(s):
    return (bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree), i32_dev(s.parent),
            i32_dev(s.tokens), logits_dev(s.logits))


def _chain(cfg, cap, pool, n_steps, pipelined, fmt="q4_0", tree_as_cache=False, per_step=True):
    """n_steps chained steps over one cache, launched without a host sync in
    between. per_step: one VerifyStep (outputs and workspaces) per step, so
    that every step's outputs survive; else one object for the whole chain
    (a pipelined one then takes its two workspaces in turn)."""
    kf, vf = W.make_context(cfg)
    cache = api.KVCache(cfg.n_kv_heads, cfg.head_dim, cap, fmt=fmt)
    cache.fill(torch.from_numpy(kf).to(DEV), torch.from_numpy(vf).to(DEV))
    ins = [_dev_inputs(s) for s in pool]

    def make():
        return api.VerifyStep(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                              cfg.window, cap, cfg.vocab, max_depth=max(cfg.max_depth, 1),
                              pipelined=pipelined)

    objs = [make() for _ in range(n_steps)] if per_step else [make()] * n_steps
    torch.cuda.synchronize()
    for i, st in enumerate(objs):
        st.run(cache, *ins[i % len(ins)], tree_as_cache=tree_as_cache)
    torch.cuda.synchronize()
    return cache, objs


def _outputs(st):
    return {k: getattr(st, k).cpu().numpy().copy()
            for k in ("out", "lse", "argmax", "accept_len", "path", "out_tokens", "status")}


def _assert_same(a, b, what):
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), f"{what}: {k} differs"


@pytest.mark.parametrize("fmt,tree_as_cache", [("q4_0", False), ("f16", False), ("q4_0", True)],
                         ids=["q4_0", "f16", "q4_0-tree-as-cache"])
@pytest.mark.parametrize("cfg", [W.TINY, W.SHORT, W.LONG_WINDOW], ids=lambda c: c.name)
def test_pipelined_chain_equals_plain(cfg, fmt, tree_as_cache):
    """Every step's outputs, the committed length and every cache byte are
    bit-identical between the pipelined and the plain chain (the kernel's
    arithmetic and merge order do not depend on the launch mode)."""
    n = 12
    pool = [W.make_step(cfg, i) for i in range(6)]
    cap = cfg.ctx_len + (n + 2) * cfg.n_nodes
    c0, s0 = _chain(cfg, cap, pool, n, False, fmt, tree_as_cache)
    c1, s1 = _chain(cfg, cap, pool, n, True, fmt, tree_as_cache)
    for i in range(n):
        a, b = _outputs(s0[i]), _outputs(s1[i])
        assert int(a["status"][0]) == 0
        _assert_same(a, b, f"step {i}")
    assert int(c0.ctx_len.item()) == int(c1.ctx_len.item()) > cfg.ctx_len + n
    assert torch.equal(c0.k, c1.k) and torch.equal(c0.v, c1.v)


def test_pipelined_chain_oracle_ctx61440():
    """The 60K-context workload, pipelined: 24 chained steps over one cache,
    every step's argmax, walk, outputs and committed bytes bit-exact against
    the oracle's replay, attention in full on four of the steps."""
    cfg = W.LONG_WINDOW
    n = 24
    pool = [W.make_step(cfg, i) for i in range(8)]
    cap = cfg.ctx_len + (n + 2) * cfg.n_nodes
    cache, objs = _chain(cfg, cap, pool, n, True)
    kf, vf = W.make_context(cfg)
    kc, vc = oracle_cache(kf, vf, cap)
    C = cfg.ctx_len
    for i, st in enumerate(objs):
        s = pool[i % len(pool)]
        lg = W.bf16_bits_to_f32(s.logits) if s.logits.dtype == np.uint16 else s.logits
        if i % 8 == 7:
            kd, vd = dequant_window(kc, vc, C, cfg.window)
            ref_out, ref_lse = oracle.attention.tree_verify_attention(
                tree_f32(s.q), kd, vd, tree_f32(s.k_tree), tree_f32(s.v_tree), s.parent, C,
                cfg.window)
            assert_attn_close(st.out.cpu().numpy(), ref_out, f"step {i}")
            assert np.abs(st.lse.cpu().numpy() - ref_lse).max() <= LSE_ATOL
        am = oracle.accept.node_argmax(lg)
        path, toks = oracle.accept.greedy_walk(s.parent, s.tokens, am)
        C = oracle.commit.kv_commit(kc, vc, C, path, tree_f32(s.k_tree), tree_f32(s.v_tree))
        L = len(path)
        assert int(st.status.item()) == 0
        assert st.argmax.cpu().numpy().tolist() == am.tolist()
        assert int(st.accept_len.item()) == L
        assert st.path.cpu().numpy()[:L].tolist() == path.tolist()
        assert st.out_tokens.cpu().numpy()[:L].tolist() == toks.tolist()
    assert int(cache.ctx_len.item()) == C
    k = cache.k.cpu().numpy()
    v = cache.v.cpu().numpy()
    assert np.array_equal(k, kc.reshape(k.shape))
    assert np.array_equal(v, vc.reshape(v.shape))


def test_pipelined_one_object_alternates_workspaces():
    """One pipelined VerifyStep for a 64-step chain (its two workspaces in
    turn) ends with the plain chain's cache, length and last outputs."""
    cfg = W.SHORT
    n = 64
    pool = [W.make_step(cfg, i) for i in range(8)]
    cap = cfg.ctx_len + (n + 2) * cfg.n_nodes
    c0, s0 = _chain(cfg, cap, pool, n, False, per_step=False)
    c1, s1 = _chain(cfg, cap, pool, n, True, per_step=False)
    assert len(s1[0].workspaces) == 2 and len(s0[0].workspaces) == 1
    _assert_same(_outputs(s0[-1]), _outputs(s1[-1]), "last step")
    assert int(s1[-1].status.item()) == 0
    assert int(c0.ctx_len.item()) == int(c1.ctx_len.item())
    assert torch.equal(c0.k, c1.k) and torch.equal(c0.v, c1.v)


def test_pipelined_attention_only():
    """dfv_tree_verify_attn with the pipelined flag, launched right after a
    plain one over the same cache (two workspaces), gives the same bits."""
    cfg = W.SHORT
    s = W.make_step(cfg, 3)
    kf, vf = W.make_context(cfg)
    cap = cfg.ctx_len + 64
    cache = api.Q4Cache(cfg.n_kv_heads, cfg.head_dim, cap)
    cache.fill(torch.from_numpy(kf).to(DEV), torch.from_numpy(vf).to(DEV))
    q, tk, tv, par = bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree), i32_dev(s.parent)
    nb = api.attn_workspace_bytes(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                  cfg.window, cap)
    modes = (False, True, True, False)
    outs = [(torch.empty(cfg.n_nodes, cfg.n_q_heads, cfg.head_dim, dtype=torch.float32,
                         device=DEV),
             torch.empty(cfg.n_nodes, cfg.n_q_heads, dtype=torch.float32, device=DEV),
             torch.zeros(1, dtype=torch.int32, device=DEV), api.workspace(nb))
            for _ in modes]
    torch.cuda.synchronize()
    for pipelined, (out, lse, status, ws) in zip(modes, outs):   # back to back
        api.tree_verify_attn(cache, q, tk, tv, par, cfg.window, cfg.max_depth, out, lse, ws,
                             status=status, pipelined=pipelined)
    torch.cuda.synchronize()
    ref = outs[0]
    assert int(ref[2].item()) == 0
    for o in outs[1:]:
        assert torch.equal(o[0], ref[0]) and torch.equal(o[1], ref[1])
        assert int(o[2].item()) == 0
    kd, vd = dequant_window(*oracle_cache(kf, vf, cap), cfg.ctx_len, cfg.window)
    ref_out, _ = oracle.attention.tree_verify_attention(
        tree_f32(s.q), kd, vd, tree_f32(s.k_tree), tree_f32(s.v_tree), s.parent, cfg.ctx_len,
        cfg.window)
    assert_attn_close(ref[0].cpu().numpy(), ref_out, "attention")
