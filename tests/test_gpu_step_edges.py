"""GPU parity of the fused verify step (dfv_verify_step) on the edges that
the other step tests do not reach: head dims 64 and 128 with the accept and
commit parts (their Q4_0 rows, 36 and 72 bytes, take the non-bulk load
path), a sequence that starts from an empty cache, a cache that the accepted
rows would overflow, and a committed length outside [0, capacity]."""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from tree_verify_attention_gb300 import api
from tree_verify_attention_gb300 import workload as W

from _helpers import DEV, i32_dev, need_gpu
from test_gpu_step import Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tree_verify_attention_gb300 import build
    build.build()


@pytest.mark.parametrize("D,hq,hkv,window", [(64, 4, 1, 0), (64, 8, 2, 100), (128, 8, 2, 0),
                                             (128, 16, 4, 300), (256, 4, 4, 64)])
def test_step_head_dims_chained(D, hq, hkv, window):
    """Three chained steps per head shape, every output and committed byte
    against the oracle, attention in full."""
    cfg = replace(W.SHORT, name=f"d{D}_h{hq}x{hkv}_w{window}", ctx_len=700, window=window,
                  n_q_heads=hq, n_kv_heads=hkv, head_dim=D, vocab=5000)
    r = Run(cfg, cfg.ctx_len + 4 * cfg.n_nodes)
    lens = [r.run(W.make_step(cfg, s)) for s in range(3)]
    assert max(lens) > 1
    r.check_cache()


@pytest.mark.parametrize("D,hq,hkv", [(64, 16, 4), (128, 16, 4)])
def test_step_multi_chunk_units_chained(D, hq, hkv):
    """Three chained whole steps at a context where the attention units
    take several key chunks each, at head dims whose Q4_0 rows are read
    from the cache directly: every output and committed byte against the
    oracle."""
    cfg = replace(W.SHORT, name=f"mc_d{D}_h{hq}x{hkv}", ctx_len=16000, window=0,
                  n_q_heads=hq, n_kv_heads=hkv, head_dim=D, vocab=5000)
    r = Run(cfg, cfg.ctx_len + 4 * cfg.n_nodes)
    lens = [r.run(W.make_step(cfg, s)) for s in range(3)]
    assert max(lens) > 1
    r.check_cache()


class EmptyRun(Run):
    """A sequence whose cache starts empty (ctx_len = 0)."""

    def __init__(self, cfg, capacity):
        self.cfg = cfg
        D = cfg.head_dim
        self.kc = np.zeros((cfg.n_kv_heads, capacity, D // 32, 18), np.uint8)
        self.vc = np.zeros_like(self.kc)
        self.cache = api.Q4Cache(cfg.n_kv_heads, D, capacity)
        self.cache.ctx_len.zero_()
        self.C = 0
        self.step = api.VerifyStep(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, D, cfg.window,
                                   capacity, cfg.vocab, max_depth=max(cfg.max_depth, 1))


@pytest.mark.parametrize("window", [0, 4, 2048])
def test_step_from_empty_cache(window):
    """Steps from C = 0: the first attends to the tree alone, each later one
    also to the rows the earlier ones committed."""
    cfg = replace(W.SHORT, name=f"empty_w{window}", ctx_len=0, window=window, vocab=3000)
    r = EmptyRun(cfg, 8 * cfg.n_nodes)
    for s in range(5):
        r.run(W.make_step(cfg, s))
    assert r.C > 5
    r.check_cache()


def test_step_capacity_overflow_writes_nothing():
    """Accepted rows that would pass the capacity: DFV_DEV_CAPACITY, no row
    written, ctx unchanged; argmax, path and tokens are still produced."""
    cfg = replace(W.SHORT, name="cap_overflow", ctx_len=500, vocab=3000)
    s = W.make_step(cfg, 0)
    lg = W.bf16_bits_to_f32(s.logits)
    am = oracle.accept.node_argmax(lg)
    path, toks = oracle.accept.greedy_walk(s.parent, s.tokens, am)
    L = len(path)
    assert L > 2
    cap = cfg.ctx_len + L - 1                 # one row short
    r = Run(cfg, cap)
    k0, v0 = r.cache.k.clone(), r.cache.v.clone()
    st = r.step
    st.status.zero_()
    st.run(r.cache, *[t for t in (_bf(s.q), _bf(s.k_tree), _bf(s.v_tree), i32_dev(s.parent),
                                   i32_dev(s.tokens), _bf(s.logits))])
    torch.cuda.synchronize()
    assert int(st.status.item()) & api.DEV_CAPACITY
    assert int(r.cache.ctx_len.item()) == cfg.ctx_len
    assert torch.equal(r.cache.k, k0) and torch.equal(r.cache.v, v0)
    assert st.argmax.cpu().numpy().tolist() == am.tolist()
    assert int(st.accept_len.item()) == L
    assert st.path.cpu().numpy()[:L].tolist() == path.tolist()
    assert st.out_tokens.cpu().numpy()[:L].tolist() == toks.tolist()


@pytest.mark.parametrize("bad_ctx", [-5, 10_000])
@pytest.mark.parametrize("pipelined", [False, True])
def test_step_bad_ctx_commits_nothing(bad_ctx, pipelined):
    """A committed length outside [0, capacity] sets DFV_DEV_CTX and, as in
    dfv_kv_commit, nothing is committed: cache bytes and ctx unchanged."""
    cfg = replace(W.SHORT, name="bad_ctx", ctx_len=300, vocab=3000)
    cap = cfg.ctx_len + 2 * cfg.n_nodes
    r = Run(cfg, cap, check_fill=False)
    st = api.VerifyStep(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.window,
                        cap, cfg.vocab, max_depth=cfg.max_depth, pipelined=pipelined)
    s = W.make_step(cfg, 0)
    r.cache.ctx_len.fill_(bad_ctx)
    k0, v0 = r.cache.k.clone(), r.cache.v.clone()
    st.run(r.cache, _bf(s.q), _bf(s.k_tree), _bf(s.v_tree), i32_dev(s.parent),
           i32_dev(s.tokens), _bf(s.logits))
    torch.cuda.synchronize()
    assert int(st.status.item()) & api.DEV_CTX
    assert int(r.cache.ctx_len.item()) == bad_ctx
    assert torch.equal(r.cache.k, k0) and torch.equal(r.cache.v, v0)


def _bf(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).to(DEV).view(torch.bfloat16)
