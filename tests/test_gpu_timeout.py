"""Failure detection of the fused verify step without a GPU fault.

Every wait between CTAs of the step is bounded by the GPU's global timer
(100 ms); when one runs out the kernel sets DFV_DEV_TIMEOUT, skips the work
that depended on it and returns, leaving the context usable. These tests make
a wait run out by corrupting the step's workspace from the host (no kernel is
altered and nothing faults):

* the walker waits until exactly grid - 1 CTAs have reported that they read
  the committed length; a report count preset far above that can never equal
  it, so the walker gives up and commits nothing;
* the splits of a (KV head, tile) group derive one generation tag from the
  group's arrival word (arrivals in the low 16 bits, the generation above);
  an arrival count preset just below 2^16 carries into the generation in the
  middle of the arrivals, the splits' tags then disagree and the merge waits
  run out.

After each, the workspace is cleared (as the header asks after a timeout) and
a clean step must match the oracle again."""

import time

import numpy as np
import pytest
import torch

import oracle
from tree_verify_attention_gb300 import api
from tree_verify_attention_gb300 import workload as W

from _helpers import (DEV, assert_attn_close, bf16_dev, i32_dev, logits_dev, need_gpu,
                      oracle_cache, tree_f32)

pytestmark = pytest.mark.gpu

DEV_TIMEOUT = 0x20


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tree_verify_attention_gb300 import build
    build.build()


def _setup(cfg, cap):
    kf, vf = W.make_context(cfg)
    kc, vc = oracle_cache(kf, vf, cap)
    cache = api.Q4Cache(cfg.n_kv_heads, cfg.head_dim, cap)
    cache.fill(torch.from_numpy(kf).to(DEV), torch.from_numpy(vf).to(DEV))
    st = api.VerifyStep(cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.window,
                        cap, cfg.vocab, max_depth=cfg.max_depth)
    return kc, vc, cache, st


def _run(st, cache, s):
    st.status.zero_()
    t0 = time.time()
    st.run(cache, bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree), i32_dev(s.parent),
           i32_dev(s.tokens), logits_dev(s.logits))
    torch.cuda.synchronize()
    return time.time() - t0


def _check_clean_step(cfg, kc, vc, cache, st, s):
    """A step after the workspace was cleared: bit-exact acceptance and
    commit, attention within tolerance."""
    api.clear_workspace(st.ws)
    C0 = int(cache.ctx_len.item())
    _run(st, cache, s)
    lg = W.bf16_bits_to_f32(s.logits) if s.logits.dtype == np.uint16 else s.logits
    ref = oracle.step.verify_step(kc, vc, C0, cfg.window, tree_f32(s.q), tree_f32(s.k_tree),
                                  tree_f32(s.v_tree), s.parent, s.tokens, lg)
    assert int(st.status.item()) == 0
    L = ref["accept_len"]
    assert int(st.accept_len.item()) == L
    assert st.path.cpu().numpy()[:L].tolist() == ref["path"].tolist()
    assert int(cache.ctx_len.item()) == ref["ctx_len"]
    k = cache.k.cpu().numpy().reshape(kc.shape)
    assert np.array_equal(k, kc) and np.array_equal(cache.v.cpu().numpy().reshape(vc.shape), vc)
    assert_attn_close(st.out.cpu().numpy(), ref["out"], "clean step after a timeout")


def test_walker_wait_times_out_and_commits_nothing():
    cfg = W.SHORT
    cap = cfg.ctx_len + 64
    kc, vc, cache, st = _setup(cfg, cap)
    s = W.make_step(cfg, 0)
    k0, v0 = cache.k.clone(), cache.v.clone()
    C0 = int(cache.ctx_len.item())
    ws = st.ws.view(torch.int32)
    ws[2] = 1 << 30            # the walker's report count: can never equal grid - 1
    dt = _run(st, cache, s)
    status = int(st.status.item())
    assert status & DEV_TIMEOUT, hex(status)
    assert 0.05 <= dt < 10.0, dt                   # bounded by the 100 ms limit, not hung
    assert int(cache.ctx_len.item()) == C0          # nothing committed
    assert torch.equal(cache.k, k0) and torch.equal(cache.v, v0)
    # the attention does not depend on the walker and still matches the oracle
    kd = np.zeros((cfg.n_kv_heads, C0, cfg.head_dim))
    vd = np.zeros_like(kd)
    lo = max(0, C0 - cfg.window + 1)
    kd[:, lo:] = oracle.q4_0.dequantize_rows(kc[:, lo:C0])
    vd[:, lo:] = oracle.q4_0.dequantize_rows(vc[:, lo:C0])
    ref_out, _ = oracle.attention.tree_verify_attention(
        tree_f32(s.q), kd, vd, tree_f32(s.k_tree), tree_f32(s.v_tree), s.parent, C0, cfg.window)
    assert_attn_close(st.out.cpu().numpy(), ref_out, "attention beside a timed-out walker")
    _check_clean_step(cfg, kc, vc, cache, st, W.make_step(cfg, 1))


def test_split_group_wait_times_out():
    cfg = W.SHORT
    cap = cfg.ctx_len + 64
    kc, vc, cache, st = _setup(cfg, cap)
    s = W.make_step(cfg, 2)
    ws = st.ws.view(torch.int32)
    # group 0's arrival word: the count carries into the generation after
    # the eighth arrival, so the later splits tag their partials differently
    ws[4] = 0xFFF8
    dt = _run(st, cache, s)
    status = int(st.status.item())
    assert status & DEV_TIMEOUT, hex(status)
    assert 0.05 <= dt < 10.0, dt
    # the walk and commit do not depend on the merge: the committed rows are
    # the oracle's
    C0 = cfg.ctx_len
    lg = W.bf16_bits_to_f32(s.logits)
    am = oracle.accept.node_argmax(lg)
    path, _ = oracle.accept.greedy_walk(s.parent, s.tokens, am)
    C1 = oracle.commit.kv_commit(kc, vc, C0, path, tree_f32(s.k_tree), tree_f32(s.v_tree))
    assert int(cache.ctx_len.item()) == C1
    assert st.argmax.cpu().numpy().tolist() == am.tolist()
    k = cache.k.cpu().numpy().reshape(kc.shape)
    assert np.array_equal(k, kc) and np.array_equal(cache.v.cpu().numpy().reshape(vc.shape), vc)
    _check_clean_step(cfg, kc, vc, cache, st, W.make_step(cfg, 3))
