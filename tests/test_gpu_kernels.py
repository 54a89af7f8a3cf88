"""GPU parity of each entry point against the CPU oracle, through the C ABI.

Bit-exact: Q4_0 bytes (prefill and commit), argmax, accept length, path,
emitted tokens, committed length. Attention: max-abs 1e-2 and relative L2
2e-3 against the fp64 oracle.
"""

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


# ---------------------------------------------------------------- Q4_0 prefill

def _special_blocks():
    rows = []
    for spec in ({0: 8.0, 1: -4.0, 16: 2.0}, {0: -8.0, 1: 8.0}, {}, {0: 3.0, 1: 1.6875},
                 {0: -0.46875, 1: -0.322265625}, {0: -0.0}, {31: 1e-30}, {5: -3e4, 6: 3e4}):
        x = np.zeros(32, np.float32)
        for k, v in spec.items():
            x[k] = v
        rows.append(x)
    return np.concatenate(rows)[None]                  # one row of 8 blocks, D = 256


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("src_dtype", ["f32", "bf16"])
def test_quantize_rows_bit_exact(D, src_dtype):
    rng = np.random.default_rng(D)
    hkv, n, cap = 3, 257, 300
    x = rng.standard_normal((hkv, n, D)).astype(np.float32)
    x *= rng.choice([1e-3, 1.0, 100.0], size=(hkv, n, 1)).astype(np.float32)
    x[0, 0, :] = 0.0
    x[1, 1, ::7] = 2.5           # magnitude ties inside blocks
    x[1, 1, 3::7] = -2.5
    if D == 256:
        x[2, 5] = _special_blocks()[0]
    if src_dtype == "bf16":
        bits = W.f32_to_bf16_bits(x)
        x = W.bf16_bits_to_f32(bits)
        src = bf16_dev(bits)
    else:
        src = torch.from_numpy(x).to(DEV)
    cache = torch.full((hkv, cap, D // 32 * 18), 0xAB, dtype=torch.uint8, device=DEV)
    api.kv_quantize_rows(cache, src, 7, hkv, D, cap, head_major=True)
    got = cache.cpu().numpy().reshape(hkv, cap, D // 32, 18)
    want = oracle.q4_0.quantize_rows(x)
    assert np.array_equal(got[:, 7:7 + n], want)
    assert np.all(got[:, :7] == 0xAB) and np.all(got[:, 7 + n:] == 0xAB)


def test_quantize_rows_token_major_strides():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((40, 2, 128)).astype(np.float32)      # [n, Hkv, D]
    cache = torch.zeros((2, 64, 72), dtype=torch.uint8, device=DEV)
    api.kv_quantize_rows(cache, torch.from_numpy(x).to(DEV), 3, 2, 128, 64)
    got = cache.cpu().numpy().reshape(2, 64, 4, 18)
    assert np.array_equal(got[:, 3:43], oracle.q4_0.quantize_rows(x.transpose(1, 0, 2)))


def test_quantize_rows_rejects_overflow():
    cache = torch.zeros((1, 10, 36), dtype=torch.uint8, device=DEV)
    src = torch.zeros((1, 5, 64), device=DEV)
    with pytest.raises(api.DfvError):
        api.kv_quantize_rows(cache, src, 6, 1, 64, 10, head_major=True)


# ---------------------------------------------------------------- commit

def _commit_case(D, hkv, n, C, cap, path, seed=0):
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 256, size=(hkv, cap, D // 32, 18)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(hkv, cap, D // 32, 18)).astype(np.uint8)
    kt = W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32))
    vt = W.f32_to_bf16_bits(rng.standard_normal((n, hkv, D)).astype(np.float32))
    kt[0, 0, :32] = 0
    cache = api.Q4Cache(hkv, D, cap)
    cache.k.copy_(torch.from_numpy(kc.reshape(hkv, cap, -1)))
    cache.v.copy_(torch.from_numpy(vc.reshape(hkv, cap, -1)))
    cache.ctx_len.fill_(C)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pth = np.full(n, -1, np.int32)
    pth[:len(path)] = path
    api.kv_commit(cache, i32_dev([len(path)]), i32_dev(pth), bf16_dev(kt), bf16_dev(vt),
                  status=status)
    torch.cuda.synchronize()
    return kc, vc, kt, vt, cache, int(status.item())


@pytest.mark.parametrize("D,hkv", [(64, 1), (128, 2), (256, 4)])
def test_commit_bit_exact(D, hkv):
    path = [0, 3, 4, 9]
    kc, vc, kt, vt, cache, st = _commit_case(D, hkv, 12, 50, 80, path)
    assert st == 0
    newc = oracle.commit.kv_commit(kc, vc, 50, path, tree_f32(kt), tree_f32(vt))
    assert int(cache.ctx_len.item()) == newc == 54
    assert np.array_equal(cache.k.cpu().numpy().reshape(kc.shape), kc)
    assert np.array_equal(cache.v.cpu().numpy().reshape(vc.shape), vc)


def test_commit_capacity_overflow_writes_nothing():
    path = [0, 1, 2]
    kc, vc, kt, vt, cache, st = _commit_case(256, 4, 5, 78, 80, path)
    assert st & api.DEV_CAPACITY
    assert int(cache.ctx_len.item()) == 78
    assert np.array_equal(cache.k.cpu().numpy().reshape(kc.shape), kc)


def test_commit_bad_path_writes_nothing():
    kc, vc, kt, vt, cache, st = _commit_case(256, 4, 5, 10, 80, [0, 7])
    assert st & api.DEV_BAD_PATH
    assert int(cache.ctx_len.item()) == 10
    assert np.array_equal(cache.v.cpu().numpy().reshape(vc.shape), vc)


# ---------------------------------------------------------------- argmax + walk

def _run_accept(logits, parent, tokens):
    n = logits.shape[0]
    ws = api.workspace(api.accept_workspace_bytes(n, logits.shape[1]))
    out = {k: torch.full((n,), -7, dtype=torch.int32, device=DEV)
           for k in ("argmax", "path", "out_tokens")}
    acc = torch.zeros(1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lg = logits_dev(logits)
    for _ in range(2):    # the second call checks that the workspace was left reusable
        api.greedy_accept(lg, i32_dev(parent), i32_dev(tokens), out["argmax"], acc, out["path"],
                          out["out_tokens"], ws, status=status)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["accept_len"] = int(acc.item())
    res["status"] = int(status.item())
    return res


def _check_accept(logits, parent, tokens):
    got = _run_accept(logits, parent, tokens)
    lg = W.bf16_bits_to_f32(logits) if logits.dtype == np.uint16 else logits
    am = oracle.accept.node_argmax(lg)
    path, toks = oracle.accept.greedy_walk(parent, tokens, am)
    L = len(path)
    assert got["status"] == 0
    assert got["argmax"].tolist() == am.tolist()
    assert got["accept_len"] == L
    assert got["path"][:L].tolist() == path.tolist() and np.all(got["path"][L:] == -1)
    assert got["out_tokens"][:L].tolist() == toks.tolist() and np.all(got["out_tokens"][L:] == -1)
    return L


@pytest.mark.parametrize("cfg", [W.TINY, W.SHORT], ids=lambda c: c.name)
def test_accept_configs(cfg):
    for step in range(3):
        s = W.make_step(cfg, step)
        _check_accept(s.logits, s.parent, s.tokens)


@pytest.mark.parametrize("budget", [0, 8, 22, 48, 64])
@pytest.mark.parametrize("shape", ["chain", "kary2", "kary4", "random"])
def test_accept_sweep_shapes(budget, shape):
    cfgs = [c for c in W.sweep_configs() if c.budget == budget and c.tree == shape and c.seed < 2]
    for c in cfgs:
        s = W.make_step(c)
        _check_accept(s.logits, s.parent, s.tokens)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_ties_and_edges(dtype):
    V, n = 151936, 9
    chunks = api.accept_workspace_bytes(n, V)   # exercise the query
    assert chunks > 0
    rng = np.random.default_rng(4)
    x = rng.standard_normal((n, V)).astype(np.float32)
    # ties at every plausible chunk / vector / lane boundary of row 0
    for k in (8191, 8192, 8200, 16383, 16384, 75968, 151935):
        x[0, k] = 6.0
    x[1] = 1.0                                   # all equal
    x[2] = -np.inf
    x[3, :] = -1.0
    x[3, 777] = 0.0
    x[3, 500] = -0.0                             # -0 before +0: 500 wins
    x[4, V - 1] = 9.0                            # max at the end
    x[5, 0] = 9.0                                # max at the start
    x[6, 100000] = 7.0
    x[6, 99999] = 7.0
    x[7] = -3.0                                  # negative maxima tied across chunks
    x[7, 40000] = -2.5
    x[7, 120000] = -2.5
    x[8] = -1.0                                  # -0 and +0 in different chunks: 10000 wins
    x[8, 30000] = 0.0
    x[8, 10000] = -0.0
    parent = np.array([-1, 0, 0, 1, 1, 2, 5, 5, 0], np.int32)
    tokens = np.zeros(n, np.int32)
    logits = W.f32_to_bf16_bits(x) if dtype == "bf16" else x
    _check_accept(logits, parent, tokens)


def test_walk_duplicate_siblings_and_bad_tree():
    V = 1024
    logits = np.zeros((4, V), np.float32)
    logits[0, 7] = 1.0
    logits[2, 5] = 1.0
    parent = np.array([-1, 0, 0, 2], np.int32)
    tokens = np.array([0, 7, 7, 5], np.int32)
    L = _check_accept(logits, parent, tokens)
    assert L == 2                                 # child 1 wins over child 2
    bad = np.array([-1, 0, 5, 1], np.int32)       # parent[2] out of range
    got = _run_accept(logits, bad, tokens)
    assert got["status"] & api.DEV_BAD_TREE


@pytest.mark.parametrize("V", [1, 7, 1000, 2049, 151936])
def test_argmax_odd_vocab_sizes(V):
    rng = np.random.default_rng(V)
    x = rng.integers(-2, 3, size=(5, V)).astype(np.float32)
    _check_accept(x, np.array([-1, 0, 1, 2, 3], np.int32), np.zeros(5, np.int32))
    # unaligned rows for bf16 when V is odd
    _check_accept(W.f32_to_bf16_bits(x), np.array([-1, 0, 1, 2, 3], np.int32),
                  np.zeros(5, np.int32))


# ---------------------------------------------------------------- attention

def _attn_case(cfg, C, window, parent=None, seed=0, cap_extra=40):
    rng = np.random.default_rng(seed)
    hkv, hq, D, n = cfg.n_kv_heads, cfg.n_q_heads, cfg.head_dim, cfg.n_nodes
    kf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    vf = rng.standard_normal((hkv, C, D)).astype(np.float32)
    cap = C + cap_extra
    kc, vc = oracle_cache(kf, vf, cap)
    s = W.make_step(cfg, seed)
    if parent is None:
        parent = s.parent
    cache = api.Q4Cache(hkv, D, cap)
    cache.k.copy_(torch.from_numpy(kc.reshape(hkv, cap, -1)))
    cache.v.copy_(torch.from_numpy(vc.reshape(hkv, cap, -1)))
    cache.ctx_len.fill_(C)
    out = torch.full((n, hq, D), float("nan"), device=DEV)
    lse = torch.full((n, hq), float("nan"), device=DEV)
    ws = api.workspace(api.attn_workspace_bytes(n, hq, hkv, D, window, cap))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.tree_verify_attn(cache, bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree),
                         i32_dev(parent), window, max(cfg.max_depth, n), out, lse, ws,
                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kd, vd = dequant_window(kc, vc, C, window)
    ref, ref_lse = oracle.attention.tree_verify_attention(
        tree_f32(s.q), kd, vd, tree_f32(s.k_tree), tree_f32(s.v_tree), parent, C, window)
    got = out.cpu().numpy()
    assert_attn_close(got, ref, f"{cfg.name} C={C} W={window}")
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_ATOL
    return got, ref


def test_attention_tiny():
    _attn_case(W.TINY, W.TINY.ctx_len, 0)


def test_attention_short():
    _attn_case(W.SHORT, W.SHORT.ctx_len, W.SHORT.window)


@pytest.mark.parametrize("C", [0, 1, 63, 64, 65, 200, 2100])
@pytest.mark.parametrize("window", [0, 3, 64, 2048])
def test_attention_context_and_window_edges(C, window):
    from dataclasses import replace
    cfg = replace(W.SHORT, n_q_heads=8, n_kv_heads=2, budget=12)
    _attn_case(cfg, C, window, seed=C + window)


@pytest.mark.parametrize("D,hq,hkv", [(64, 4, 1), (128, 8, 2), (256, 6, 1), (128, 32, 4)])
def test_attention_head_dims_and_groups(D, hq, hkv):
    from dataclasses import replace
    cfg = replace(W.SHORT, n_q_heads=hq, n_kv_heads=hkv, head_dim=D)
    _attn_case(cfg, 700, 300)


@pytest.mark.parametrize("D,hq,hkv", [(64, 16, 4), (128, 16, 4), (256, 8, 2)])
@pytest.mark.parametrize("window", [0, 5000])
def test_attention_multi_chunk_units(D, hq, hkv, window):
    """Contexts long enough that the attention units take several 128-key
    chunks each (the pipelined chunk loop: the next chunk's rows read and
    decoded while the current one's P V runs): 4 KV heads x 1 row tile x
    126 chunks cannot give every split one chunk on any GPU of up to 256
    SMs. At head dims 64 and 128 the Q4_0 rows are read from the cache
    directly, at 256 through the staged copies."""
    from dataclasses import replace
    cfg = replace(W.SHORT, n_q_heads=hq, n_kv_heads=hkv, head_dim=D)
    _attn_case(cfg, 16000, window, seed=D + window)


@pytest.mark.parametrize("budget", [0, 8, 22, 48, 64])
@pytest.mark.parametrize("shape", ["chain", "kary4", "random"])
def test_attention_sweep_shapes(budget, shape):
    c = [x for x in W.sweep_configs() if x.budget == budget and x.tree == shape][0]
    from dataclasses import replace
    c = replace(c, ctx_len=2600)
    _attn_case(c, c.ctx_len, c.window)


def test_attention_long_window_equals_none():
    from dataclasses import replace
    cfg = replace(W.SHORT, n_q_heads=8, n_kv_heads=2)
    a, _ = _attn_case(cfg, 500, 0, seed=3)
    b, _ = _attn_case(cfg, 500, 500 + 17, seed=3)
    assert np.array_equal(a, b)


def test_attention_bad_tree_reports():
    cfg = W.TINY
    parent = W.make_step(cfg).parent.copy()
    parent[3] = 7
    rng = np.random.default_rng(0)
    cache = api.Q4Cache(1, 64, 100)
    cache.ctx_len.fill_(10)
    s = W.make_step(cfg)
    out = torch.empty((9, 4, 64), device=DEV)
    ws = api.workspace(api.attn_workspace_bytes(9, 4, 1, 64, 0, 100))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.tree_verify_attn(cache, bf16_dev(s.q), bf16_dev(s.k_tree), bf16_dev(s.v_tree),
                         i32_dev(parent), 0, 1, out, None, ws, status=status)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & api.DEV_BAD_TREE and st & api.DEV_DEPTH
    assert torch.isfinite(out).all()
