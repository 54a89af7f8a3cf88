"""bench.py's workload plumbing on the CPU: every --workload name maps to a
workload config of the stated shape and has a metric, the algorithmic
bytes and FLOPs follow the closed forms, and the sampled oracle timing used
at the 131072-token context runs and reports a per-step time."""

import json
from dataclasses import replace

import numpy as np
import pytest

import bench
from tree_verify_attention_gb300 import workload as W


def test_workload_names_and_shapes():
    assert set(bench.WORKLOADS) == set(bench.METRICS) == {"long", "full", "short"}
    shapes = {"long": (61440, 2048), "full": (131072, 0), "short": (4096, 2048)}
    for name, (ctx, window) in shapes.items():
        cfg, wname = bench.workload_cfg(name)
        assert (cfg.ctx_len, cfg.window) == (ctx, window)
        assert wname == cfg.name
        assert (cfg.n_nodes, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.vocab) == (23, 24, 4, 256, 151936)
    assert bench.workload_cfg("long")[1] == bench.WORKLOAD


@pytest.mark.parametrize("name", ["long", "full", "short"])
def test_algorithmic_bytes_and_flops(name):
    cfg, _ = bench.workload_cfg(name)
    s = W.make_step(cfg, 0)
    kv, lg, flops = bench.algorithmic_per_step(cfg, [s.parent])
    C, Wn, D, hkv, hq, N = cfg.ctx_len, cfg.window, cfg.head_dim, cfg.n_kv_heads, cfg.n_q_heads, cfg.n_nodes
    keys = min(Wn - 1, C) if Wn else C
    assert kv == keys * (D // 32 * 18) * 2 * hkv
    assert lg == N * cfg.vocab * 2
    depth = np.zeros(N, dtype=np.int64)
    for i in range(1, N):
        depth[i] = depth[s.parent[i]] + 1
    # node i sits at position C + depth_i: with a window it sees the committed
    # keys j with C + depth_i - j < W (W - 1 - depth_i of them here), without
    # one all C; plus its ancestors and itself
    committed = np.minimum(C, Wn - 1 - depth) if Wn else np.full(N, C)
    assert flops == pytest.approx(4.0 * D * hq * float(np.sum(committed + depth + 1)))
    if Wn:
        assert flops == pytest.approx(4.0 * D * hq * N * Wn)   # every node sees W keys in all


def test_full_context_is_tensor_bound_by_the_measured_ridge():
    # 469 flop per byte at ctx 131072 against a ridge of about 255 (sustained
    # bf16 / copy bandwidth); the windowed contexts sit far below it
    for name, above in (("full", True), ("long", False), ("short", False)):
        cfg, _ = bench.workload_cfg(name)
        kv, lg, flops = bench.algorithmic_per_step(cfg, [W.make_step(cfg, 0).parent])
        assert (flops / (kv + lg) > 1729.9e12 / 6790.7e9) == above


def test_sampled_oracle_timing_reports_a_step(capsys):
    cfg = replace(W.TINY, ctx_len=512, window=0)
    bench.cpu_oracle_sampled(cfg, 0.05)
    out = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    sp = out["sampled"]
    assert sp["rows_per_step"] == cfg.n_nodes * cfg.n_q_heads
    assert sp["rows_timed"] >= 2 and sp["row_s"] > 0
    step_s = sp["dequant_s"] + sp["row_s"] * sp["rows_per_step"] + sp["accept_commit_s"]
    assert out["seconds"] == pytest.approx(step_s)
    assert out["value"] == pytest.approx(1.0 / step_s)
