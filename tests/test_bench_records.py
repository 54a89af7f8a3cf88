"""bench.py's use of the committed ncu record (CPU): the kernel source hash
ignores comments and whitespace but not code, and the recorded DRAM traffic
is reported only for the run it was taken on."""

import os
import shutil

import bench


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "tree_verify_attention_gb300", "csrc"),
                    root / "tree_verify_attention_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    return root


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    step = root / "tree_verify_attention_gb300" / "csrc" / "step.cu"
    text = step.read_text()
    step.write_text("// a new leading comment\n/* and a block\n   comment */\n" +
                    text.replace("\n", "\n  ", 3))
    assert bench.kernel_source_hash() == h0
    step.write_text(text.replace("kRescaleLog2 = 8.0f", "kRescaleLog2 = 7.0f"))
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_only_for_its_own_run(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    # one record per workload, each opened by its "workload:" line
    recs, cur = {}, None
    for line in open(root / "profiles" / "step_kernel_traffic.txt"):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            k, v = k.strip(), v.strip()
            if k == "workload":
                cur = recs.setdefault(v, {})
            elif cur is not None:
                cur[k] = v
    assert bench.WORKLOAD in recs
    for wname, rec in recs.items():
        if rec["source_hash"] == bench.kernel_source_hash():
            assert bench.recorded_traffic("q4_0", False, wname) == int(rec["dram_bytes_per_launch"])
    assert bench.recorded_traffic("q4_0", False, "no_such_workload") is None
    assert bench.recorded_traffic("f16") is None
    assert bench.recorded_traffic("q4_0", tree_as_cache=True) is None
    step = root / "tree_verify_attention_gb300" / "csrc" / "step.cu"
    step.write_text(step.read_text().replace("kRescaleLog2 = 8.0f", "kRescaleLog2 = 7.0f"))
    for wname in recs:
        assert bench.recorded_traffic("q4_0", False, wname) is None
