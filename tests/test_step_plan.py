"""Host-side invariants of the verify step's launch plan (no GPU): builds
tests/step_plan_check.cu (the step kernel's translation unit plus a host
main, device code only to PTX) and runs it over shapes from head dim 64 to
256, 1 to 65 nodes, vocabularies from 1 to 262144 and both logits types, on
devices of 100 to 300 SMs (the grid is capped at 256 CTAs).
Checked there: the 128-row tiles cover every row, every logits slice is
staged by exactly one CTA (a CTA without a unit, or a unit of a tile of at
most 32 rows, which stages one round in the smem its tile leaves free), a
round of staged slices fits half of a staging area, bulk-copied slices
stay 16-byte aligned, the argmax partials fit the walker's Q tile, the
walker holds no attention unit, the split merge's staging fits, and the
workspace regions are ordered, aligned and large enough."""

import os
import shutil
import subprocess

import pytest

from tree_verify_attention_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))


def test_step_plan_invariants(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "step_plan_check"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=compute_103a", "-O1",
                        "-std=c++17", "--expt-relaxed-constexpr",
                        "-I", os.path.join(B.ROOT, "include"),
                        "-I", os.path.join(B.ROOT, "tree_verify_attention_gb300", "csrc"),
                        "-o", str(exe), os.path.join(HERE, "step_plan_check.cu")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    fails = [l for l in r.stdout.splitlines() if l.startswith("FAIL")]
    assert r.returncode == 0 and not fails, "\n".join(fails[:20])
    assert r.stdout.strip().splitlines()[-1] == "ok (0 failures)"
    # the benchmarked workload is planned as measured: 136 attention units
    # (4 KV heads x 2 tiles (128 + 10 rows) x 17 key chunks), logits slices
    # staged on the CTAs without a unit and the 10-row tiles' units, tree rows
    # on the walker
    bench = [l for l in r.stdout.splitlines()
             if l.startswith("sms=152 N=23 hq=24 hkv=4 D=256 W=2048 cap=62912 V=151936 dt=1 fmt=2:")]
    assert bench and "units 136 splits 17 tiles 2 lunits 92 lbulk 1 walker_local 1" in bench[0], bench
