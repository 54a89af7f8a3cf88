"""The Python binding's own checks (CPU): it marshals only contiguous CUDA
tensors of the right dtype and size, rejects unknown formats, and fails
loudly, with a build hint, when the library is missing. None of these
reach a kernel."""

import pytest
import torch

from tree_verify_attention_gb300 import _lib, api


class _HostCache:
    """A cache-shaped object on the host (never valid for the library)."""

    def __init__(self):
        self.n_kv_heads, self.head_dim, self.capacity = 1, 64, 32
        self.fmt, self.kv_format = "q4_0", api.KV_Q4_0
        self.k = torch.zeros(1, 32, 36, dtype=torch.uint8)
        self.v = torch.zeros(1, 32, 36, dtype=torch.uint8)
        self.ctx_len = torch.zeros(1, dtype=torch.int32)


def test_host_tensors_are_refused():
    with pytest.raises(api.DfvError, match="contiguous CUDA tensor"):
        api._dev(torch.zeros(4, dtype=torch.int32), "parent", (torch.int32,), 4)
    with pytest.raises(api.DfvError, match="required"):
        api._dev(None, "parent", (torch.int32,))


def test_entry_points_check_before_calling_the_library():
    n, hq, d = 3, 2, 64
    q = torch.zeros(n, hq, d, dtype=torch.bfloat16)
    tk = torch.zeros(n, 1, d, dtype=torch.bfloat16)
    par = torch.tensor([-1, 0, 1], dtype=torch.int32)
    with pytest.raises(api.DfvError):
        api.tree_verify_attn(_HostCache(), q, tk, tk, par, 0, 4,
                             torch.zeros(n, hq, d), None, torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(api.DfvError):
        api.build_tree_mask(par, torch.zeros(n, dtype=torch.int32),
                            torch.zeros(n, api.MASK_WORDS, dtype=torch.int32))
    i32 = torch.zeros(n, dtype=torch.int32)
    with pytest.raises(api.DfvError):
        api.greedy_accept(torch.zeros(n, 10), par, i32, i32, torch.zeros(1, dtype=torch.int32),
                          i32, i32, torch.zeros(256, dtype=torch.uint8))


def test_formats_and_row_sizes():
    assert api.row_bytes(256) == 144 and api.row_bytes(128) == 72 and api.row_bytes(64) == 36
    assert api.row_bytes(256, "f16") == 512
    assert api._fmt_code("q4_0") == api.KV_Q4_0 and api._fmt_code("f16") == api.KV_F16
    with pytest.raises(api.DfvError, match="unknown cache format"):
        api._fmt_code("q8_0")


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libdfv.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not found.*build"):
        _lib.load()
    with pytest.raises(RuntimeError):
        api.lib()
