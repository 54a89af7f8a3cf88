"""dfv_greedy_accept_static, the no-allocation variant of the argmax + walk
entry point, against dfv_greedy_accept, called through the C ABI.

Some callers cannot allocate device memory where they verify: a plugin
whose host framework owns every device allocation only receives its input
and output buffers, and a latency-critical decode loop cannot call
cudaMalloc / cudaFree because they may synchronise the device. The static
variant keeps its scratch in a fixed array inside the library; this test
checks that it gives the same results as the workspace version on two
calls in a row (the second call must not see stale scratch from the first).

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""

import numpy as np
import pytest
import torch

from tree_verify_attention_gb300 import _lib
from tree_verify_attention_gb300 import api
from tree_verify_attention_gb300 import workload as W

pytestmark = pytest.mark.gpu

FIELDS = ("argmax", "path", "out_tokens", "accept_len", "status")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_verify_attention_gb300 import build
    build.build()
    return _lib.load()


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def _inputs(cfg, step):
    s = W.make_step(cfg, step)
    if s.logits.dtype == np.uint16:
        logits, dt = _dev(s.logits.view(np.int16), torch.bfloat16), api.DTYPE_BF16
    else:
        logits, dt = _dev(s.logits), api.DTYPE_F32
    return dt, logits, _dev(s.parent), _dev(s.tokens)


def _outputs(n):
    return [torch.full((n,), -5, dtype=torch.int32, device="cuda") for _ in range(3)] + \
           [torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2)]


def _call(lib, static, n, vocab, dt, logits, parent, tokens, outs):
    argmax, path, out_tokens, accept_len, status = outs
    stream = torch.cuda.current_stream().cuda_stream
    if static:
        return lib.dfv_greedy_accept_static(n, vocab, dt, logits.data_ptr(), parent.data_ptr(),
                                            tokens.data_ptr(), argmax.data_ptr(),
                                            accept_len.data_ptr(), path.data_ptr(),
                                            out_tokens.data_ptr(), status.data_ptr(), stream)
    nb = lib.dfv_greedy_accept_workspace_bytes(n, vocab)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")   # the workspace version's scratch
    st = lib.dfv_greedy_accept(n, vocab, dt, logits.data_ptr(), parent.data_ptr(),
                               tokens.data_ptr(), argmax.data_ptr(), accept_len.data_ptr(),
                               path.data_ptr(), out_tokens.data_ptr(), ws.data_ptr(), nb,
                               status.data_ptr(), stream)
    torch.cuda.synchronize()
    return st


def _host(outs):
    return {k: o.cpu().numpy().copy() for k, o in zip(FIELDS, outs)}


@pytest.mark.parametrize("cfg", [W.TINY, W.SHORT], ids=lambda c: c.name)
def test_static_matches_workspace_version_twice(lib, cfg):
    for step in (0, 1):                       # two calls in a row
        dt, logits, parent, tokens = _inputs(cfg, step)
        want_o, got_o = _outputs(cfg.n_nodes), _outputs(cfg.n_nodes)
        assert _call(lib, False, cfg.n_nodes, cfg.vocab, dt, logits, parent, tokens, want_o) == 0
        assert _call(lib, True, cfg.n_nodes, cfg.vocab, dt, logits, parent, tokens, got_o) == 0
        torch.cuda.synchronize()
        want, got = _host(want_o), _host(got_o)
        assert want["status"][0] == 0 and want["accept_len"][0] >= 1
        for k in FIELDS:
            assert np.array_equal(got[k], want[k]), (cfg.name, step, k, got[k], want[k])


def test_static_back_to_back_calls_without_sync(lib):
    """Two calls queued on one stream before any synchronisation: the second
    starts from whatever the first left in the array."""
    cfg = W.SHORT
    queued = []
    for step in (2, 3):
        args = _inputs(cfg, step)
        outs = _outputs(cfg.n_nodes)
        assert _call(lib, True, cfg.n_nodes, cfg.vocab, *args, outs) == 0
        queued.append((args, outs))
    torch.cuda.synchronize()
    for args, outs in queued:
        want_o = _outputs(cfg.n_nodes)
        assert _call(lib, False, cfg.n_nodes, cfg.vocab, *args, want_o) == 0
        want, got = _host(want_o), _host(outs)
        for k in FIELDS:
            assert np.array_equal(got[k], want[k]), k


def test_static_rejects_invalid_arguments(lib):
    assert lib.dfv_greedy_accept_static(0, 10, 0, None, None, None, None, None, None, None,
                                        None, None) == 1
    assert lib.dfv_greedy_accept_static(4, 10, 7, None, None, None, None, None, None, None,
                                        None, None) == 2
