"""Thin Python binding of libdfv (include/dfv.h) over torch device tensors.

PyTorch provides device memory and streams only; each function checks
dtypes/shapes, passes raw pointers to the C ABI and raises DfvError on a
non-OK status. No compute happens here.
"""

import torch

from . import _lib

DTYPE_F32 = 0
DTYPE_BF16 = 1
KV_F16 = 1
KV_Q4_0 = 2
KV_TREE_AS_CACHE = 0x100
STEP_PIPELINED = 0x200
_FORMATS = {"q4_0": KV_Q4_0, "f16": KV_F16}
MAX_NODES = 65
MASK_WORDS = (MAX_NODES + 31) // 32

DEV_BAD_TREE = 0x1
DEV_DEPTH = 0x2
DEV_CAPACITY = 0x4
DEV_CTX = 0x8
DEV_BAD_PATH = 0x10
DEV_TIMEOUT = 0x20


class DfvError(RuntimeError):
    pass


def lib():
    return _lib.load()


def _check(st, name):
    if st != 0:
        msg = lib().dfv_status_string(st).decode()
        raise DfvError(f"{name}: {msg} (status {st})")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _p(t):
    return None if t is None else t.data_ptr()


def _dev(t, name, dtypes, numel=None):
    if t is None:
        raise DfvError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise DfvError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype not in dtypes:
        raise DfvError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if numel is not None and t.numel() < numel:
        raise DfvError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t


_BF16 = (torch.bfloat16, torch.int16)
_I32 = (torch.int32,)
_F32 = (torch.float32,)


def q4_0_row_bytes(head_dim):
    return head_dim // 32 * 18


def row_bytes(head_dim, fmt="q4_0"):
    """Bytes of one cache row (one KV head, one position)."""
    if fmt == "f16":
        return head_dim * 2
    return q4_0_row_bytes(head_dim)


def _fmt_code(fmt):
    if fmt not in _FORMATS:
        raise DfvError(f"unknown cache format {fmt!r} (expected one of {sorted(_FORMATS)})")
    return _FORMATS[fmt]


class KVCache:
    """Device KV cache of one sequence in format ``fmt`` ("q4_0" or "f16"):
    K and V byte tensors [Hkv, capacity, row bytes] and the committed length
    (device int32)."""

    def __init__(self, n_kv_heads, head_dim, capacity, device="cuda", fmt="q4_0"):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        self.fmt = fmt
        self.kv_format = _fmt_code(fmt)
        shape = (n_kv_heads, capacity, row_bytes(head_dim, fmt))
        self.k = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.v = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.ctx_len = torch.zeros(1, dtype=torch.int32, device=device)

    def fill(self, k_rows, v_rows, pos0=0, stream=None):
        """Encode float rows [Hkv, n, D] (f32 or bf16) into positions
        [pos0, pos0 + n) and set the committed length to pos0 + n."""
        n = k_rows.shape[1]
        for src, dst in ((k_rows, self.k), (v_rows, self.v)):
            kv_quantize_rows(dst, src, pos0, self.n_kv_heads, self.head_dim, self.capacity,
                             head_major=True, stream=stream, fmt=self.fmt)
        self.ctx_len.fill_(pos0 + n)


class Q4Cache(KVCache):
    """Device Q4_0 KV cache of one sequence: K and V byte tensors
    [Hkv, capacity, D/32 * 18] and the committed length (device int32)."""

    def __init__(self, n_kv_heads, head_dim, capacity, device="cuda"):
        super().__init__(n_kv_heads, head_dim, capacity, device=device, fmt="q4_0")


def kv_quantize_rows(cache, src, pos0, n_kv_heads, head_dim, capacity, head_major=False,
                     stream=None, fmt="q4_0"):
    """Encode rows of ``src`` into ``cache`` positions [pos0, pos0 + n) in
    format ``fmt`` ("q4_0" or "f16").
    ``src`` is [n, Hkv, D] (or [Hkv, n, D] with head_major=True), f32 or
    bf16, last axis contiguous."""
    if src.dtype not in (torch.float32, torch.bfloat16) or not src.is_cuda:
        raise DfvError("src must be a CUDA f32 or bf16 tensor")
    if src.stride(-1) != 1:
        raise DfvError("src rows must be contiguous")
    if head_major:
        n, s_row, s_head = src.shape[1], src.stride(1), src.stride(0)
    else:
        n, s_row, s_head = src.shape[0], src.stride(0), src.stride(1)
    dt = DTYPE_F32 if src.dtype == torch.float32 else DTYPE_BF16
    _dev(cache, "cache", (torch.uint8,))
    _check(lib().dfv_kv_quantize_rows(n_kv_heads, head_dim, _fmt_code(fmt), capacity, pos0, n,
                                      src.data_ptr(), dt, s_row, s_head, cache.data_ptr(),
                                      _stream(stream)), "dfv_kv_quantize_rows")


def attn_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window, capacity):
    return lib().dfv_tree_verify_attn_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim,
                                                      window, capacity)


def accept_workspace_bytes(n_nodes, vocab):
    return lib().dfv_greedy_accept_workspace_bytes(n_nodes, vocab)


def step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window, capacity, vocab):
    return lib().dfv_verify_step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim,
                                                 window, capacity, vocab)


def step_launches(n_nodes, n_q_heads, n_kv_heads, head_dim, window, capacity):
    return lib().dfv_verify_step_launches(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                          capacity)


def workspace(nbytes, device="cuda", stream=None):
    """A zeroed, 256-byte aligned device workspace of ``nbytes``."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _check(lib().dfv_workspace_clear(ws.data_ptr(), ws.numel(), _stream(stream)),
           "dfv_workspace_clear")
    return ws


def clear_workspace(ws, stream=None):
    """Zero a workspace on the device (dfv_workspace_clear): before its first
    use, and again after a step reported DFV_DEV_TIMEOUT."""
    _dev(ws, "workspace", (torch.uint8,))
    _check(lib().dfv_workspace_clear(ws.data_ptr(), ws.numel(), _stream(stream)),
           "dfv_workspace_clear")


def tree_verify_attn(cache, q, tree_k, tree_v, parent, window, max_depth, out, lse, ws,
                     scale=0.0, status=None, stream=None, tree_as_cache=False, pipelined=False):
    n, hq, d = q.shape
    hkv = tree_k.shape[1]
    _dev(q, "q", _BF16)
    _dev(tree_k, "tree_k", _BF16, n * hkv * d)
    _dev(tree_v, "tree_v", _BF16, n * hkv * d)
    _dev(parent, "parent", _I32, n)
    _dev(out, "out", _F32, n * hq * d)
    if lse is not None:
        _dev(lse, "lse", _F32, n * hq)
    kvf = (cache.kv_format | (KV_TREE_AS_CACHE if tree_as_cache else 0)
           | (STEP_PIPELINED if pipelined else 0))
    _check(lib().dfv_tree_verify_attn(
        n, max_depth, hq, hkv, d, window, kvf, cache.capacity, cache.ctx_len.data_ptr(),
        cache.k.data_ptr(), cache.v.data_ptr(), q.data_ptr(), tree_k.data_ptr(),
        tree_v.data_ptr(), parent.data_ptr(), float(scale), out.data_ptr(), _p(lse),
        ws.data_ptr(), ws.numel(), _p(status), _stream(stream)), "dfv_tree_verify_attn")


def build_tree_mask(parent, depth, anc_mask, status=None, stream=None):
    """depth [N] (int32) and ancestor-or-self bitmasks [N, MASK_WORDS]
    (int32 tensor holding the uint32 words) of the tree given by ``parent``."""
    n = parent.numel()
    _dev(parent, "parent", _I32, n)
    _dev(depth, "depth", _I32, n)
    _dev(anc_mask, "anc_mask", _I32, n * MASK_WORDS)
    _check(lib().dfv_build_tree_mask(n, parent.data_ptr(), depth.data_ptr(), anc_mask.data_ptr(),
                                     _p(status), _stream(stream)), "dfv_build_tree_mask")


def greedy_accept(logits, parent, tokens, argmax, accept_len, path, out_tokens, ws,
                  status=None, stream=None):
    n, vocab = logits.shape
    dt = DTYPE_F32 if logits.dtype == torch.float32 else DTYPE_BF16
    _dev(logits, "logits", (torch.float32,) + _BF16)
    for t, nm in ((parent, "parent"), (tokens, "tokens"), (argmax, "argmax"), (path, "path"),
                  (out_tokens, "out_tokens")):
        _dev(t, nm, _I32, n)
    _dev(accept_len, "accept_len", _I32, 1)
    _check(lib().dfv_greedy_accept(
        n, vocab, dt, logits.data_ptr(), parent.data_ptr(), tokens.data_ptr(), argmax.data_ptr(),
        accept_len.data_ptr(), path.data_ptr(), out_tokens.data_ptr(), ws.data_ptr(), ws.numel(),
        _p(status), _stream(stream)), "dfv_greedy_accept")


def kv_commit(cache, accept_len, path, tree_k, tree_v, status=None, stream=None):
    n = tree_k.shape[0]
    _dev(tree_k, "tree_k", _BF16)
    _dev(tree_v, "tree_v", _BF16)
    _dev(accept_len, "accept_len", _I32, 1)
    _dev(path, "path", _I32)
    _check(lib().dfv_kv_commit(
        n, cache.n_kv_heads, cache.head_dim, cache.kv_format, cache.capacity, cache.ctx_len.data_ptr(),
        accept_len.data_ptr(), path.data_ptr(), tree_k.data_ptr(), tree_v.data_ptr(),
        cache.k.data_ptr(), cache.v.data_ptr(), _p(status), _stream(stream)), "dfv_kv_commit")


class VerifyStep:
    """Outputs and workspace of the verify step for one problem shape; call
    :meth:`run` once per step. All buffers live on the device.

    ``pipelined=True`` launches each step so that it overlaps the previous
    kernel of the stream (``DFV_STEP_PIPELINED``); the object then keeps two
    workspaces and uses them in turn, as consecutive pipelined steps need."""

    def __init__(self, n_nodes, n_q_heads, n_kv_heads, head_dim, window, capacity, vocab,
                 max_depth=16, device="cuda", pipelined=False):
        self.shape = (n_nodes, n_q_heads, n_kv_heads, head_dim, window, capacity, vocab)
        self.max_depth = max_depth
        dev = torch.device(device)
        self.out = torch.empty(n_nodes, n_q_heads, head_dim, dtype=torch.float32, device=dev)
        self.lse = torch.empty(n_nodes, n_q_heads, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(n_nodes, dtype=torch.int32, device=dev)
        self.accept_len = torch.zeros(1, dtype=torch.int32, device=dev)
        self.path = torch.empty(n_nodes, dtype=torch.int32, device=dev)
        self.out_tokens = torch.empty(n_nodes, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        nb = step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window, capacity,
                                  vocab)
        if nb == 0:
            raise DfvError(f"unsupported step shape {self.shape}")
        self.pipelined = bool(pipelined)
        self.workspaces = [workspace(nb, device=dev) for _ in range(2 if self.pipelined else 1)]
        self.ws = self.workspaces[0]
        self._turn = 0

    def run(self, cache, q, tree_k, tree_v, parent, tokens, logits, scale=0.0, stream=None,
            tree_as_cache=False):
        n, hq, hkv, d, window, cap, vocab = self.shape
        if cache.capacity != cap:
            raise DfvError("cache capacity differs from the planned one")
        _dev(q, "q", _BF16, n * hq * d)
        _dev(tree_k, "tree_k", _BF16, n * hkv * d)
        _dev(tree_v, "tree_v", _BF16, n * hkv * d)
        _dev(parent, "parent", _I32, n)
        _dev(tokens, "tokens", _I32, n)
        _dev(logits, "logits", (torch.float32,) + _BF16, n * vocab)
        dt = DTYPE_F32 if logits.dtype == torch.float32 else DTYPE_BF16
        kvf = (cache.kv_format | (KV_TREE_AS_CACHE if tree_as_cache else 0)
               | (STEP_PIPELINED if self.pipelined else 0))
        ws = self.workspaces[self._turn]
        self._turn = (self._turn + 1) % len(self.workspaces)
        _check(lib().dfv_verify_step(
            n, self.max_depth, hq, hkv, d, window, kvf, cap, vocab, dt,
            cache.ctx_len.data_ptr(), cache.k.data_ptr(), cache.v.data_ptr(), q.data_ptr(),
            tree_k.data_ptr(), tree_v.data_ptr(), parent.data_ptr(), tokens.data_ptr(),
            logits.data_ptr(), float(scale), self.out.data_ptr(), self.lse.data_ptr(),
            self.argmax.data_ptr(), self.accept_len.data_ptr(), self.path.data_ptr(),
            self.out_tokens.data_ptr(), ws.data_ptr(), ws.numel(),
            self.status.data_ptr(), _stream(stream)), "dfv_verify_step")
