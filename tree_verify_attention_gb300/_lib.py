"""ctypes loader of libdfv.so with the argument types of include/dfv.h.

Argument marshalling only: every step of the verify step runs in the CUDA
kernels of the library. Loading fails loudly if the library is missing.
"""

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdfv.so")

_i32, _i64, _f32, _sz, _vp = C.c_int, C.c_int64, C.c_float, C.c_size_t, C.c_void_p

# name -> (restype, argtypes), in the order of include/dfv.h
SIGNATURES = {
    "dfv_status_string": (C.c_char_p, [_i32]),
    "dfv_version": (_i32, []),
    "dfv_tree_verify_attn_workspace_bytes": (_sz, [_i32] * 6),
    "dfv_tree_verify_attn": (_i32, [_i32] * 8 + [_vp] * 7 + [_f32, _vp, _vp, _vp, _sz, _vp, _vp]),
    "dfv_greedy_accept_workspace_bytes": (_sz, [_i32, _i32]),
    "dfv_greedy_accept": (_i32, [_i32, _i32, _i32] + [_vp] * 7 + [_vp, _sz, _vp, _vp]),
    "dfv_greedy_accept_static": (_i32, [_i32, _i32, _i32] + [_vp] * 7 + [_vp, _vp]),
    "dfv_kv_commit": (_i32, [_i32] * 5 + [_vp] * 7 + [_vp, _vp]),
    "dfv_kv_quantize_rows": (_i32, [_i32] * 6 + [_vp, _i32, _i64, _i64, _vp, _vp]),
    "dfv_verify_step_workspace_bytes": (_sz, [_i32] * 7),
    "dfv_verify_step": (_i32, [_i32] * 10 + [_vp] * 9 + [_f32] + [_vp] * 6 + [_vp, _sz, _vp, _vp]),
    "dfv_verify_step_launches": (_i32, [_i32] * 6),
    "dfv_workspace_clear": (_i32, [_vp, _sz, _vp]),
    "dfv_build_tree_mask": (_i32, [_i32] + [_vp] * 5),
}

_lib = None


def load():
    """Load (once) and return the library; raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libdfv.so not found at {LIB_PATH}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
