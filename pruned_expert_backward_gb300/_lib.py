"""ctypes view of liblrm.so (include/lrm.h).  Argument types only; no logic."""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblrm.so")
# the same library built with -DLRM_DEBUG (index checks on the kernels' own indices); chosen by
# the environment variable LRM_DEBUG=1 when the library is first loaded
LIB_DEBUG_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblrm_debug.so")

# status codes, dtypes, quota kinds and flags of include/lrm.h
LRM_OK = 0
STATUS_NAMES = {0: "LRM_OK", 1: "LRM_ERR_INVALID_ARG", 2: "LRM_ERR_SHAPE", 3: "LRM_ERR_DTYPE",
                4: "LRM_ERR_WORKSPACE", 5: "LRM_ERR_CUDA", 6: "LRM_ERR_CAPACITY", 7: "LRM_ERR_NONFINITE",
                8: "LRM_ERR_TIMEOUT", 9: "LRM_ERR_BAD_INDEX", 10: "LRM_ERR_UNSUPPORTED",
                11: "LRM_ERR_BAD_SEGMENTS"}
LRM_BF16, LRM_F32 = 0, 1
LRM_QUOTA_RATIO, LRM_QUOTA_CAP, LRM_QUOTA_EXPLICIT = 0, 1, 2
LRM_GEMM_DEFAULT, LRM_GEMM_FORCE_SIMT = 0, 1
LRM_SCORE_LRM, LRM_SCORE_GRAD_SQ, LRM_SCORE_GRAD_ABS = 0, 1, 2
LRM_MAX_EXPERTS, LRM_MAX_TOPK = 1024, 16

_p, _i32, _i64, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t

SIGNATURES = {
    "lrm_status_string": (C.c_char_p, [C.c_int]),
    "lrm_workspace_size": (C.c_int, [_i64, _i32, _i32, _i32, _i32, C.c_int, C.POINTER(_sz)]),
    "lrm_plan_quotas": (C.c_int, [_p, _i64, _i32, _i32, C.c_int, _i32, _i32, _i32, _p, _p, _p, _p, _p]),
    "lrm_score": (C.c_int, [_p, _p, _p, _i64, _i32, _i32, _i32, C.c_int, _p, _p, _p]),
    "lrm_select": (C.c_int, [_p, _p, _p, _i64, _i32, _i32, _i64, _p, _p, _p, _p, _sz, _p, _p]),
    "lrm_compact": (C.c_int, [_p, _p, _p, _p, _p, _p, _i64, _i32, _i32, _i32, C.c_int, _i64, _p, _p, _p, _p,
                              _p, _p]),
    "lrm_grouped_backward": (C.c_int, [_p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, C.c_int, _i64, _p, _p,
                                       _p, _p, _p, _p, _sz, _i32, _p, _p]),
    "lrm_router_grad": (C.c_int, [_p, _p, _p, _i64, _i32, _i64, _p, _p]),
    "lrm_grouped_backward_gather": (C.c_int, [_p, _p, _i64, _i32, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, C.c_int,
                                              _i64, _p, _p, _p, _p, _p, _p, _sz, _i32, _p, _p]),
    "lrm_route": (C.c_int, [_p, _i64, _i32, _i32, C.c_int, _i32, _i32, _i32, _p, _p, _p, _p, _p, _p, _sz, _p, _p]),
    "lrm_swiglu_forward": (C.c_int, [_p, _i64, _i32, C.c_int, _p, _p, _p]),
    "lrm_score_norms": (C.c_int, [_p, _p, _p, _i64, _i32, _i32, C.c_int, _p, _p, _p]),
    "lrm_scatter_dx": (C.c_int, [_p, _p, _i64, _i32, _i32, C.c_int, _i64, _p, _p, _p]),
    "lrm_recompute_forward": (C.c_int, [_p, _p, _p, _i32, _i32, _i32, C.c_int, _i64, _p, _p, _p, _sz, _i32, _p,
                                        _p]),
    "lrm_selftest_wait_timeout": (C.c_int, [_p, _i64, _p]),
    "lrm_score_mode": (C.c_int, [_p, _p, _p, _i64, _i32, _i32, _i32, C.c_int, C.c_int, _p, _p, _p]),
}

_lib = None


def library_path() -> str:
    return LIB_DEBUG_PATH if os.environ.get("LRM_DEBUG") == "1" else LIB_PATH


def load():
    """Load liblrm.so (liblrm_debug.so with LRM_DEBUG=1); raise (never fall back) when it has not
    been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m pruned_expert_backward_gb300.build` (needs nvcc, CUDA 13)")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
