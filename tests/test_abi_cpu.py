"""CPU checks of the C ABI: the library loads, exports every entry point include/lrm.h declares,
and rejects bad arguments on the host before any GPU work (no compute call needs a GPU)."""
import ctypes as C
import os
import re

import pytest

from helpers import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lrm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lrm_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ensure_built()
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    lib = ensure_built()
    for code in range(0, 12):
        assert lib.lrm_status_string(code)
    assert lib.lrm_status_string(99) == b"unknown status"


def test_workspace_size_and_host_validation():
    lib = ensure_built()
    out = C.c_size_t(0)
    assert lib.lrm_workspace_size(8192, 8, 128, 2048, 768, 0, C.byref(out)) == 0
    assert out.value >= 8192 * 8 * 8
    assert lib.lrm_workspace_size(8, 8, 128, 2048, 768, 0, None) == 1        # null out pointer
    assert lib.lrm_workspace_size(8, 0, 128, 2048, 768, 0, C.byref(out)) == 1  # k = 0
    assert lib.lrm_workspace_size(8, 8, 2000, 2048, 768, 0, C.byref(out)) == 2  # E too large
    assert lib.lrm_workspace_size(8, 8, 128, 2047, 768, 0, C.byref(out)) == 2  # H not a multiple of 8
    assert lib.lrm_workspace_size(8, 8, 128, 2048, 768, 7, C.byref(out)) == 3  # bad dtype
    # null device pointers are refused before any launch
    assert lib.lrm_score(None, None, None, 16, 2, 64, 32, 0, None, None, None) == 1
    assert lib.lrm_select(None, None, None, 16, 2, 4, 32, None, None, None, None, 0, None, None) == 1
    assert lib.lrm_compact(None, None, None, None, None, None, 16, 2, 64, 32, 0, 32, None, None, None, None,
                           None, None) == 1
    assert lib.lrm_scatter_dx(None, None, 16, 2, 64, 0, 32, None, None, None) == 1
    fake16 = C.c_void_p(0x1000)
    assert lib.lrm_scatter_dx(fake16, fake16, 16, 2, 64, 0, -1, fake16, None, None) == 1  # negative cap
    assert lib.lrm_plan_quotas(None, 16, 2, 4, 0, 8, 10, 0, None, None, None, None, None) == 1
    # unknown GEMM flag
    fake = C.c_void_p(0x1000)
    assert lib.lrm_grouped_backward(fake, fake, fake, fake, fake, fake, fake, 4, 64, 32, 0, 16, fake, fake, fake,
                                    fake, None, fake, 1 << 20, 5, None, None) == 1
    # row_dot needs room for the dphi . phi parts of every row in the workspace
    small = C.c_size_t(0)
    assert lib.lrm_workspace_size(0, 1, 4, 64, 32, 0, C.byref(small)) == 0
    assert lib.lrm_grouped_backward(fake, fake, fake, fake, fake, fake, fake, 4, 64, 32, 0, 1 << 20, fake, fake,
                                    fake, fake, fake, fake, small.value, 0, None, None) == 4
    # forward-side entry points
    assert lib.lrm_route(None, 16, 8, 2, 0, 8, 10, 0, None, fake, fake, fake, fake, fake, 64, None, None) == 1
    assert lib.lrm_route(fake, 16, 8, 9, 0, 8, 10, 0, None, fake, fake, fake, fake, fake, 64, None, None) == 2
    assert lib.lrm_route(fake, 16, 8, 2, 0, 0, 10, 0, None, fake, fake, fake, fake, fake, 64, None, None) == 1
    assert lib.lrm_route(fake, 16, 8, 2, 2, 0, 1, 0, None, fake, fake, fake, fake, fake, 64, None, None) == 1
    assert lib.lrm_route(fake, 16, 8, 2, 0, 8, 10, 0, None, fake, fake, fake, fake, None, 0, None, None) == 4
    assert lib.lrm_swiglu_forward(None, 16, 32, 0, fake, None, None) == 1
    assert lib.lrm_swiglu_forward(fake, 16, 30, 0, fake, None, None) == 2   # I not a multiple of 8
    assert lib.lrm_swiglu_forward(C.c_void_p(0x1001), 16, 32, 0, fake, None, None) == 1
    assert lib.lrm_score_norms(fake, fake, None, 16, 2, 64, 0, fake, None, None) == 1
    assert lib.lrm_score_norms(fake, fake, fake, 16, 2, 64, 5, fake, None, None) == 3
    # router gradient: null pointers, negative cap
    assert lib.lrm_router_grad(None, fake, fake, 16, 2, 32, fake, None) == 1
    assert lib.lrm_router_grad(fake, fake, None, 16, 2, 32, fake, None) == 1
    assert lib.lrm_router_grad(fake, fake, fake, 16, 2, -1, fake, None) == 1
    # workspace too small for select
    assert lib.lrm_select(fake, fake, fake, 16, 2, 4, 32, fake, fake, fake, fake, 8, None, None) == 4
    # misaligned pointer
    odd = C.c_void_p(0x1001)
    assert lib.lrm_score(fake, odd, fake, 16, 2, 64, 32, 0, fake, None, None) == 1


def test_python_binding_refuses_cpu_tensors():
    import torch
    import pruned_expert_backward_gb300 as lrm
    ensure_built()
    with pytest.raises(ValueError):
        lrm.lrm_score(torch.zeros(4, 2), torch.zeros(4, 8), torch.zeros(4, 2, 8))


def test_sizes_that_would_overflow_are_refused():
    # T * k is never formed before T is known to keep it within int32 (no wrap-around to a
    # small or negative pair count that would pass the later checks)
    lib = ensure_built()
    out = C.c_size_t(0)
    assert lib.lrm_workspace_size(1 << 62, 8, 128, 2048, 768, 0, C.byref(out)) == 2
    assert lib.lrm_workspace_size((1 << 31) // 8, 8, 128, 64, 64, 0, C.byref(out)) == 2   # P = 2^31
    assert lib.lrm_workspace_size((1 << 31) // 8 - 1, 8, 8, 64, 64, 0, C.byref(out)) == 0
    fn = lib.lrm_select_static
    fn.restype = C.c_int
    fn.argtypes = [C.c_void_p] * 3 + [C.c_int64, C.c_int32, C.c_int32, C.c_int64] + [C.c_void_p] * 5
    fake = C.c_void_p(0x1000)
    assert fn(fake, fake, fake, 1 << 62, 8, 16, 0, fake, fake, fake, None, None) == 2
    assert fn(fake, fake, fake, (1 << 63) // 8, 8, 16, 0, fake, fake, fake, None, None) == 2


def test_recompute_forward_host_validation():
    lib = ensure_built()
    fn = lib.lrm_recompute_forward
    fake = C.c_void_p(0x1000)
    ws = C.c_size_t(0)
    assert lib.lrm_workspace_size(0, 1, 8, 64, 32, 0, C.byref(ws)) == 0
    # null seg_offsets / weights; null row buffers with rows to hold
    assert fn(None, fake, fake, 8, 64, 32, 0, 16, fake, fake, fake, ws.value, 0, None, None) == 1
    assert fn(fake, fake, None, 8, 64, 32, 0, 16, fake, fake, fake, ws.value, 0, None, None) == 1
    assert fn(fake, None, fake, 8, 64, 32, 0, 16, fake, fake, fake, ws.value, 0, None, None) == 1
    # unknown flag, bad dtype, sizes outside the limits, misaligned pointer, workspace too small
    assert fn(fake, fake, fake, 8, 64, 32, 0, 16, fake, fake, fake, ws.value, 7, None, None) == 1
    assert fn(fake, fake, fake, 8, 64, 32, 9, 16, fake, fake, fake, ws.value, 0, None, None) == 3
    assert fn(fake, fake, fake, 8, 60, 32, 0, 16, fake, fake, fake, ws.value, 0, None, None) == 2
    assert fn(fake, C.c_void_p(0x1008), fake, 8, 64, 32, 0, 16, fake, fake, fake, ws.value, 0, None, None) == 1
    assert fn(fake, fake, fake, 8, 64, 32, 0, 16, fake, fake, fake, 16, 0, None, None) == 4
    # nothing to recompute (cap = 0): accepted, nothing launched
    assert fn(fake, None, fake, 8, 64, 32, 0, 0, None, None, fake, ws.value, 0, None, None) == 0
