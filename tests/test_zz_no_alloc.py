"""lrm_select_static — selection for callers that cannot allocate — against lrm_select.

Callers such as a plugin whose host framework owns all device memory (and passes only inputs and
outputs), or a process whose device memory is fully reserved by a pool allocator, cannot hand the
library a workspace.  lrm_select_static keeps its scratch in a fixed array inside the library.
This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test.  It must pass alone in a fresh process and after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W
from helpers import ensure_built

pytestmark = pytest.mark.gpu

MAX_PAIRS = 524288
_p, _i32, _i64 = C.c_void_p, C.c_int32, C.c_int64


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ensure_built()
    fn = lib.lrm_select_static
    fn.restype = C.c_int
    fn.argtypes = [_p, _p, _p, _i64, _i32, _i32, _i64, _p, _p, _p, _p, _p]
    return lib


def _select_both(lib, wl, seed, quota):
    import pruned_expert_backward_gb300 as lrm
    inp = W.generate(wl, "cuda", seed=seed)
    _, q = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, "ratio", *quota)
    scores = lrm.lrm_score(inp["alpha"], inp["g"], inp["phi"])
    ref_seg, ref_kept, ref_rop = lrm.lrm_select(inp["topk_idx"], scores, q, wl.E)
    P = wl.T * wl.k
    seg = torch.full((wl.E + 1,), -7, dtype=torch.int32, device="cuda")
    kept = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    rop = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.lrm_select_static(inp["topk_idx"].data_ptr(), scores.data_ptr(), q.data_ptr(), wl.T, wl.k, wl.E, P,
                               seg.data_ptr(), kept.data_ptr(), rop.data_ptr(), st.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(st.item()) == 0
    R = int(ref_seg[-1])
    return (seg, kept[:R], rop), (ref_seg, ref_kept[:R], ref_rop)


def test_static_select_matches_workspace_select_twice(lib):
    # two calls in a row on different problems: stale scratch from the first must not leak
    cases = [(W.small_workload("na1", 4096, 256, 128, 128, 8), 1, (8, 10)),
             (W.small_workload("na2", 3000, 128, 64, 64, 6, zipf_s=1.5), 2, (7, 10))]
    for wl, seed, quota in cases:
        got, want = _select_both(lib, wl, seed, quota)
        for a, b in zip(got, want):
            assert torch.equal(a, b)  # selection is integer work: bit-exact


def test_static_select_matches_the_oracle(lib):
    # the same selection, checked against the oracle's top-quota rule on the GPU's own fp32 scores
    import oracle
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("na3", 2500, 256, 128, 32, 8)
    inp = W.generate(wl, "cuda", seed=3)
    _, q = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, "ratio", 8, 10)
    scores = lrm.lrm_score(inp["alpha"], inp["g"], inp["phi"])
    P = wl.T * wl.k
    seg = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    kept = torch.empty(P, dtype=torch.int32, device="cuda")
    rop = torch.empty(P, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.lrm_select_static(inp["topk_idx"].data_ptr(), scores.data_ptr(), q.data_ptr(), wl.T, wl.k, wl.E, P,
                               seg.data_ptr(), kept.data_ptr(), rop.data_ptr(), st.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    oseg, okept, orop = oracle.select(inp["topk_idx"].cpu().numpy(), scores.cpu().numpy(), q.cpu().numpy(), wl.E)
    R = int(oseg[-1])
    assert np.array_equal(seg.cpu().numpy(), oseg)
    assert np.array_equal(kept[:R].cpu().numpy(), okept)
    assert np.array_equal(rop.cpu().numpy(), orop)


def test_static_select_rejects_sizes_beyond_its_array(lib):
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    T = MAX_PAIRS // 8 + 1
    rc = lib.lrm_select_static(p, p, p, T, 8, 16, T * 8, p, p, p, None, None)
    assert rc == 2  # LRM_ERR_SHAPE, before any GPU work
