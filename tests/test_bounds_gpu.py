"""Index checks of the CUDA path, on the GPU, through the C ABI.

Indices that one call hands to the next (row_of_pair, seg_offsets, kept_pair) are checked where
they are used: an index out of range is never followed, the pair (or the whole grouped backward)
is skipped, and the status word says why.  Every bad index below is planted so that even a
broken check would only touch allocated memory (the buffers carry spare rows past `cap`) and
never start a TMA copy at a negative coordinate, so no case can fault the GPU.  A second library
built with -DLRM_DEBUG also checks the kernels' own indices; it must give bit-identical results.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads as W
from helpers import ensure_built, run_cuda_path

pytestmark = pytest.mark.gpu

BAD_INDEX, BAD_SEGMENTS = 9, 11
SIMT, TC = 1, 0
SPARE = 64  # rows past cap in every compacted buffer


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _case():
    wl = W.small_workload("bounds", 300, 256, 128, 8, 4)
    inp, loads, q, pb = run_cuda_path(wl, seed=3, flags=TC)
    assert int(pb.dev_status.item()) == 0
    return wl, inp, q, pb


def test_scatter_skips_and_flags_rows_outside_cap():
    import pruned_expert_backward_gb300 as lrm
    wl, inp, q, pb = _case()
    cap = int(pb.seg_offsets[-1])
    dx_c = torch.zeros(cap + SPARE, wl.H, dtype=torch.bfloat16, device="cuda")
    dx_c[:cap] = pb.dx_c[:cap]
    dx_c[cap:] = 1.0  # what a broken check would add
    rop = pb.row_of_pair.clone()
    bad = torch.tensor([3, 17, 41, 100], device="cuda")
    rop[bad] = torch.tensor([cap, cap + 5, cap + SPARE - 1, -7], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = lrm.lrm_scatter_dx(rop, dx_c, wl.T, wl.k, cap=cap, dev_status=st)
    # the same call with those pairs dropped on purpose
    rop_ok = rop.clone()
    rop_ok[bad] = -1
    st_ok = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = lrm.lrm_scatter_dx(rop_ok, dx_c, wl.T, wl.k, cap=cap, dev_status=st_ok)
    torch.cuda.synchronize()
    assert int(st.item()) == BAD_INDEX
    assert int(st_ok.item()) == 0
    assert torch.equal(got, want)


def test_compact_skips_and_flags_rows_outside_cap():
    import pruned_expert_backward_gb300 as lrm
    wl, inp, q, pb = _case()
    cap = int(pb.seg_offsets[-1])
    rop = pb.row_of_pair.clone()
    bad = torch.tensor([2, 33, 90], device="cuda")
    rop[bad] = torch.tensor([cap, cap + SPARE - 1, -2], dtype=torch.int32, device="cuda")
    rop_ok = rop.clone()
    rop_ok[bad] = -1

    def run(r):
        bufs = [torch.full((cap + SPARE, n), 7.0, dtype=torch.bfloat16, device="cuda")
                for n in (wl.H, wl.H, 2 * wl.I, wl.I)]
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        lrm.lrm_compact(r, inp["alpha"], inp["g"], inp["x"], inp["h"], inp["phi"], cap, dy_c=bufs[0], x_c=bufs[1],
                        h_c=bufs[2], phi_c=bufs[3], dev_status=st)
        torch.cuda.synchronize()
        return bufs, int(st.item())

    got, st = run(rop)
    want, st_ok = run(rop_ok)
    assert st == BAD_INDEX and st_ok == 0
    for a, b in zip(got, want):
        assert torch.equal(a, b)
        assert torch.all(a[cap:] == 7.0)  # nothing written past cap


@pytest.mark.parametrize("flags", [TC, SIMT], ids=["tcgen05", "simt"])
@pytest.mark.parametrize("kind", ["first_not_zero", "decreasing", "beyond_cap"])
def test_grouped_backward_refuses_bad_segments(flags, kind):
    import pruned_expert_backward_gb300 as lrm
    wl, inp, q, pb = _case()
    E = wl.E
    seg = pb.seg_offsets.clone()
    R = int(seg[-1])
    cap = R
    if kind == "first_not_zero":
        seg[0] = 1
    elif kind == "decreasing":
        # expert 2's segment ends before it starts (no negative row anywhere)
        assert int(seg[2]) >= 8
        seg[3] = seg[2] - 5
    else:
        cap = R - 3
    rows = R + SPARE
    cmp = {n: torch.zeros(rows, c, dtype=torch.bfloat16, device="cuda")
           for n, c in (("dy_c", wl.H), ("x_c", wl.H), ("h_c", 2 * wl.I), ("phi_c", wl.I))}
    for n in cmp:
        cmp[n][:R] = getattr(pb, n)[:R]
    out = {"dw_gate_up": torch.full((E, 2 * wl.I, wl.H), 3.0, device="cuda"),
           "dw_down": torch.full((E, wl.H, wl.I), 3.0, device="cuda"),
           "dh_c": torch.full((rows, 2 * wl.I), 3.0, dtype=torch.bfloat16, device="cuda"),
           "dx_c": torch.full((rows, wl.H), 3.0, dtype=torch.bfloat16, device="cuda")}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lrm.lrm_grouped_backward(seg, cmp["dy_c"], cmp["x_c"], cmp["h_c"], cmp["phi_c"], inp["w_gate_up"],
                             inp["w_down"], cap, flags=flags, dev_status=st, **out)
    torch.cuda.synchronize()
    assert int(st.item()) == BAD_SEGMENTS
    for n, t in out.items():
        assert torch.all(t == 3.0), n  # nothing computed, nothing written


def test_compaction_free_flags_pairs_outside_range():
    import pruned_expert_backward_gb300 as lrm
    wl, inp, q, pb = _case()
    R = int(pb.seg_offsets[-1])
    P = wl.P
    # x / h / phi carry spare rows, so even an unchecked pair index stays inside allocated memory
    x = torch.zeros(wl.T + SPARE, wl.H, dtype=torch.bfloat16, device="cuda")
    h = torch.zeros(P + SPARE * wl.k, 2 * wl.I, dtype=torch.bfloat16, device="cuda")
    phi = torch.zeros(P + SPARE * wl.k, wl.I, dtype=torch.bfloat16, device="cuda")
    x[:wl.T] = inp["x"]
    h[:P] = inp["h"].view(P, -1)
    phi[:P] = inp["phi"].view(P, -1)
    kept = pb.kept_pair.clone()
    kept[R // 2] = P + 3
    for flags in (TC, SIMT):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = lrm.lrm_grouped_backward_gather(pb.seg_offsets, kept, wl.k, pb.dy_c, x[:wl.T], h[:P], phi[:P],
                                              inp["w_gate_up"], inp["w_down"], pb.cap, flags=flags, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == BAD_INDEX, flags
        dwg, dwd, dh_c, dx_c = out
        for t in (dwg, dwd, dh_c[:R], dx_c[:R]):
            assert torch.isfinite(t.float()).all()


_DEBUG_SCRIPT = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from pruned_expert_backward_gb300 import _lib
assert _lib.library_path().endswith("liblrm_debug.so")
import workloads as W
from helpers import run_cuda_path
wl = W.small_workload("dbg", 1000, 384, 320, 16, 4)
for flags in (0, 1):
    inp, loads, q, pb = run_cuda_path(wl, seed=1, flags=flags)
    assert int(pb.dev_status.item()) == 0, int(pb.dev_status.item())
    torch.save({n: getattr(pb, n).cpu() for n in ("seg_offsets", "kept_pair", "row_of_pair", "dw_down",
                                                   "dw_gate_up", "dx")}, sys.argv[2] + f".{flags}")
"""


def test_debug_build_checks_and_matches_release(tmp_path):
    """liblrm_debug.so (index checks on every index the kernels form) runs the whole path with no
    check failing and gives bit-identical results to liblrm.so."""
    from pruned_expert_backward_gb300 import _lib
    assert os.path.exists(_lib.LIB_DEBUG_PATH)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = str(tmp_path / "dbg")
    env = dict(os.environ, LRM_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", _DEBUG_SCRIPT, root, out], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    wl = W.small_workload("dbg", 1000, 384, 320, 16, 4)
    for flags in (0, 1):
        inp, loads, q, pb = run_cuda_path(wl, seed=1, flags=flags)
        dbg = torch.load(out + f".{flags}")
        for n, t in dbg.items():
            mine = getattr(pb, n).cpu()
            if n == "kept_pair":
                R = int(pb.seg_offsets[-1])
                mine, t = mine[:R], t[:R]
            assert torch.equal(mine, t), (n, flags)
