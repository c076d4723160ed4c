"""GPU parity of the variant whose forward keeps x and ||phi_u||^2 instead of h and phi: the
retained rows' h and phi are recomputed from x (lrm_recompute_forward, a tcgen05 var-M GEMM with
the SwiGLU forward in its epilogue) before the grouped backward.  Checked through the C ABI
against the oracle's pruned_backward_recompute (the same readings, fp64):
  * selection bit-exact when the oracle selects on the GPU's scores (from the norms);
  * h_c within one rounding of the storage type plus the fp32 summation bound of the fp64
    product, phi_c bit-identical to
    lrm_swiglu_forward of the stored h_c rows (same formula, same rounding);
  * dW per expert and dX within the usual relative Frobenius bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import TOL, ensure_built, gpu_quotas, rel_fro, to_np

pytestmark = pytest.mark.gpu

TC, SIMT = 0, 1
GEMM_MODES = {"bf16": [TC, SIMT], "f32": [SIMT]}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def lean_inputs(inp):
    """The forward's state in this variant: x, g, alpha, routing, weights and ||phi_u||^2."""
    import pruned_expert_backward_gb300 as lrm
    _, phi_sq = lrm.lrm_swiglu_forward(inp["h"])
    out = {n: v for n, v in inp.items() if n not in ("h", "phi")}
    out["phi_sq"] = phi_sq
    return out


def run_recompute(wl, seed, flags, quotas=None, cap=None):
    import pruned_expert_backward_gb300 as lrm
    inp = W.generate(wl, "cuda", seed=seed)
    loads, q = gpu_quotas(inp, wl)
    if quotas is not None:
        q = torch.as_tensor(np.asarray(quotas), dtype=torch.int32, device="cuda")
    lean = lean_inputs(inp)
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, flags=flags, cap=cap,
                            compaction="recompute")
    pb.run(lean, q)
    torch.cuda.synchronize()
    return inp, lean, q, pb


CASES = [
    W.WORKLOADS["tiny_f32"],
    W.small_workload("rc_tiles_ragged", 1000, 384, 320, 16, 4),
    W.small_workload("rc_qwen_shape", 700, 2048, 768, 128, 8),
    W.small_workload("rc_i136_k6", 1536, 256, 136, 24, 6, quota=("ratio", 7, 10)),
    W.small_workload("rc_h200_i96", 800, 200, 96, 12, 4),
    W.small_workload("rc_zipf15_cap", 2048, 512, 256, 32, 8, zipf_s=1.5, quota=("cap", 300)),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_recompute_parity(wl):
    import pruned_expert_backward_gb300 as lrm
    tol = TOL[wl.dtype]
    for flags in GEMM_MODES[wl.dtype]:
        inp, lean, q, pb = run_recompute(wl, seed=4, flags=flags)
        assert int(pb.dev_status.item()) == 0
        cpu = {n: v.cpu() for n, v in lean.items()}
        ref = oracle.pruned_backward_recompute(cpu, to_np(q), scores=pb.scores.view(wl.T, wl.k).cpu())
        seg = to_np(pb.seg_offsets)
        assert np.array_equal(seg, ref["seg_offsets"])
        R = int(seg[-1])
        assert np.array_equal(to_np(pb.kept_pair)[:R], ref["kept_pair"])
        # h_c: an fp32 sum of the products (within the fp32 parity bound, 1e-5) rounded once to the
        # storage type (half an ulp: 2^-8 relative for bf16; fp32 rows are stored as summed)
        h = to_np(pb.h_c[:R])
        u = 2.0 ** -8 if wl.dtype == "bf16" else 0.0
        assert rel_fro(h, ref["H_c"]) <= u + TOL["f32"], rel_fro(h, ref["H_c"])
        # phi_c: the forward's SwiGLU of the stored h_c rows, bit for bit
        phi_fw, _ = lrm.lrm_swiglu_forward(pb.h_c[:R].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(pb.phi_c[:R], phi_fw)
        assert rel_fro(to_np(pb.phi_c[:R]), ref["Phi_c"]) <= tol
        dwd, dwg = to_np(pb.dw_down), to_np(pb.dw_gate_up)
        for e in range(wl.E):
            if seg[e + 1] == seg[e]:
                assert np.all(dwd[e] == 0) and np.all(dwg[e] == 0)
            else:
                assert rel_fro(dwd[e], ref["dw_down"][e]) <= tol, ("dw_down", e, flags)
                assert rel_fro(dwg[e], ref["dw_gate_up"][e]) <= tol, ("dw_gate_up", e, flags)
        assert rel_fro(to_np(pb.dx), ref["dx"]) <= tol


def test_recompute_matches_the_saved_state_path():
    """On the same inputs the recompute variant and the materialised path agree within the bf16
    bound (h recomputed by the tensor cores instead of taken from the forward)."""
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("rc_vs_saved", 1200, 512, 256, 32, 8)
    inp, lean, q, pb = run_recompute(wl, seed=5, flags=TC)
    ref = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I)
    ref.run(dict(inp, phi_sq=lean["phi_sq"]), q)
    torch.cuda.synchronize()
    assert torch.equal(pb.seg_offsets, ref.seg_offsets)
    R = int(pb.seg_offsets[-1])
    assert rel_fro(to_np(pb.h_c[:R]), to_np(ref.h_c[:R])) <= 2.0 ** -7
    for n in ("dw_down", "dw_gate_up", "dx"):
        assert rel_fro(to_np(getattr(pb, n)), to_np(getattr(ref, n))) <= TOL["bf16"], n


def test_recompute_edges():
    wl = W.small_workload("rc_edges", 400, 256, 128, 8, 2)
    for flags in GEMM_MODES["bf16"]:
        inp, lean, q, pb = run_recompute(wl, seed=6, flags=flags, quotas=np.zeros(8, np.int32))
        assert int(pb.dev_status.item()) == 0
        assert torch.all(pb.dw_down == 0) and torch.all(pb.dw_gate_up == 0) and torch.all(pb.dx == 0)
        # cap = 0 with nothing to keep: every gradient exactly zero
        inp, lean, q, pb = run_recompute(wl, seed=6, flags=flags, quotas=np.zeros(8, np.int32), cap=0)
        assert int(pb.dev_status.item()) == 0
        assert torch.all(pb.dw_down == 0) and torch.all(pb.dx == 0)
        # cap = 0 with rows to keep: capacity overflow, nothing kept, still exact zeros
        inp, lean, q, pb = run_recompute(wl, seed=6, flags=flags, cap=0)
        assert int(pb.dev_status.item()) == 6  # LRM_ERR_CAPACITY
        assert torch.all(pb.dw_down == 0) and torch.all(pb.dx == 0)
    one = W.small_workload("rc_one_expert", 333, 128, 64, 1, 1)
    for flags in GEMM_MODES["bf16"]:
        inp, lean, q, pb = run_recompute(one, seed=7, flags=flags)
        cpu = {n: v.cpu() for n, v in lean.items()}
        ref = oracle.pruned_backward_recompute(cpu, to_np(q), scores=pb.scores.view(one.T, one.k).cpu())
        assert rel_fro(to_np(pb.dx), ref["dx"]) <= TOL["bf16"]
