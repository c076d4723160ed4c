"""GPU parity of the forward-side steps (through the C ABI) against the fp64 oracle.

  * lrm_route: top-k indices bit-exact, alpha within 1e-6 relative of the fp64 softmax, loads and
    quotas bit-exact with the oracle's rule applied to the oracle's routing;
  * lrm_swiglu_forward: phi within one rounding of the storage type of the fp64 value, phi_sq within
    1e-5 relative of the fp64 norm of the stored row;
  * lrm_score_norms inside the whole path: the same agreement rules as the phi-based path.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import TOL, ensure_built, rel_fro, to_np
from test_parity_gpu import full_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


ROUTE_CASES = [
    W.WORKLOADS["tiny_f32"],
    W.small_workload("route_e48_k5", 3000, 64, 64, 48, 5),
    W.small_workload("route_zipf15_cap", 2048, 64, 64, 32, 8, zipf_s=1.5, quota=("cap", 300)),
    W.small_workload("route_e300_k16", 700, 64, 64, 300, 16, quota=("ratio", 7, 10)),
    W.small_workload("route_e1024_k2", 257, 64, 64, 1024, 2),
]


def check_route(logits, k, kind, num, den, cap, expl):
    import pruned_expert_backward_gb300 as lrm
    T, E = logits.shape
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ex = None if expl is None else torch.tensor(expl, dtype=torch.int32, device="cuda")
    idx, alpha, loads, quotas = lrm.lrm_route(logits, k, kind, num, den, cap, explicit=ex, dev_status=st)
    torch.cuda.synchronize()
    L = logits.cpu().numpy()
    oidx, oalpha = oracle.route(L, k)
    assert np.array_equal(to_np(idx), oidx)
    assert np.max(np.abs(to_np(alpha) - oalpha) / oalpha, initial=0.0) <= 1e-6
    ol, oq = oracle.plan_quotas(oidx, E, kind, num, den, cap, expl)
    assert np.array_equal(to_np(loads), ol)
    assert np.array_equal(to_np(quotas), oq)
    return int(st.item())


@pytest.mark.parametrize("wl", ROUTE_CASES, ids=lambda w: w.name)
def test_route_parity(wl):
    inp = W.generate(wl, "cuda", seed=3)
    kind, num, den, cap, expl = W.quota_policy(wl)
    assert check_route(inp["logits"], wl.k, kind, num, den, cap, expl) == 0


def test_route_ties_edges_and_nonfinite():
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    # integer logits: ties everywhere, broken toward the lower expert id
    L = torch.randint(-2, 3, (600, 40), generator=gen, device="cuda").float()
    assert check_route(L, 7, "ratio", 1, 2, 0, None) == 0
    # k = E: every expert, in logit order
    assert check_route(L[:, :7].contiguous(), 7, "cap", 0, 1, 3, None) == 0
    # explicit quotas, E not a multiple of 32
    assert check_route(L[:, :37].contiguous(), 3, "explicit", 0, 1, 0, list(range(37))) == 0
    # empty batch: loads 0, quotas from the rule
    assert check_route(L[:0].contiguous(), 3, "ratio", 8, 10, 0, None) == 0
    # a NaN logit is never chosen ahead of a finite one and is reported
    import pruned_expert_backward_gb300 as lrm
    bad = L[:4].clone()
    bad[1, 0] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, alpha, _, _ = lrm.lrm_route(bad, 3, "ratio", 1, 1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 7  # LRM_ERR_NONFINITE
    assert 0 not in to_np(idx[1]).tolist()
    assert torch.all(torch.isfinite(alpha))


SWIGLU_CASES = [
    W.WORKLOADS["tiny_f32"],
    W.small_workload("fwd_i136", 300, 64, 136, 8, 4),
    W.small_workload("fwd_qwen_i", 200, 64, 768, 8, 8),
    W.small_workload("fwd_glm_i", 100, 64, 1408, 8, 8),
    W.small_workload("fwd_wide_i", 40, 64, 3072, 8, 2),  # beyond the unrolled bound: looped kernel
]


@pytest.mark.parametrize("wl", SWIGLU_CASES, ids=lambda w: w.name)
def test_swiglu_forward_parity(wl):
    import pruned_expert_backward_gb300 as lrm
    inp = W.generate(wl, "cuda", seed=4)
    phi, phi_sq = lrm.lrm_swiglu_forward(inp["h"])
    torch.cuda.synchronize()
    want, _ = oracle.swiglu_forward(to_np(inp["h"]), wl.I)
    got = to_np(phi)
    ulp = 2.0 ** -8 if wl.dtype == "bf16" else 2.0 ** -21
    assert np.all(np.abs(got - want) <= ulp * np.abs(want) + 1e-30)
    norm = np.sum(got * got, axis=-1)
    assert np.max(np.abs(to_np(phi_sq) - norm) / np.maximum(norm, 1e-300)) <= 1e-5
    # without norms only phi is written
    phi2, none = lrm.lrm_swiglu_forward(inp["h"], norms=False)
    assert none is None and torch.equal(phi2, phi)


@pytest.mark.parametrize("wl", [W.WORKLOADS["tiny_f32"], W.small_workload("norms_bf16", 1000, 384, 320, 16, 4)],
                         ids=lambda w: w.name)
def test_path_scored_from_forward_norms(wl):
    """The forward emits phi and ||phi||^2; the backward scores from the norms and never reads phi
    for scoring.  Everything downstream meets the usual agreement rules."""
    import pruned_expert_backward_gb300 as lrm
    from helpers import gpu_quotas
    inp = W.generate(wl, "cuda", seed=5)
    phi, phi_sq = lrm.lrm_swiglu_forward(inp["h"])
    inp["phi"], inp["phi_sq"] = phi, phi_sq
    loads, q = gpu_quotas(inp, wl)
    flags = 1 if wl.dtype == "f32" else 0
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, flags=flags)
    pb.run(inp, q)
    torch.cuda.synchronize()
    del inp["phi_sq"]
    full_check(wl, inp, loads, q, pb)
    # same scores as the phi-based kernel, to fp32 summation order
    s_phi = lrm.lrm_score(inp["alpha"], inp["g"], inp["phi"])
    torch.cuda.synchronize()
    assert rel_fro(to_np(pb.scores), to_np(s_phi)) <= 1e-6
    assert TOL[wl.dtype] > 0
