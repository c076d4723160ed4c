"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared element by element at every step; they span several GEMM tiles
with ragged tails.  Rules (from the method's stated agreement bar):
  * quotas, seg_offsets, kept_pair, row_of_pair: bit-exact (selection re-run by the oracle
    on the GPU's fp32 scores); against fp64 scores only cutoff-adjacent pairs may differ;
  * scores: <= 1e-5 relative to fp64;
  * compacted copies x_c, h_c, phi_c: bit-exact; dy_c within one fp32 product rounding plus one
    rounding to the storage type;
  * dW per expert and dX: relative Frobenius <= 1e-2 (bf16) / 1e-5 (fp32), exact zeros for
    experts with no rows and tokens with nothing kept.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (TOL, check_selection_bit_exact, check_selection_vs_fp64, ensure_built, rel_fro,
                     run_cuda_path, to_np)

pytestmark = pytest.mark.gpu

SIMT, TC = 1, 0
GEMM_MODES = {"bf16": [TC, SIMT], "f32": [SIMT]}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def full_check(wl, inp, loads, q, pb, quotas_from_rule=True):
    tol = TOL[wl.dtype]
    E, T, k = wl.E, wl.T, wl.k
    cpu = {n: v.cpu() for n, v in inp.items()}
    idx = to_np(cpu["topk_idx"])
    assert int(pb.dev_status.item()) == 0

    kind, num, den, cap, expl = W.quota_policy(wl)
    ol, oq = oracle.plan_quotas(idx, E, kind, num, den, cap, expl)
    assert np.array_equal(to_np(loads), ol)
    if quotas_from_rule:
        assert np.array_equal(to_np(q), oq)

    R64 = oracle.lrm_scores(to_np(cpu["alpha"]), to_np(cpu["g"]), to_np(cpu["phi"])).reshape(-1)
    s = pb.scores.cpu().double().numpy()
    pos = R64 > 0
    assert np.all(s[~pos] == 0)
    assert np.max(np.abs(s[pos] - R64[pos]) / R64[pos], initial=0.0) <= 1e-5

    seg, kept, rop = check_selection_bit_exact(cpu, q, pb, E)
    check_selection_vs_fp64(cpu, q, pb, E)

    ref = oracle.pruned_backward(cpu, to_np(q), scores=pb.scores.view(T, k).cpu())
    R = int(seg[-1])
    for mine, theirs in (("x_c", "X_c"), ("h_c", "H_c"), ("phi_c", "Phi_c")):
        assert np.array_equal(to_np(getattr(pb, mine)[:R]), ref[theirs]), mine
    # dy_c = round_dt(fl32(alpha * g)): the fp32 product is within 2^-24 of the exact one and one
    # round-to-nearest into dt is within half an ulp, i.e. u = 2^-p relative with p significant
    # bits (p = 8 for bf16, 24 for fp32): |dy_c - alpha g| <= (u + 2^-24 (1 + u)) |alpha g|
    dy = to_np(pb.dy_c[:R])
    u = 2.0 ** -8 if wl.dtype == "bf16" else 0.0
    rel = u + 2.0 ** -24 * (1 + u)
    assert np.all(np.abs(dy - ref["dY_c"]) <= rel * np.abs(ref["dY_c"]))

    dwd, dwg = to_np(pb.dw_down), to_np(pb.dw_gate_up)
    for e in range(E):
        if seg[e + 1] == seg[e]:
            assert np.all(dwd[e] == 0) and np.all(dwg[e] == 0), e
        else:
            assert rel_fro(dwd[e], ref["dw_down"][e]) <= tol, ("dw_down", e, rel_fro(dwd[e], ref["dw_down"][e]))
            assert rel_fro(dwg[e], ref["dw_gate_up"][e]) <= tol, ("dw_gate_up", e)
    if R > 0:
        assert rel_fro(to_np(pb.dh_c[:R]), ref["dH_c"]) <= tol
        assert rel_fro(to_np(pb.dx_c[:R]), ref["dX_c"]) <= tol
    dx = to_np(pb.dx)
    none_kept = np.all(rop.reshape(T, k) < 0, axis=1)
    assert np.all(dx[none_kept] == 0)
    assert rel_fro(dx, ref["dx"]) <= tol
    return ref


SMALL = [
    W.WORKLOADS["tiny_f32"],
    W.small_workload("bf16_tiles_ragged", 1000, 384, 320, 16, 4),
    W.small_workload("bf16_qwen_shape_small_T", 700, 2048, 768, 128, 8),
    W.small_workload("bf16_zipf15_cap", 2048, 512, 256, 32, 8, zipf_s=1.5, quota=("cap", 300)),
    W.small_workload("bf16_drop30", 1536, 256, 136, 24, 6, quota=("ratio", 7, 10)),
    # H = 200 and I = 96: the last 32-column dX_c store box is clipped by its map, and neither weight
    # map's column count allows one box per 128-column half
    W.small_workload("bf16_h_ragged", 800, 200, 96, 12, 4),
    # T*k = 131072 pairs: selection leaves the rows in bucket order and scatters row_of_pair in a
    # launch of its own (the path of the large workloads), on shapes the oracle checks in full
    W.small_workload("bf16_deferred_rows", 16384, 64, 64, 64, 8),
    # the limits of the ABI: top-1 routing, top-16 (LRM_MAX_TOPK: the generic score kernel, 16
    # rows per token in compaction and scatter), and 1024 experts (LRM_MAX_EXPERTS: one plan and
    # selection thread per expert, most experts holding a few rows)
    W.small_workload("bf16_top1", 1000, 256, 128, 16, 1),
    W.small_workload("bf16_top16", 600, 256, 128, 64, 16),
    W.small_workload("bf16_e1024", 4096, 128, 64, 1024, 8),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_parity(wl):
    for flags in GEMM_MODES[wl.dtype]:
        inp, loads, q, pb = run_cuda_path(wl, seed=1, flags=flags)
        full_check(wl, inp, loads, q, pb)


def check_router_grad(wl, inp, pb):
    """dL/dalpha against the oracle on the GPU's own selection; dropped pairs exactly 0; row_dot of
    row r equals alpha_u * dalpha_u of its pair."""
    tol = TOL[wl.dtype]
    cpu = {n: v.cpu() for n, v in inp.items()}
    P = wl.P
    rop = to_np(pb.row_of_pair)[:P]
    want = oracle.router_grad(rop, to_np(cpu["topk_idx"]), to_np(cpu["g"]), to_np(cpu["phi"]),
                              to_np(cpu["w_down"]))
    got = to_np(pb.dalpha)[:P]
    assert np.all(got[rop < 0] == 0)
    kept = rop >= 0
    if kept.any():
        assert rel_fro(got[kept], want[kept]) <= tol, rel_fro(got[kept], want[kept])
        alpha = to_np(cpu["alpha"]).reshape(-1)
        rd = to_np(pb.row_dot)[rop[kept]]
        assert rel_fro(rd, alpha[kept] * want[kept]) <= tol


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_router_grad_parity(wl):
    for flags in GEMM_MODES[wl.dtype]:
        inp, loads, q, pb = run_cuda_path(wl, seed=2, flags=flags, router_grad=True)
        assert int(pb.dev_status.item()) == 0
        check_router_grad(wl, inp, pb)
        # the other outputs are unchanged by the extra epilogue work
        full_check(wl, inp, loads, q, pb)


def test_router_grad_edges():
    wl = W.small_workload("router_edges", 400, 256, 136, 8, 2)
    for flags in GEMM_MODES["bf16"]:
        # nothing kept: every dalpha is 0
        inp, loads, q, pb = run_cuda_path(wl, flags=flags, quotas=np.zeros(8, np.int32), router_grad=True)
        assert int(pb.dev_status.item()) == 0
        assert torch.all(pb.dalpha == 0)
        # everything kept: the unpruned router gradient
        inp, loads, q, pb = run_cuda_path(wl, flags=flags, quotas=np.full(8, 10 ** 6, np.int32), router_grad=True)
        assert int(pb.seg_offsets[-1]) == wl.P
        check_router_grad(wl, inp, pb)


def test_load_example():
    wl = W.WORKLOADS["load_example"]
    inp, loads, q, pb = run_cuda_path(wl, flags=SIMT)
    assert to_np(loads).tolist() == [4, 2, 3]
    assert to_np(pb.seg_offsets).tolist() == [0, 3, 4, 6]
    full_check(wl, inp, loads, q, pb)


def test_zero_quota_keeps_nothing():
    wl = W.small_workload("zero_quota", 400, 256, 128, 8, 2)
    for flags in GEMM_MODES["bf16"]:
        inp, loads, q, pb = run_cuda_path(wl, flags=flags, quotas=np.zeros(8, np.int32))
        assert int(pb.dev_status.item()) == 0
        assert torch.all(pb.seg_offsets == 0)
        assert torch.all(pb.row_of_pair == -1)
        assert torch.all(pb.dw_down == 0) and torch.all(pb.dw_gate_up == 0) and torch.all(pb.dx == 0)


def test_full_quota_is_unpruned_backward():
    wl = W.small_workload("keep_all", 500, 256, 128, 8, 4, quota=("ratio", 1, 1))
    for flags in GEMM_MODES["bf16"]:
        inp, loads, q, pb = run_cuda_path(wl, flags=flags)
        assert torch.equal(q, loads)
        assert int(pb.seg_offsets[-1]) == wl.P
        ref = full_check(wl, inp, loads, q, pb)
        un = oracle.unpruned_backward({n: v.cpu() for n, v in inp.items()})
        assert rel_fro(to_np(pb.dx), un["dx"]) <= TOL["bf16"]
        assert np.array_equal(ref["kept_pair"], un["kept_pair"])


def test_single_expert():
    wl = W.small_workload("one_expert", 333, 128, 64, 1, 1, quota=("ratio", 8, 10))
    for flags in GEMM_MODES["bf16"]:
        inp, loads, q, pb = run_cuda_path(wl, flags=flags)
        full_check(wl, inp, loads, q, pb)


def test_empty_batch():
    import pruned_expert_backward_gb300 as lrm
    pb = lrm.PrunedBackward(0, 2, 4, 64, 32, dtype=torch.bfloat16, cap=0, flags=SIMT)
    inp = {"topk_idx": torch.zeros(0, 2, dtype=torch.int32, device="cuda"),
           "alpha": torch.zeros(0, 2, device="cuda"),
           "x": torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"),
           "g": torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"),
           "h": torch.zeros(0, 2, 64, dtype=torch.bfloat16, device="cuda"),
           "phi": torch.zeros(0, 2, 32, dtype=torch.bfloat16, device="cuda"),
           "w_gate_up": torch.randn(4, 64, 64, device="cuda").bfloat16(),
           "w_down": torch.randn(4, 64, 32, device="cuda").bfloat16()}
    pb.dw_down.fill_(1.0)
    pb.dw_gate_up.fill_(1.0)
    pb.run(inp, torch.zeros(4, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(pb.dev_status.item()) == 0
    assert torch.all(pb.seg_offsets == 0)
    assert torch.all(pb.dw_down == 0) and torch.all(pb.dw_gate_up == 0)


def test_all_scores_tied_keep_smallest_pair_index():
    wl = W.small_workload("ties", 300, 64, 32, 4, 2)
    inp = W.generate(wl, "cuda", seed=0)
    inp["alpha"].fill_(0.5)
    inp["g"][:] = inp["g"][0]
    inp["phi"][:] = inp["phi"][0, 0]
    import pruned_expert_backward_gb300 as lrm
    loads, q = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, "ratio", 1, 3)
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, flags=SIMT)
    pb.run(inp, q)
    torch.cuda.synchronize()
    assert torch.unique(pb.scores).numel() == 1
    seg, kept, _ = check_selection_bit_exact({n: v.cpu() for n, v in inp.items()}, q, pb, wl.E)
    idx = to_np(inp["topk_idx"]).reshape(-1)
    for e in range(wl.E):
        first = np.nonzero(idx == e)[0][: int(to_np(q)[e])]
        assert np.array_equal(kept[seg[e]:seg[e + 1]], first)


def test_capacity_overflow_keeps_nothing_and_flags():
    wl = W.small_workload("overflow", 256, 64, 32, 4, 2)
    inp, loads, q, pb = run_cuda_path(wl, flags=SIMT, cap=10)
    assert int(pb.dev_status.item()) == 6  # LRM_ERR_CAPACITY
    assert torch.all(pb.seg_offsets == 0)
    assert torch.all(pb.row_of_pair == -1)
    assert torch.all(pb.dx == 0)


def test_bad_expert_index_flags_and_drops_pair():
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("bad_idx", 128, 64, 32, 4, 2)
    inp = W.generate(wl, "cuda", seed=0)
    inp["topk_idx"][5, 1] = 7
    inp["topk_idx"][9, 0] = -3
    loads, q = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, "ratio", 1, 1)
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, flags=SIMT)
    pb.dev_status.zero_()
    pb.run(inp, q)
    torch.cuda.synchronize()
    assert int(pb.dev_status.item()) == 9  # LRM_ERR_BAD_INDEX
    rop = pb.row_of_pair.view(wl.T, wl.k)
    assert int(rop[5, 1]) == -1 and int(rop[9, 0]) == -1
    assert int(pb.seg_offsets[-1]) == wl.P - 2


def test_nonfinite_score_flags():
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("nonfinite", 64, 64, 32, 4, 2)
    inp = W.generate(wl, "cuda", seed=0)
    inp["g"][3, 7] = float("inf")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lrm.lrm_score(inp["alpha"], inp["g"], inp["phi"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 7  # LRM_ERR_NONFINITE


def test_bounded_wait_times_out_and_context_survives():
    """Failure detection without a fault: a wait that nothing satisfies gives up, reports
    LRM_ERR_TIMEOUT in the status word, and the GPU keeps working afterwards."""
    import time
    from pruned_expert_backward_gb300 import _lib
    lib = _lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    assert lib.lrm_selftest_wait_timeout(st.data_ptr(), 20_000_000, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 8  # LRM_ERR_TIMEOUT
    assert 0.015 <= dt < 2.0
    wl = W.small_workload("after_timeout", 256, 256, 128, 8, 2)
    inp, loads, q, pb = run_cuda_path(wl, flags=TC)
    full_check(wl, inp, loads, q, pb)


def test_host_pipeline_matches_device_path():
    """Pinned-host batches through HostPipeline (copies overlapping compute) give, step after
    step, exactly the results of the device-resident path."""
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("host_pipe", 600, 256, 128, 16, 4)
    w = W.generate(wl, "cuda", seed=3)
    refs, batches = [], []
    for seed in (3, 4, 5):
        inp = W.generate(wl, "cuda", seed=seed)
        inp["w_gate_up"], inp["w_down"] = w["w_gate_up"], w["w_down"]
        _, q = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, "ratio", 8, 10)
        pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I)
        pb.run(inp, q)
        torch.cuda.synchronize()
        refs.append((pb.dx.cpu().clone(), pb.seg_offsets.cpu().clone()))
        batches.append(({n: inp[n].cpu().pin_memory() for n in lrm.HostPipeline.NAMES}, q.cpu().pin_memory()))
    pipe = lrm.HostPipeline(lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I), w["w_gate_up"], w["w_down"])
    seen = []
    got = pipe.run(batches + batches[::-1], on_result=lambda i, dx, seg: seen.append((dx.clone(), seg.clone())))
    order = [0, 1, 2, 2, 1, 0]
    assert got == [int(refs[j][1][-1]) for j in order]
    for (dx, seg), j in zip(seen, order):
        assert torch.equal(seg, refs[j][1])
        assert torch.equal(dx, refs[j][0])


@pytest.mark.parametrize("mode", ["grad_sq", "grad_abs", "random"])
def test_ablation_scores_and_selection(mode):
    """The pages' selection ablations: gradient-only scores (fp64 parity 1e-5) and random
    dropping (caller-drawn uniform scores); selection on them is bit-exact with the oracle's."""
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("ablate", 1500, 512, 256, 32, 8)
    inp = W.generate(wl, "cuda", seed=7)
    _, q = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, "ratio", 8, 10)
    if mode == "random":
        gen = torch.Generator(device="cuda").manual_seed(11)
        scores = torch.rand(wl.P, generator=gen, device="cuda")
    else:
        scores = lrm.lrm_score_mode(None, inp["g"], inp["phi"], mode)
        fn = oracle.grad_sq_scores if mode == "grad_sq" else oracle.grad_abs_scores
        want = fn(to_np(inp["g"]), wl.k).reshape(-1)
        got = scores.cpu().double().numpy()
        assert np.max(np.abs(got - want) / want) <= 1e-5
    seg, kept, rop = lrm.lrm_select(inp["topk_idx"], scores, q, wl.E)
    torch.cuda.synchronize()
    oseg, okept, orop = oracle.select(to_np(inp["topk_idx"]), scores.cpu().numpy(), to_np(q), wl.E)
    assert np.array_equal(to_np(seg), oseg)
    assert np.array_equal(to_np(kept)[: int(oseg[-1])], okept)
    assert np.array_equal(to_np(rop), orop)


GATHER_CASES = SMALL + [W.small_workload("gather_i136_k6", 1536, 256, 136, 24, 6, quota=("ratio", 7, 10))]


@pytest.mark.parametrize("wl", GATHER_CASES, ids=lambda w: w.name)
def test_compaction_free_variant_is_bit_identical(wl):
    """The gather variant reads x / h / phi rows in place; every output must equal the
    materialised path's bit for bit (same values, same order of arithmetic), which the oracle
    checks above."""
    import pruned_expert_backward_gb300 as lrm
    from helpers import gpu_quotas
    inp = W.generate(wl, "cuda", seed=6)
    loads, q = gpu_quotas(inp, wl)
    for flags in GEMM_MODES[wl.dtype]:
        outs = []
        for mode in ("materialised", "gather"):
            pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, flags=flags,
                                    router_grad=True, compaction=mode)
            pb.run(inp, q)
            torch.cuda.synchronize()
            assert int(pb.dev_status.item()) == 0, mode
            outs.append(pb)
        a, b = outs
        R = int(a.seg_offsets[-1])
        assert torch.equal(a.seg_offsets, b.seg_offsets)
        for name in ("dw_gate_up", "dw_down", "dx", "dalpha"):
            assert torch.equal(getattr(a, name), getattr(b, name)), (name, flags)
        for name in ("dy_c", "dh_c", "dx_c", "row_dot"):
            assert torch.equal(getattr(a, name)[:R], getattr(b, name)[:R]), (name, flags)
    full_check(wl, inp, loads, q, a)


def test_compaction_free_edges():
    import pruned_expert_backward_gb300 as lrm
    wl = W.small_workload("gather_edges", 400, 256, 128, 8, 2)
    inp = W.generate(wl, "cuda", seed=7)
    for flags in GEMM_MODES["bf16"]:
        for quotas in (np.zeros(8, np.int32), np.full(8, 10 ** 6, np.int32)):
            q = torch.as_tensor(quotas, device="cuda")
            res = []
            for mode in ("materialised", "gather"):
                pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, flags=flags, compaction=mode)
                pb.run(inp, q)
                torch.cuda.synchronize()
                assert int(pb.dev_status.item()) == 0
                res.append(pb)
            assert torch.equal(res[0].dw_down, res[1].dw_down) and torch.equal(res[0].dw_gate_up, res[1].dw_gate_up)
            assert torch.equal(res[0].dx, res[1].dx)
        # cap = 0: nothing can be kept, every dW is exactly zero
        pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, flags=flags, compaction="gather", cap=0)
        pb.run(inp, torch.zeros(8, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert int(pb.dev_status.item()) == 0
        assert torch.all(pb.dw_down == 0) and torch.all(pb.dw_gate_up == 0) and torch.all(pb.dx == 0)
