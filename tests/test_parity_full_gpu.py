"""Parity at the full workload sizes, in the launch configuration bench.py times.

The oracle cannot redo a whole 32k-token layer quickly, so it checks what it can compute one
by one: every score (fp64, in token chunks), the whole selection (bit-exact when the oracle
selects on the GPU's scores; cutoff rule against fp64 scores), sampled compacted rows, the full
per-expert dW of sampled experts (largest, median, smallest non-empty, one more), and dX of
sampled tokens.  Properties that hold at any size are checked everywhere: exact zeros of dW for
empty experts and of dX for tokens with nothing kept, kept counts = min(quota, load).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import TOL, ensure_built, gpu_quotas, rel_fro, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FULL = ["qwen3_t8k_d20", "qwen3_t32k_d0", "qwen3_t32k_d20", "qwen3_t32k_d30", "glm45_t32k_d20",
        "qwen3_t64k_zipf15_cap"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _np(t):
    t = t.detach().cpu()
    return t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity(name):
    import pruned_expert_backward_gb300 as lrm
    wl = W.WORKLOADS[name]
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    tol = TOL[wl.dtype]
    inp = W.generate(wl, "cuda", seed=0)
    loads, q = gpu_quotas(inp, wl)
    pb = lrm.PrunedBackward(T, k, E, H, I, dtype=wl.torch_dtype)  # same configuration as bench.py
    pb.run(inp, q)
    torch.cuda.synchronize()
    assert int(pb.dev_status.item()) == 0

    cpu = {n: _np(v) for n, v in inp.items() if n not in ("w_gate_up", "w_down")}

    def weights(e):  # one expert's weights on the host, as stored
        return _np(inp["w_gate_up"][e])[None], _np(inp["w_down"][e])[None]

    idx = cpu["topk_idx"].astype(np.int64)
    kind, num, den, cap, expl = W.quota_policy(wl)
    ol, oq = oracle.plan_quotas(idx, E, kind, num, den, cap, expl)
    assert np.array_equal(to_np(loads), ol) and np.array_equal(to_np(q), oq)

    # every score against fp64
    s = pb.scores.cpu().numpy().astype(np.float64).reshape(T, k)
    R64 = np.empty((T, k))
    for t0 in range(0, T, 4096):
        sl = slice(t0, min(T, t0 + 4096))
        R64[sl] = oracle.lrm_scores(cpu["alpha"][sl], cpu["g"][sl], cpu["phi"][sl])
    assert np.max(np.abs(s - R64) / R64) <= 1e-5

    # whole selection: bit-exact on the GPU's scores, cutoff rule on fp64 scores
    seg, kept, rop = oracle.select(idx, pb.scores.cpu().numpy(), oq, E)
    R = int(seg[-1])
    assert np.array_equal(to_np(pb.seg_offsets), seg)
    assert np.array_equal(to_np(pb.kept_pair)[:R], kept)
    assert np.array_equal(to_np(pb.row_of_pair), rop)
    assert np.array_equal(np.diff(seg), np.minimum(oq, ol))
    seg64, kept64, _ = oracle.select(idx, R64, oq, E)
    assert np.array_equal(seg64, seg)
    R64f = R64.reshape(-1)
    for e in range(E):
        a, b = kept[seg[e]:seg[e + 1]], kept64[seg[e]:seg[e + 1]]
        if not np.array_equal(a, b):
            diff = np.setxor1d(a, b)
            cut = R64f[b].min()
            assert np.all(np.abs(R64f[diff] - cut) <= 1e-5 * cut), e

    # sampled compacted rows
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(R, size=min(R, 2048), replace=False))
    dY, Xc, Hc, Phic = oracle.compact(kept[rows], cpu["alpha"], cpu["g"], cpu["x"], cpu["h"], cpu["phi"], k)
    rows_t = torch.as_tensor(rows, device="cuda")
    assert np.array_equal(_np(pb.x_c.index_select(0, rows_t)).astype(np.float64), Xc)
    assert np.array_equal(_np(pb.h_c.index_select(0, rows_t)).astype(np.float64), Hc)
    assert np.array_equal(_np(pb.phi_c.index_select(0, rows_t)).astype(np.float64), Phic)
    dyg = _np(pb.dy_c.index_select(0, rows_t)).astype(np.float64)
    assert np.all(np.abs(dyg - dY) <= 2.0 ** -8 * np.abs(dY) + 1e-38)

    # dW: exact zeros for empty experts (all), full per-expert check on sampled experts
    sizes = np.diff(seg)
    for e in np.nonzero(sizes == 0)[0]:
        assert torch.all(pb.dw_down[e] == 0) and torch.all(pb.dw_gate_up[e] == 0)
    nz = np.nonzero(sizes > 0)[0]
    order = nz[np.argsort(sizes[nz], kind="stable")]
    picks = sorted({int(order[-1]), int(order[len(order) // 2]), int(order[0]), int(rng.choice(nz))})
    for e in picks:
        seg_e = kept[seg[e]:seg[e + 1]]
        dY, Xc, Hc, Phic = oracle.compact(seg_e, cpu["alpha"], cpu["g"], cpu["x"], cpu["h"], cpu["phi"], k)
        dWgu, dWd, dH, dXc = oracle.expert_backward(np.array([0, len(seg_e)]), dY, Xc, Hc, Phic, *weights(e))
        assert rel_fro(_np(pb.dw_down[e]), dWd[0]) <= tol, (name, e, "dw_down")
        assert rel_fro(_np(pb.dw_gate_up[e]), dWgu[0]) <= tol, (name, e, "dw_gate_up")
        r0 = int(seg[e])
        got_dh = _np(pb.dh_c[r0:r0 + len(seg_e)]).astype(np.float64)
        assert rel_fro(got_dh, dH) <= tol, (name, e, "dh_c")

    # dX: exact zeros where nothing is kept (all tokens), sampled tokens against the oracle
    none_kept = torch.as_tensor(np.all(rop.reshape(T, k) < 0, axis=1), device="cuda")
    assert torch.all(pb.dx[none_kept] == 0)
    toks = np.sort(rng.choice(T, size=min(T, 256), replace=False))
    pairs = np.array([u for t in toks for u in range(t * k, t * k + k) if rop[u] >= 0], dtype=np.int64)
    pe = idx.reshape(-1)[pairs]
    dXc = np.zeros((len(pairs), H))
    for e in np.unique(pe):
        sel = np.nonzero(pe == e)[0]
        dY, Xc, Hc, Phic = oracle.compact(pairs[sel], cpu["alpha"], cpu["g"], cpu["x"], cpu["h"], cpu["phi"], k)
        dXc[sel] = oracle.expert_backward(np.array([0, len(sel)]), dY, Xc, Hc, Phic, *weights(e))[3]
    sub_rop = np.full(T * k, -1, np.int64)
    sub_rop[pairs] = np.arange(len(pairs))
    want = oracle.scatter_dx(sub_rop, dXc, T, k)[toks]
    got = _np(pb.dx.index_select(0, torch.as_tensor(toks, device="cuda"))).astype(np.float64)
    assert rel_fro(got, want) <= tol, (name, "dx", rel_fro(got, want))


@pytest.mark.parametrize("name", ["qwen3_t8k_d20", "glm45_t32k_d20"])
def test_full_size_router_grad(name):
    """dL/dalpha at full size: exact zeros for every dropped pair, sampled retained pairs against
    the oracle (one expert's weights at a time)."""
    import pruned_expert_backward_gb300 as lrm
    wl = W.WORKLOADS[name]
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    inp = W.generate(wl, "cuda", seed=0)
    _, q = gpu_quotas(inp, wl)
    pb = lrm.PrunedBackward(T, k, E, H, I, dtype=wl.torch_dtype, router_grad=True)
    pb.run(inp, q)
    torch.cuda.synchronize()
    assert int(pb.dev_status.item()) == 0
    rop = to_np(pb.row_of_pair)
    dalpha = pb.dalpha.cpu().numpy().astype(np.float64)
    assert np.all(dalpha[rop < 0] == 0)
    rng = np.random.default_rng(1)
    kept = np.nonzero(rop >= 0)[0]
    pairs = np.sort(rng.choice(kept, size=min(len(kept), 2048), replace=False))
    idx = inp["topk_idx"].reshape(-1).cpu().numpy()[pairs]
    g = _np(inp["g"].index_select(0, torch.as_tensor(pairs // k, device="cuda"))).astype(np.float64)
    phi = _np(inp["phi"].reshape(T * k, I).index_select(0, torch.as_tensor(pairs, device="cuda")))
    want = np.zeros(len(pairs))
    for e in np.unique(idx):
        sel = np.nonzero(idx == e)[0]
        wd = _np(inp["w_down"][int(e)])[None]
        # one pseudo-token per pair (k = 1), all retained, expert index 0 of the one-expert weights
        want[sel] = oracle.router_grad(np.zeros(len(sel), np.int64), np.zeros((len(sel), 1), np.int64),
                                       g[sel], phi[sel].astype(np.float64), wd)
    assert rel_fro(dalpha[pairs], want) <= TOL[wl.dtype], (name, rel_fro(dalpha[pairs], want))


@pytest.mark.parametrize("name", ["qwen3_t8k_d20", "qwen3_t64k_zipf15_cap"])
def test_full_size_compaction_free_bit_identical(name):
    """At full size, in the launch configuration bench.py times: the compaction-free variant's
    outputs equal the materialised path's bit for bit."""
    import pruned_expert_backward_gb300 as lrm
    wl = W.WORKLOADS[name]
    inp = W.generate(wl, "cuda", seed=0)
    _, q = gpu_quotas(inp, wl)
    res = []
    for mode in ("materialised", "gather"):
        pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, compaction=mode)
        pb.run(inp, q)
        torch.cuda.synchronize()
        assert int(pb.dev_status.item()) == 0
        res.append(pb)
        del pb
    a, b = res
    R = int(a.seg_offsets[-1])
    for n in ("dw_gate_up", "dw_down", "dx"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    assert torch.equal(a.dh_c[:R], b.dh_c[:R]) and torch.equal(a.dx_c[:R], b.dx_c[:R])


@pytest.mark.parametrize("name", ["qwen3_t8k_d20", "glm45_t32k_d20"])
def test_full_size_recompute(name):
    """The variant whose forward kept x and ||phi_u||^2 only, at full size: selection bit-exact on its
    own scores, recomputed h of sampled rows within one bf16 rounding (plus the fp32 sum bound) of the
    oracle's, full per-expert dW of sampled experts and dX of sampled tokens against the oracle."""
    import pruned_expert_backward_gb300 as lrm
    wl = W.WORKLOADS[name]
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    tol = TOL[wl.dtype]
    inp = W.generate(wl, "cuda", seed=0)
    _, q = gpu_quotas(inp, wl)
    _, phi_sq = lrm.lrm_swiglu_forward(inp["h"])
    lean = {n: v for n, v in inp.items() if n not in ("h", "phi")}
    lean["phi_sq"] = phi_sq
    pb = lrm.PrunedBackward(T, k, E, H, I, dtype=wl.torch_dtype, compaction="recompute")
    pb.run(lean, q)
    torch.cuda.synchronize()
    assert int(pb.dev_status.item()) == 0
    del inp
    cpu = {n: _np(v) for n, v in lean.items() if n not in ("w_gate_up", "w_down")}
    idx = cpu["topk_idx"].astype(np.int64)
    seg, kept, rop = oracle.select(idx, pb.scores.cpu().numpy(), to_np(q), E)
    R = int(seg[-1])
    assert np.array_equal(to_np(pb.seg_offsets), seg)
    assert np.array_equal(to_np(pb.kept_pair)[:R], kept)

    def weights(e):
        return _np(lean["w_gate_up"][e])[None], _np(lean["w_down"][e])[None]

    def expert_state(pairs, e):  # the oracle's compacted and recomputed rows of expert e's pairs
        t = pairs // k
        dY = cpu["alpha"].reshape(-1)[pairs].astype(np.float64)[:, None] * cpu["g"][t].astype(np.float64)
        X = cpu["x"][t].astype(np.float64)
        Hc, Phic = oracle.recompute_saved_state(np.arange(len(pairs)), np.zeros(len(pairs), np.int64), X,
                                                weights(e)[0], 1)
        return dY, X, Hc, Phic

    rng = np.random.default_rng(2)
    sizes = np.diff(seg)
    nz = np.nonzero(sizes > 0)[0]
    order = nz[np.argsort(sizes[nz], kind="stable")]
    picks = sorted({int(order[-1]), int(order[len(order) // 2]), int(order[0])})
    u = 2.0 ** -8
    for e in picks:
        pairs = kept[seg[e]:seg[e + 1]]
        dY, X, Hc, Phic = expert_state(pairs, e)
        r0 = int(seg[e])
        assert rel_fro(_np(pb.h_c[r0:r0 + len(pairs)]).astype(np.float64), Hc) <= u + TOL["f32"], (name, e, "h_c")
        dWgu, dWd, dH, dXc = oracle.expert_backward(np.array([0, len(pairs)]), dY, X, Hc, Phic, *weights(e))
        assert rel_fro(_np(pb.dw_down[e]), dWd[0]) <= tol, (name, e, "dw_down")
        assert rel_fro(_np(pb.dw_gate_up[e]), dWgu[0]) <= tol, (name, e, "dw_gate_up")
    toks = np.sort(rng.choice(T, size=min(T, 128), replace=False))
    pairs = np.array([v for t in toks for v in range(t * k, t * k + k) if rop[v] >= 0], dtype=np.int64)
    pe = idx.reshape(-1)[pairs]
    dXc = np.zeros((len(pairs), H))
    for e in np.unique(pe):
        sel = np.nonzero(pe == e)[0]
        dY, X, Hc, Phic = expert_state(pairs[sel], int(e))
        dXc[sel] = oracle.expert_backward(np.array([0, len(sel)]), dY, X, Hc, Phic, *weights(int(e)))[3]
    sub_rop = np.full(T * k, -1, np.int64)
    sub_rop[pairs] = np.arange(len(pairs))
    want = oracle.scatter_dx(sub_rop, dXc, T, k)[toks]
    got = _np(pb.dx.index_select(0, torch.as_tensor(toks, device="cuda"))).astype(np.float64)
    assert rel_fro(got, want) <= tol, (name, "dx", rel_fro(got, want))
