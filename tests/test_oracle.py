"""Pins of the fp64 oracle against what the LRMoE pages and plain mathematics fix.

Each pin checks the oracle against something other than itself: an explicit outer
product, the articles' worked example, brute force over subsets, exact rational
arithmetic, central finite differences, and torch fp64 autograd of an explicitly
written forward.  The last test plants plausible mistakes in the oracle (on the CPU)
and shows that some pin catches each of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.lrm_oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- pin helpers ---------
def score_pin_error(seed=0, T=5, k=3, H=7, I=6):
    """max relative gap between R_u and ||(alpha_u g_t) phi_u^T||_F^2 built explicitly."""
    rng = np.random.default_rng(seed)
    alpha = rng.uniform(0.05, 1.0, (T, k))
    g = rng.normal(0, 1, (T, H))
    phi = rng.normal(0, 1, (T, k, I))
    R = O.lrm_scores(alpha, g, phi)
    worst = 0.0
    for t in range(T):
        for j in range(k):
            G = np.outer(alpha[t, j] * g[t], phi[t, j])          # H x I rank-one gradient
            fro2 = float(np.sum(G * G))
            worst = max(worst, abs(R[t, j] - fro2) / fro2)
    return worst


def brute_force_select(scores, idx, quotas, E):
    """Per expert: among all subsets of size min(q, load) maximise the score sum; among
    maximisers take the lexicographically smallest sorted tuple of pair indices."""
    kept_all = []
    for e in range(E):
        pairs = [u for u in range(len(idx)) if idx[u] == e]
        n = min(quotas[e], len(pairs))
        best = None
        for comb in itertools.combinations(pairs, n):   # combinations come out sorted
            s = sum(scores[u] for u in comb)
            if best is None or s > best[0] or (s == best[0] and comb < best[1]):
                best = (s, comb)
        kept_all.append(list(best[1]))
    return kept_all


def select_pin_mismatches(select_fn, trials=60, seed=1):
    rng = np.random.default_rng(seed)
    bad = 0
    for _ in range(trials):
        E = int(rng.integers(1, 4))
        P = int(rng.integers(0, 13))
        idx = rng.integers(0, E, P)
        scores = rng.integers(0, 5, P).astype(np.float64)   # small integers: many exact ties
        quotas = rng.integers(0, 7, E)
        seg, kept, rop = select_fn(idx, scores, quotas, E)
        want = brute_force_select(list(scores), list(idx), list(quotas), E)
        got = [list(kept[seg[e]:seg[e + 1]]) for e in range(E)]
        if got != want:
            bad += 1
    return bad


def explicit_forward_grads(inp):
    """torch fp64 autograd of the explicitly written MoE-layer forward
    out_t = sum_j alpha_{t,j} W_down[e] (SiLU(W_gate[e] x_t) * (W_up[e] x_t)), loss = sum_t g_t . out_t."""
    x = torch.tensor(inp["x"], dtype=torch.float64, requires_grad=True)
    Wgu = torch.tensor(inp["w_gate_up"], dtype=torch.float64, requires_grad=True)
    Wd = torch.tensor(inp["w_down"], dtype=torch.float64, requires_grad=True)
    alpha = torch.tensor(inp["alpha"], dtype=torch.float64, requires_grad=True)
    g = torch.tensor(inp["g"], dtype=torch.float64)
    idx = inp["topk_idx"]
    T, k = idx.shape
    I = Wd.shape[2]
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(T):
        out = torch.zeros(Wd.shape[1], dtype=torch.float64)
        for j in range(k):
            e = int(idx[t, j])
            hid = Wgu[e] @ x[t]
            act = torch.nn.functional.silu(hid[:I]) * hid[I:]
            out = out + alpha[t, j] * (Wd[e] @ act)
        loss = loss + torch.dot(g[t], out)
    loss.backward()
    return Wgu.grad.numpy(), Wd.grad.numpy(), x.grad.numpy(), alpha.grad.numpy()


def fp64_consistent_inputs(seed=0, T=11, H=6, I=5, E=4, k=2):
    """Small fp64 inputs whose saved state (h, phi) is exactly the fp64 forward of x."""
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 1, (T, E))
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    ch = np.take_along_axis(logits, idx, 1)
    alpha = np.exp(ch - ch.max(1, keepdims=True))
    alpha /= alpha.sum(1, keepdims=True)
    x = rng.normal(0, 1, (T, H))
    g = rng.normal(0, 1, (T, H))
    Wgu = rng.normal(0, 1 / math.sqrt(H), (E, 2 * I, H))
    Wd = rng.normal(0, 1 / math.sqrt(I), (E, H, I))
    h = np.zeros((T, k, 2 * I))
    for t in range(T):
        for j in range(k):
            h[t, j] = Wgu[idx[t, j]] @ x[t]
    gate, up = h[..., :I], h[..., I:]
    phi = gate / (1 + np.exp(-gate)) * up
    return {"topk_idx": idx, "alpha": alpha, "x": x, "g": g, "h": h, "phi": phi,
            "w_gate_up": Wgu, "w_down": Wd}


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (d if d > 0 else 1.0)


def autograd_pin_error(seed=0):
    inp = fp64_consistent_inputs(seed)
    out = O.unpruned_backward(inp)
    gWgu, gWd, gx, _ = explicit_forward_grads(inp)
    return max(rel(out["dw_gate_up"], gWgu), rel(out["dw_down"], gWd), rel(out["dx"], gx))


def recompute_autograd_pin_error(seed=0):
    """quota = load on inputs without h and phi: the backward on the recomputed saved state against
    torch fp64 autograd of the explicit forward."""
    inp = fp64_consistent_inputs(seed)
    T, k = inp["topk_idx"].shape
    I = inp["w_down"].shape[2]
    phi_sq = np.sum(inp["phi"] ** 2, axis=2)
    lean = {n: v for n, v in inp.items() if n not in ("h", "phi")}
    lean["phi_sq"] = phi_sq
    loads = O.expert_loads(inp["topk_idx"], inp["w_down"].shape[0])
    out = O.pruned_backward_recompute(lean, loads)
    gWgu, gWd, gx, _ = explicit_forward_grads(inp)
    return max(rel(out["dw_gate_up"], gWgu), rel(out["dw_down"], gWd), rel(out["dx"], gx))


def recompute_matches_saved_state_error(seed=3):
    """With the saved state exactly the fp64 forward of x, recomputing it changes nothing: the
    pruned backward (quota below load) is the same either way."""
    inp = fp64_consistent_inputs(seed, T=13, E=3, k=2)
    E = inp["w_down"].shape[0]
    _, q = O.plan_quotas(inp["topk_idx"], E, "ratio", 3, 5)
    full = O.pruned_backward(inp, q)
    lean = {n: v for n, v in inp.items() if n not in ("h", "phi")}
    lean["phi_sq"] = np.sum(inp["phi"] ** 2, axis=2)
    lean_out = O.pruned_backward_recompute(lean, q)
    assert np.array_equal(full["kept_pair"], lean_out["kept_pair"])
    return max(rel(lean_out[n], full[n]) for n in ("H_c", "Phi_c", "dw_gate_up", "dw_down", "dx"))


def router_autograd_pin_error(seed=0):
    """quota = load: the oracle's dalpha against torch fp64 autograd's dL/dalpha."""
    inp = fp64_consistent_inputs(seed)
    out = O.unpruned_backward(inp)
    dalpha = O.router_grad(out["row_of_pair"], inp["topk_idx"], inp["g"], inp["phi"], inp["w_down"])
    *_, galpha = explicit_forward_grads(inp)
    return rel(dalpha, galpha.reshape(-1))


def router_masked_pin_error(seed=0):
    """Pruned selection: dalpha against the zero-masked full-shape route, where every pair's
    dPhi_u = (mask_u alpha_u g_t) W_down[e] and dalpha_u = (dPhi_u . phi_u) / alpha_u.
    Returns (relative error, number of dropped pairs)."""
    inp = fp64_consistent_inputs(seed, T=13, E=3, k=2)
    idx = inp["topk_idx"]
    E = inp["w_down"].shape[0]
    _, quotas = O.plan_quotas(idx, E, "ratio", 1, 2)
    out = O.pruned_backward(inp, quotas)
    rop = out["row_of_pair"].reshape(-1)
    dalpha = O.router_grad(rop, idx, inp["g"], inp["phi"], inp["w_down"])
    T, k = idx.shape
    alt = np.zeros(T * k)
    for t in range(T):
        for j in range(k):
            u = t * k + j
            a = inp["alpha"][t, j]
            dy = (a if rop[u] >= 0 else 0.0) * inp["g"][t]
            dphi = dy @ inp["w_down"][idx[t, j]]
            alt[u] = float(dphi @ inp["phi"][t, j]) / a
    assert np.all(dalpha[rop < 0] == 0.0)
    return rel(dalpha, alt), int(np.sum(rop < 0))


def swiglu_fd_error(seed=0):
    rng = np.random.default_rng(seed)
    gate = rng.normal(0, 2, 200)
    up = rng.normal(0, 2, 200)
    dphi = rng.normal(0, 1, 200)

    def phi(gt, u):
        return gt / (1 + np.exp(-gt)) * u

    eps = 1e-6
    fd_gate = dphi * (phi(gate + eps, up) - phi(gate - eps, up)) / (2 * eps)
    fd_up = dphi * (phi(gate, up + eps) - phi(gate, up - eps)) / (2 * eps)
    dgate, dup = O.swiglu_backward(dphi, gate, up)
    return max(np.max(np.abs(dgate - fd_gate)), np.max(np.abs(dup - fd_up)))


def masking_pin_error():
    inp = W.generate(W.WORKLOADS["tiny_f32"], "cpu", seed=3)
    E = inp["w_down"].shape[0]
    _, quotas = O.plan_quotas(inp["topk_idx"].numpy(), E, "ratio", 7, 10)
    a = O.pruned_backward(inp, quotas)
    b = O.masked_backward(inp, quotas)
    return max(rel(a["dw_gate_up"], b["dw_gate_up"]), rel(a["dw_down"], b["dw_down"]), rel(a["dx"], b["dx"]))


# ---------------------------------------------------------------- pins ----------------
def test_score_is_frobenius_norm_of_rank_one_gradient():
    assert score_pin_error() < 1e-12


def test_load_example_golden():
    gold = json.load(open(os.path.join(GOLDEN, "load_example.json")))
    wl = W.WORKLOADS["load_example"]
    inp = W.generate(wl, "cpu", seed=0)
    idx = inp["topk_idx"].numpy()
    loads, quotas = O.plan_quotas(idx, wl.E, "explicit", explicit=list(wl.quota[1]))
    assert list(loads) == gold["loads"]
    assert list(quotas) == gold["quotas"]
    R = O.lrm_scores(inp["alpha"].numpy(), inp["g"].numpy(), inp["phi"].numpy())
    seg, kept, rop = O.select(idx, R, quotas, wl.E)
    assert list(np.diff(seg)) == gold["segment_sizes"]
    assert list(seg[:-1]) == gold["segment_starts"]
    assert list(seg) == gold["seg_offsets"]
    flat = idx.reshape(-1)
    Rf = R.reshape(-1)
    for e in range(wl.E):
        pairs = np.nonzero(flat == e)[0]
        kept_e = set(kept[seg[e]:seg[e + 1]].tolist())
        dropped = [u for u in pairs if u not in kept_e]
        for u in kept_e:
            for v in dropped:
                assert Rf[u] >= Rf[v]
    assert sorted(np.nonzero(rop >= 0)[0].tolist()) == sorted(kept.tolist())


def test_selection_is_optimal_by_brute_force():
    assert select_pin_mismatches(O.select) == 0


def test_quota_rules_exact():
    loads = np.concatenate([np.arange(0, 2000), np.array([65399, 99999, 599999, 1000000])])
    for num, den in [(8, 10), (7, 10), (1, 1), (1, 3)]:
        idx = np.repeat(np.arange(len(loads)), loads)
        got_loads, q = O.plan_quotas(idx, len(loads), "ratio", num, den)
        assert np.array_equal(got_loads, loads)
        want = [math.ceil(Fraction(num, den) * int(l)) for l in loads]
        assert q.tolist() == want
    idx = np.repeat(np.arange(5), [0, 1, 2867, 2868, 9000])
    _, q = O.plan_quotas(idx, 5, "cap", cap=2868)
    assert q.tolist() == [0, 1, 2867, 2868, 2868]
    # the stress workload's budget ceil(0.7 * T * 8 / E)
    assert W.WORKLOADS["qwen3_t64k_zipf15_cap"].quota[1] == math.ceil(Fraction(7, 10) * 65536 * 8 / 128)


def test_swiglu_derivative_finite_differences():
    assert swiglu_fd_error() < 1e-7


def test_full_quota_reduces_to_autograd_backward():
    for seed in range(3):
        assert autograd_pin_error(seed) < 1e-12


def test_recomputed_state_full_quota_equals_autograd():
    for seed in range(3):
        assert recompute_autograd_pin_error(seed) < 1e-12


def test_recomputed_state_equals_saved_state():
    assert recompute_matches_saved_state_error() < 1e-12


def test_router_grad_full_quota_equals_autograd():
    for seed in range(3):
        assert router_autograd_pin_error(seed) < 1e-12


def test_router_grad_pruned_equals_masked_route():
    err, n_dropped = router_masked_pin_error()
    assert n_dropped > 0
    assert err < 1e-12


def route_pin_mismatches(route_fn, trials=200, seed=5):
    """Brute-force ranking: expert e's rank is the number of experts with a larger logit or an
    equal logit and a smaller id; the top-k are ranks 0..k-1 in rank order."""
    rng = np.random.default_rng(seed)
    bad = 0
    for _ in range(trials):
        T, E = int(rng.integers(1, 5)), int(rng.integers(1, 9))
        k = int(rng.integers(1, E + 1))
        L = rng.integers(-2, 3, (T, E)).astype(np.float64)   # small integers: ties everywhere
        idx, alpha = route_fn(L, k)
        for t in range(T):
            rank = [sum(1 for f in range(E) if L[t, f] > L[t, e] or (L[t, f] == L[t, e] and f < e))
                    for e in range(E)]
            want = sorted(range(E), key=lambda e: rank[e])[:k]
            if list(idx[t]) != want:
                bad += 1
    return bad


def route_alpha_pin_error(route_fn, seed=6):
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 2, (50, 6))
    idx, alpha = route_fn(L, 2)
    gap = np.take_along_axis(L, idx, 1)
    logistic = 1.0 / (1.0 + np.exp(-(gap[:, 0] - gap[:, 1])))
    err = np.max(np.abs(alpha[:, 0] - logistic))
    idx4, alpha4 = route_fn(L, 4)
    err = max(err, np.max(np.abs(alpha4.sum(1) - 1.0)))
    assert np.all(np.diff(alpha4, axis=1) <= 0)
    return err


def test_route_ranks_by_brute_force():
    assert route_pin_mismatches(O.route) == 0


def test_route_alpha_closed_forms():
    assert route_alpha_pin_error(O.route) < 1e-14


def swiglu_forward_pin_error(seed=7):
    rng = np.random.default_rng(seed)
    I = 9
    h = rng.normal(0, 3, (20, 2 * I))
    phi, phi_sq = O.swiglu_forward(h, I)
    ht = torch.tensor(h, dtype=torch.float64)
    want = torch.nn.functional.silu(ht[:, :I]) * ht[:, I:]
    err = np.max(np.abs(phi - want.numpy()))
    err = max(err, np.max(np.abs(phi_sq - (want * want).sum(1).numpy()) / (want * want).sum(1).numpy()))
    # the derivative of this phi is the backward closed form (central differences)
    eps = 1e-6
    dphi = rng.normal(0, 1, (20, I))
    hp, hm = h.copy(), h.copy()
    hp[:, :I] += eps
    hm[:, :I] -= eps
    fd_gate = dphi * (O.swiglu_forward(hp, I)[0] - O.swiglu_forward(hm, I)[0]) / (2 * eps)
    dgate, _ = O.swiglu_backward(dphi, h[:, :I], h[:, I:])
    return err, np.max(np.abs(fd_gate - dgate))


def test_swiglu_forward_matches_torch_and_backward():
    err, fd = swiglu_forward_pin_error()
    assert err < 1e-12 and fd < 1e-5


def test_scores_from_norms_equal_lrm_scores():
    rng = np.random.default_rng(8)
    alpha = rng.uniform(0.05, 1.0, (6, 3))
    g = rng.normal(0, 1, (6, 11))
    phi = rng.normal(0, 1, (6, 3, 5))
    want = O.lrm_scores(alpha, g, phi)
    got = O.lrm_scores_from_norms(alpha, g, np.sum(phi * phi, axis=2))
    assert np.max(np.abs(got - want) / want) < 1e-14


def test_compacted_equals_zero_masked_full_shape():
    assert masking_pin_error() < 1e-12


def test_zero_quota_gives_exact_zeros():
    inp = W.generate(W.WORKLOADS["tiny_f32"], "cpu", seed=0)
    out = O.pruned_backward(inp, np.zeros(8, np.int64))
    assert out["kept_pair"].size == 0
    assert np.all(out["row_of_pair"] == -1)
    assert np.all(out["dw_gate_up"] == 0) and np.all(out["dw_down"] == 0) and np.all(out["dx"] == 0)


def test_segments_are_u_ascending_and_row_of_pair_inverts_kept():
    inp = W.generate(W.WORKLOADS["tiny_f32"], "cpu", seed=1)
    idx = inp["topk_idx"].numpy()
    _, quotas = O.plan_quotas(idx, 8, "ratio", 8, 10)
    out = O.pruned_backward(inp, quotas)
    seg, kept, rop = out["seg_offsets"], out["kept_pair"], out["row_of_pair"]
    for e in range(8):
        s = kept[seg[e]:seg[e + 1]]
        assert np.all(np.diff(s) > 0)
        assert np.all(idx.reshape(-1)[s] == e)
        assert len(s) == min(quotas[e], np.sum(idx == e))
    assert np.array_equal(rop[kept], np.arange(len(kept)))
    assert np.sum(rop >= 0) == len(kept)


def test_tiny_workload_drop_fraction():
    wl = W.WORKLOADS["tiny_f32"]
    inp = W.generate(wl, "cpu", seed=0)
    loads, quotas = O.plan_quotas(inp["topk_idx"].numpy(), wl.E, "ratio", 8, 10)
    assert loads.sum() == wl.P
    assert 0.8 * wl.P <= quotas.sum() <= 0.8 * wl.P + wl.E


# ------------------------------------------------- planted mistakes are caught ---------
def _planted_scores_no_alpha(alpha, g, phi):
    return np.sum(np.asarray(g, float) ** 2, 1)[:, None] * np.sum(np.asarray(phi, float) ** 2, 2)


def _planted_scores_abs_g(alpha, g, phi):
    a = np.asarray(alpha, float)
    return a * a * np.sum(np.abs(np.asarray(g, float)), 1)[:, None] * np.sum(np.asarray(phi, float) ** 2, 2)


def _planted_select_u_desc(topk_idx, scores, quotas, E):
    flat = np.asarray(topk_idx).reshape(-1)
    s = np.asarray(scores).reshape(-1)
    seg = np.zeros(E + 1, np.int64)
    kept = []
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]
        n = int(min(quotas[e], len(pairs)))
        order = np.lexsort((-pairs, -s[pairs]))          # ties to the LARGER u
        kept.append(np.sort(pairs[order[:n]]))
        seg[e + 1] = seg[e] + n
    kept = np.concatenate(kept) if kept else np.zeros(0, np.int64)
    rop = np.full(len(flat), -1)
    rop[kept] = np.arange(len(kept))
    return seg, kept, rop


def _planted_swiglu_missing_term(dphi, gate, up):
    s = O.sigmoid(gate)
    return dphi * up * s, dphi * gate * s


_true_swiglu_backward = O.swiglu_backward


def _planted_swiglu_swapped(dphi, gate, up):
    return _true_swiglu_backward(dphi, up, gate)


def _planted_scatter_drops_last_choice(row_of_pair, dX_c, T, k):
    rop = np.asarray(row_of_pair).reshape(T, k)
    dX = np.zeros((T, dX_c.shape[1]))
    for j in range(k - 1):
        m = rop[:, j] >= 0
        dX[m] += dX_c[rop[m, j]]
    return dX


def test_planted_mistakes_fail_a_pin(monkeypatch):
    with monkeypatch.context() as m:
        m.setattr(O, "lrm_scores", _planted_scores_no_alpha)
        assert score_pin_error() > 1e-3
    with monkeypatch.context() as m:
        m.setattr(O, "lrm_scores", _planted_scores_abs_g)
        assert score_pin_error() > 1e-3
    assert select_pin_mismatches(_planted_select_u_desc) > 0
    with monkeypatch.context() as m:
        m.setattr(O, "swiglu_backward", _planted_swiglu_missing_term)
        assert swiglu_fd_error() > 1e-3 and autograd_pin_error() > 1e-3
    with monkeypatch.context() as m:
        m.setattr(O, "swiglu_backward", _planted_swiglu_swapped)
        assert autograd_pin_error() > 1e-3
    with monkeypatch.context() as m:
        m.setattr(O, "scatter_dx", _planted_scatter_drops_last_choice)
        assert autograd_pin_error() > 1e-3
    # recomputed saved state: gate and up rows of W_gate_up taken the wrong way round
    real_recompute = O.recompute_saved_state

    def recompute_swapped(kept_pair, topk_idx, x, w_gate_up, k):
        W = np.asarray(w_gate_up)
        I = W.shape[1] // 2
        return real_recompute(kept_pair, topk_idx, x, np.concatenate([W[:, I:], W[:, :I]], axis=1), k)

    with monkeypatch.context() as m:
        m.setattr(O, "recompute_saved_state", recompute_swapped)
        assert recompute_autograd_pin_error() > 1e-3
    # forward-side steps
    def route_ties_to_higher_id(L, k):
        idx, alpha = O.route(np.asarray(L)[:, ::-1], k)
        return np.asarray(L).shape[1] - 1 - idx, alpha

    def route_softmax_over_all(L, k):
        idx, _ = O.route(L, k)
        L = np.asarray(L, np.float64)
        w = np.exp(L - L.max(1, keepdims=True))
        return idx, np.take_along_axis(w / w.sum(1, keepdims=True), idx, 1)

    assert route_pin_mismatches(route_ties_to_higher_id) > 0
    assert route_alpha_pin_error(route_softmax_over_all) > 1e-3
    real_sigmoid = O.sigmoid
    with monkeypatch.context() as m:
        m.setattr(O, "sigmoid", lambda z: real_sigmoid(2 * z))
        assert swiglu_forward_pin_error()[0] > 1e-3
    real_router = O.router_grad

    def router_scaled_by_alpha(rop, idx, g, phi, w_down, pairs=None):
        # returns alpha_u * g_t . y_u (the gradient of the alpha-scaled output row)
        T, k = np.asarray(idx).shape
        a = fp64_consistent_inputs(0)["alpha"].reshape(-1)
        return real_router(rop, idx, g, phi, w_down, pairs) * (a if a.size == T * k else 1.0)

    def router_ignores_selection(rop, idx, g, phi, w_down, pairs=None):
        return real_router(np.zeros_like(np.asarray(rop)), idx, g, phi, w_down, pairs)

    def router_first_choice_expert(rop, idx, g, phi, w_down, pairs=None):
        idx = np.asarray(idx).copy()
        idx[:, 1:] = idx[:, :1]
        return real_router(rop, idx, g, phi, w_down, pairs)

    with monkeypatch.context() as m:
        m.setattr(O, "router_grad", router_scaled_by_alpha)
        assert router_autograd_pin_error() > 1e-3
    with monkeypatch.context() as m:
        m.setattr(O, "router_grad", router_first_choice_expert)
        assert router_autograd_pin_error() > 1e-3
    with monkeypatch.context() as m:
        m.setattr(O, "router_grad", router_ignores_selection)
        with pytest.raises(AssertionError):
            router_masked_pin_error()


@pytest.mark.parametrize("name", ["tiny_f32", "load_example"])
def test_generator_shapes(name):
    wl = W.WORKLOADS[name]
    inp = W.generate(wl, "cpu")
    assert inp["topk_idx"].shape == (wl.T, wl.k)
    assert inp["h"].shape == (wl.T, wl.k, 2 * wl.I)
    assert inp["phi"].shape == (wl.T, wl.k, wl.I)
    assert torch.allclose(inp["alpha"].sum(1), torch.ones(wl.T), atol=1e-6)
    # no expert is chosen twice by one token
    for row in inp["topk_idx"].tolist():
        assert len(set(row)) == wl.k


# ------------------------------------------------- ablation score modes ---------------
def test_grad_sq_is_lrm_with_unit_alpha_and_unit_phi():
    rng = np.random.default_rng(5)
    T, k, H, I = 6, 3, 9, 4
    g = rng.normal(0, 1, (T, H))
    phi = rng.normal(0, 1, (T, k, I))
    phi /= np.linalg.norm(phi, axis=2, keepdims=True)
    assert np.allclose(O.grad_sq_scores(g, k), O.lrm_scores(np.ones((T, k)), g, phi), rtol=1e-12)


def test_grad_abs_closed_forms():
    rng = np.random.default_rng(6)
    T, k, H, c = 5, 2, 16, 0.37
    g = c * rng.choice([-1.0, 1.0], size=(T, H))
    assert np.allclose(O.grad_abs_scores(g, k), O.grad_sq_scores(g, k) / c, rtol=1e-12)
    onehot = np.zeros((3, H))
    onehot[np.arange(3), [2, 7, 11]] = [-4.0, 0.5, 3.0]
    assert np.allclose(O.grad_abs_scores(onehot, 2), [[4.0, 4.0], [0.5, 0.5], [3.0, 3.0]])


def test_gradient_only_scores_tie_within_a_token_and_pick_smaller_u():
    # all k pairs of a token score alike: selection falls back to the pair-index tie-break
    idx = np.array([[0, 1], [0, 1], [1, 0]])
    g = np.array([[1.0, 0.0], [2.0, 0.0], [1.0, 1.0]])
    for fn in (O.grad_sq_scores, O.grad_abs_scores):
        R = fn(g, 2)
        seg, kept, _ = O.select(idx, R, np.array([1, 1]), 2)
        # expert 0 owns pairs 0, 2, 5 with scores R[0,0], R[1,0], R[2,1]; expert 1 owns 1, 3, 4
        assert kept[0] == [0, 2, 5][int(np.argmax([R[0, 0], R[1, 0], R[2, 1]]))]
