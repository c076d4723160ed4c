"""Oracle of the LRM-pruned MoE expert backward: plain, slow, obviously correct, fp64, CPU, numpy.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline /
reference arm may import or run anything in this package. The product path (the
CUDA library and its Python binding) never imports it and shares no code with it.

Sources, all web pages about LRMoE (cited by title and section):
  [EN] "LRMoE: Trimming Backward Work in Memory-Bound MoE Training" (aimodeling.com, English)
  [ZH] the same article in Chinese (aimodeling.com), section "LRM:一个能分解的贡献度打分"
  [PT] "LRMoE poda a passagem reversa do MoE e acelera o treinamento em 21–45%" (news.hamidun.com),
       section "O que o LRMoE faz: forward completo, backward podado" (the five-step list)
  [ES] "LRMoE recorta el paso hacia atrás de MoE y acelera el entrenamiento entre un 21 y un 45%",
       section "Qué hace LRMoE: paso hacia delante completo, paso hacia atrás recortado"

The method's result (a pruned gradient) is an approximation with no closed form of its
own, so the oracle runs the algorithm's steps in the pages' order:
  quotas -> LRM score -> per-expert top-quota selection -> physical compaction ->
  grouped expert backward on the compacted rows -> back to the original token layout.
Every library call below (np.lexsort, the @ matmul, np.exp) is a plain step of that
definition; nothing is blocked, fused or reordered.

Notation: T tokens, k routed experts per token, pair u = t*k + j (token-major), E experts,
H hidden, I expert intermediate. h_u = [gate_u; up_u] (2I), phi_u = SiLU(gate_u)*up_u (I),
W_gate_up[e] (2I x H, gate rows first), W_down[e] (H x I), upstream gradient g_t (H) of the
layer output out_t = sum_j alpha_{t,j} W_down[e_{t,j}] phi_{t,j}.

Readings where the pages are silent:
  * phi is the input of the down projection, so G_u = (alpha_u g_t) phi_u^T is exactly
    pair u's term of dW_down ("protected expert projection", [EN] "LRM: ...").
  * A dropped pair contributes nothing to any part of the expert backward (dW_down,
    dW_gate_up, dX): only retained rows are packed and computed ([EN] "The part that is
    easy to get wrong"; [PT] step "Compactação física").
  * Ties in score are broken by pair index u ascending; inside a segment the compacted
    rows are in u ascending order.
  * The routing-weight gradient dL/dalpha_u = g_t . (W_down[e] phi_u) is computed for the
    retained pairs only; a dropped pair's is 0 (same reading as the one above).
  * Quotas are integers; ratio rule quota = ceil(num/den * load) in exact integer math,
    cap rule quota = min(load, cap); an explicit quota above the load keeps the whole load.

Pins: every function here is checked in tests/test_oracle.py against something other
than itself (see each docstring). Nothing here is "parity unpinned".
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------------------
# quotas  ([EN] "Backward demand is not a constant": before the expert forward the
# controller looks at each expert's routed demand and fixes a retention quota that holds
# for the whole layer call; [PT] second bullet)
# ----------------------------------------------------------------------------------------
def expert_loads(topk_idx, E):
    """load_e = number of routed pairs whose expert is e.
    Pinned: the articles' example loads [4, 2, 3] (tests/golden/load_example.json)."""
    flat = np.asarray(topk_idx).reshape(-1).astype(np.int64)
    return np.bincount(flat, minlength=E).astype(np.int64)


def plan_quotas(topk_idx, E, kind, num=0, den=1, cap=0, explicit=None):
    """Per-expert retention quota.
    ratio: ceil(num/den * load) computed as (num*load + den - 1) // den;
    cap:   min(load, cap);
    explicit: the given list, unchanged (selection keeps min(quota, load)).
    Pinned: exact-rational ceil/min over every load up to 10^6 and the worked example."""
    loads = expert_loads(topk_idx, E)
    if kind == "ratio":
        quotas = (num * loads + den - 1) // den
    elif kind == "cap":
        quotas = np.minimum(loads, cap)
    elif kind == "explicit":
        quotas = np.asarray(explicit, dtype=np.int64).copy()
        assert quotas.shape == (E,)
    else:
        raise ValueError(kind)
    return loads, quotas.astype(np.int64)


# ----------------------------------------------------------------------------------------
# forward-side steps beside the path  ([EN] "Backward demand is not a constant": the controller
# fixes each expert's quota from its routed demand before the expert forward, so the quota rule
# can run where the routing is decided; [EN] "LRM: a decomposable contribution score": the score
# needs only ||phi_u||^2 of the saved projection input, a number the forward can emit while it
# forms phi)
# ----------------------------------------------------------------------------------------
def route(logits, k):
    """Top-k routing of every token: the k largest logits in descending order (ties to the lower
    expert id) and alpha = softmax over those k logits, in fp64.
    Pinned: brute-force ranking on small integer logits full of ties; alpha sums to 1, follows the
    logit order, and for k = 2 equals the logistic function of the logit gap."""
    L = np.asarray(logits, dtype=np.float64)
    T, E = L.shape
    idx = np.zeros((T, k), dtype=np.int64)
    alpha = np.zeros((T, k))
    for t in range(T):
        order = np.lexsort((np.arange(E), -L[t]))   # logit descending, then expert id ascending
        idx[t] = order[:k]
        chosen = L[t, idx[t]]
        w = np.exp(chosen - chosen[0])
        alpha[t] = w / w.sum()
    return idx, alpha


def swiglu_forward(h, I):
    """Rows h = [gate ; up] (2I) -> phi = SiLU(gate) * up = gate * sigmoid(gate) * up (fp64) and
    phi_sq = ||phi||_2^2 of every row.
    Pinned: torch fp64 silu; the derivative of this phi is what swiglu_backward returns."""
    H2 = np.asarray(h, dtype=np.float64)
    gate, up = H2[..., :I], H2[..., I:]
    phi = gate * sigmoid(gate) * up
    return phi, np.sum(phi * phi, axis=-1)


def lrm_scores_from_norms(alpha, g, phi_sq):
    """R[t, j] = alpha[t,j]^2 * ||g_t||_2^2 * phi_sq[t,j]: the LRM score with ||phi_u||^2 handed in.
    Pinned: equals lrm_scores when phi_sq = ||phi_u||^2."""
    a = np.asarray(alpha, dtype=np.float64)
    G = np.asarray(g, dtype=np.float64)
    g2 = np.sum(G * G, axis=1)
    return a * a * g2[:, None] * np.asarray(phi_sq, dtype=np.float64)


# ----------------------------------------------------------------------------------------
# LRM score  ([EN] "LRM: a decomposable contribution score": G_u = (alpha_u g_t) phi_u^T is
# rank one, so ||G_u||_F^2 splits into routing strength alpha_u^2, backward signal
# ||g_t||^2 and expert-state magnitude ||phi_u||^2; [PT] "Seleção pela métrica LRM")
# ----------------------------------------------------------------------------------------
def lrm_scores(alpha, g, phi):
    """R[t, j] = alpha[t,j]^2 * ||g_t||_2^2 * ||phi[t,j]||_2^2 in fp64.
    alpha [T,k], g [T,H], phi [T,k,I] -> R [T,k].
    Pinned: equals the squared Frobenius norm of the explicit H x I outer product."""
    a = np.asarray(alpha, dtype=np.float64)
    gg = np.asarray(g, dtype=np.float64)
    pp = np.asarray(phi, dtype=np.float64)
    g_sq = np.sum(gg * gg, axis=1)            # ||g_t||^2, [T]
    phi_sq = np.sum(pp * pp, axis=2)          # ||phi_u||^2, [T,k]
    return (a * a) * g_sq[:, None] * phi_sq


# ----------------------------------------------------------------------------------------
# ablation scores  ([EN] "What the measurements show": LRM is compared with selecting by the
# squared gradient norm, by the absolute gradient magnitude, and with random dropping).
# Reading: the gradient-only rules look at the upstream gradient g_t of the pair's token alone,
# so the k pairs of a token score alike ("a gradient-only rule scores them as interchangeable",
# section "LRM: ..."); "absolute magnitude" is the L1 norm; random dropping selects on caller-
# drawn uniform numbers with the same top-quota rule.
# ----------------------------------------------------------------------------------------
def grad_sq_scores(g, k):
    """R[t, j] = ||g_t||_2^2 for every choice j of token t.
    Pinned: equals lrm_scores with alpha = 1 and a unit-norm phi."""
    gg = np.asarray(g, dtype=np.float64)
    return np.repeat(np.sum(gg * gg, axis=1)[:, None], k, axis=1)


def grad_abs_scores(g, k):
    """R[t, j] = ||g_t||_1 = sum_h |g_t[h]|.
    Pinned: on +-c vectors equals ||g||_2^2 / c; equals |g_t[h]| for a one-hot g_t."""
    gg = np.asarray(g, dtype=np.float64)
    return np.repeat(np.sum(np.abs(gg), axis=1)[:, None], k, axis=1)


# ----------------------------------------------------------------------------------------
# selection  ([PT]/[ES] "Seleção pela métrica LRM": inside the quota the highest-scoring
# pairs are kept; [EN] "Three things worth flagging": the guarantee covers an additive
# local objective, i.e. the kept set maximises the kept score sum per expert)
# ----------------------------------------------------------------------------------------
def select(topk_idx, scores, quotas, E):
    """Keep, per expert e, the min(quota_e, load_e) pairs with the largest score, ties to
    the smaller u.  Returns
      seg_offsets int64 [E+1]: exclusive prefix sum of the kept counts,
      kept_pair   int64 [R]:   kept pairs, expert-major, u ascending inside a segment,
      row_of_pair int64 [P]:   compacted row of each pair, -1 if dropped.
    Works on any score dtype (fp64 oracle scores, or fp32 scores compared exactly).
    Pinned: brute force over all subsets on small segments; the worked example."""
    flat_idx = np.asarray(topk_idx).reshape(-1).astype(np.int64)
    s = np.asarray(scores).reshape(-1)
    P = flat_idx.shape[0]
    q = np.asarray(quotas, dtype=np.int64)
    seg_offsets = np.zeros(E + 1, dtype=np.int64)
    kept_lists = []
    for e in range(E):
        pairs = np.nonzero(flat_idx == e)[0]            # u ascending
        keep_n = int(min(max(q[e], 0), pairs.shape[0]))
        # order by score descending, then u ascending (lexsort: last key is primary)
        order = np.lexsort((pairs, -s[pairs]))
        kept = np.sort(pairs[order[:keep_n]])
        kept_lists.append(kept)
        seg_offsets[e + 1] = seg_offsets[e] + keep_n
    kept_pair = np.concatenate(kept_lists) if kept_lists else np.zeros(0, np.int64)
    row_of_pair = np.full(P, -1, dtype=np.int64)
    row_of_pair[kept_pair] = np.arange(kept_pair.shape[0], dtype=np.int64)
    return seg_offsets, kept_pair.astype(np.int64), row_of_pair


# ----------------------------------------------------------------------------------------
# physical compaction  ([EN] "The part that is easy to get wrong": retained gradient rows
# and their saved activations are repacked into contiguous expert-specific buffers, with
# no padding; [PT] "Compactação física")
# ----------------------------------------------------------------------------------------
def compact(kept_pair, alpha, g, x, h, phi, k):
    """Gather the kept pairs' rows, in kept_pair order, in fp64:
      dY_c[r] = alpha_u * g_t,  X_c[r] = x_t,  H_c[r] = h_u,  Phi_c[r] = phi_u  (u = kept_pair[r], t = u // k).
    Pinned: the compacted backward equals the full-shape backward with dropped pairs'
    gradient rows zero-masked (the articles' negative result: masking gives the same
    numbers, only without the saving)."""
    kp = np.asarray(kept_pair, dtype=np.int64)
    t = kp // k
    # gather the rows first, then widen (same values; avoids widening whole tensors)
    a = np.asarray(alpha).reshape(-1)[kp].astype(np.float64)
    gg = np.asarray(g)[t].astype(np.float64)
    dY_c = a[:, None] * gg
    X_c = np.asarray(x)[t].astype(np.float64)
    hh = np.asarray(h)
    H_c = hh.reshape(-1, hh.shape[-1])[kp].astype(np.float64)
    pp = np.asarray(phi)
    Phi_c = pp.reshape(-1, pp.shape[-1])[kp].astype(np.float64)
    return dY_c, X_c, H_c, Phi_c


# ----------------------------------------------------------------------------------------
# grouped expert backward on the compacted rows  ([EN] "The part that is easy to get
# wrong": the retained row counts drive variable-size grouped GEMMs; the expert is the
# SwiGLU MLP whose down projection consumes phi)
# ----------------------------------------------------------------------------------------
def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def swiglu_backward(dphi, gate, up):
    """phi = SiLU(gate) * up, SiLU(z) = z * sigmoid(z).  With s = sigmoid(gate):
      d phi / d up   = gate * s
      d phi / d gate = up * (s + gate * s * (1 - s)) = up * s * (1 + gate * (1 - s)).
    Pinned: central finite differences in fp64, and torch fp64 autograd."""
    s = sigmoid(gate)
    dgate = dphi * up * s * (1.0 + gate * (1.0 - s))
    dup = dphi * gate * s
    return dgate, dup


def expert_backward(seg_offsets, dY_c, X_c, H_c, Phi_c, w_gate_up, w_down):
    """For each expert e over its segment rows (R_e of them):
      dW_down[e]    = dY_c[e]^T Phi_c[e]                         (H x I)
      dPhi          = dY_c[e] W_down[e]                          (R_e x I)
      [dgate; dup]  = SwiGLU backward of dPhi at H_c[e]          (R_e x 2I)
      dW_gate_up[e] = [dgate; dup]^T X_c[e]                      (2I x H)
      dX_c[e]       = [dgate; dup] W_gate_up[e]                  (R_e x H)
    An expert with no rows gets dW = 0.
    Pinned: with quota = load it equals torch fp64 autograd of the explicit forward."""
    E = len(seg_offsets) - 1
    Wgu = np.asarray(w_gate_up, dtype=np.float64)
    Wd = np.asarray(w_down, dtype=np.float64)
    H = Wd.shape[1]
    I = Wd.shape[2]
    R = dY_c.shape[0]
    dW_down = np.zeros((E, H, I))
    dW_gate_up = np.zeros((E, 2 * I, H))
    dH_c = np.zeros((R, 2 * I))
    dX_c = np.zeros((R, H))
    for e in range(E):
        r0, r1 = int(seg_offsets[e]), int(seg_offsets[e + 1])
        if r1 == r0:
            continue
        dy = dY_c[r0:r1]
        dW_down[e] = dy.T @ Phi_c[r0:r1]
        dphi = dy @ Wd[e]
        dgate, dup = swiglu_backward(dphi, H_c[r0:r1, :I], H_c[r0:r1, I:])
        dh = np.concatenate([dgate, dup], axis=1)
        dH_c[r0:r1] = dh
        dW_gate_up[e] = dh.T @ X_c[r0:r1]
        dX_c[r0:r1] = dh @ Wgu[e]
    return dW_gate_up, dW_down, dH_c, dX_c


# ----------------------------------------------------------------------------------------
# back to the original layout  ([PT] "Depois, o resultado volta ao layout original")
# ----------------------------------------------------------------------------------------
def scatter_dx(row_of_pair, dX_c, T, k):
    """dX[t] = sum over j = 0..k-1 (in that order) of dX_c[row_of_pair[t*k+j]] for kept pairs;
    a token with no kept pair gets 0.
    Pinned: with quota = load the whole path equals torch fp64 autograd's dL/dx."""
    rop = np.asarray(row_of_pair, dtype=np.int64).reshape(T, k)
    H = dX_c.shape[1]
    dX = np.zeros((T, H))
    for j in range(k):
        rows = rop[:, j]
        m = rows >= 0
        dX[m] += dX_c[rows[m]]
    return dX


# ----------------------------------------------------------------------------------------
# router gradient  (the layer output is out_t = sum_j alpha_{t,j} y_{t,j} with the expert
# output y_{t,j} = W_down[e] phi_{t,j}, so the loss gradient with respect to a routing weight
# is dL/dalpha_{t,j} = g_t . y_{t,j}.  The pages say nothing about it under pruning.  Reading:
# a dropped pair is removed from the whole expert backward, so its routing-weight gradient is
# 0 as well; a retained pair's is the exact one.)
# ----------------------------------------------------------------------------------------
def router_grad(row_of_pair, topk_idx, g, phi, w_down, pairs=None):
    """dalpha[u] = g_t . (W_down[e_u] phi_u) for a retained pair u = t*k + j (row_of_pair[u] >= 0),
    0 for a dropped one; returned flat, [T*k].  `pairs` limits the work to those pair indices
    (the rest stay 0), for sampled checks at large sizes.
    Pinned: with quota = load it equals torch fp64 autograd's dL/dalpha of the explicit forward;
    on a pruned selection it equals (dPhi_u . phi_u) / alpha_u with dPhi taken from the
    zero-masked full-shape rows."""
    idx = np.asarray(topk_idx).reshape(-1)
    rop = np.asarray(row_of_pair).reshape(-1)
    T = np.asarray(g).shape[0]
    k = idx.size // T if T > 0 else 1
    G = np.asarray(g, dtype=np.float64)
    Phi = np.asarray(phi, dtype=np.float64).reshape(idx.size, -1)
    Wd = np.asarray(w_down, dtype=np.float64)
    out = np.zeros(idx.size)
    todo = range(idx.size) if pairs is None else (int(u) for u in pairs)
    for u in todo:
        if rop[u] < 0:
            continue
        y = Wd[int(idx[u])] @ Phi[u]          # the expert's output for this pair (H)
        out[u] = float(G[u // k] @ y)
    return out


# ----------------------------------------------------------------------------------------
# the whole path
# ----------------------------------------------------------------------------------------
def pruned_backward(inp, quotas, scores=None):
    """Run score -> select -> compact -> grouped backward -> scatter on the inputs dict
    (numpy or torch CPU arrays: topk_idx [T,k], alpha [T,k], x [T,H], g [T,H], h [T,k,2I],
    phi [T,k,I], w_gate_up [E,2I,H], w_down [E,H,I]).  `scores` overrides the fp64 scores
    used for selection (e.g. the GPU's fp32 scores, for the bit-exact selection check)."""
    idx = _np(inp["topk_idx"])
    T, k = idx.shape
    E = _np(inp["w_down"]).shape[0]
    R_u = lrm_scores(_np(inp["alpha"]), _np(inp["g"]), _np(inp["phi"]))
    sel_scores = R_u if scores is None else _np(scores)
    seg, kept, rop = select(idx, sel_scores, quotas, E)
    dY_c, X_c, H_c, Phi_c = compact(kept, _np(inp["alpha"]), _np(inp["g"]), _np(inp["x"]),
                                    _np(inp["h"]), _np(inp["phi"]), k)
    dWgu, dWd, dH_c, dX_c = expert_backward(seg, dY_c, X_c, H_c, Phi_c,
                                            _np(inp["w_gate_up"]), _np(inp["w_down"]))
    dX = scatter_dx(rop, dX_c, T, k)
    return {"scores": R_u, "seg_offsets": seg, "kept_pair": kept, "row_of_pair": rop,
            "dY_c": dY_c, "X_c": X_c, "H_c": H_c, "Phi_c": Phi_c,
            "dH_c": dH_c, "dX_c": dX_c, "dw_gate_up": dWgu, "dw_down": dWd, "dx": dX}


# ----------------------------------------------------------------------------------------
# saved state recomputed from x  ([EN] "The part that is easy to get wrong": the pages insist on
# physically compacted rows; a variant that keeps less forward state recomputes, for the retained
# rows only, what the forward would have saved.  Reading: the forward keeps x and the score's
# ||phi_u||^2 (see swiglu_forward), and the backward forms h_u = W_gate_up[e] x_t and
# phi_u = SiLU(gate_u) * up_u again for the pairs it keeps.)
# ----------------------------------------------------------------------------------------
def recompute_saved_state(kept_pair, topk_idx, x, w_gate_up, k):
    """For the kept pairs u = kept_pair[r] (token t = u // k, expert e = topk_idx[u]):
      H_c[r] = W_gate_up[e] x_t  (2I: gate rows first),  Phi_c[r] = SiLU(gate) * up  (swiglu_forward),
    in fp64.  Pinned: the pruned backward on this recomputed state equals torch fp64 autograd of
    the explicit forward at quota = load; a gate/up swap fails that pin."""
    kp = np.asarray(kept_pair, dtype=np.int64)
    idx = np.asarray(topk_idx).reshape(-1).astype(np.int64)
    X = np.asarray(x)
    Wgu = np.asarray(w_gate_up)
    I = Wgu.shape[1] // 2
    H_c = np.zeros((kp.shape[0], 2 * I))
    for r, u in enumerate(kp):
        H_c[r] = Wgu[idx[u]].astype(np.float64) @ X[u // k].astype(np.float64)
    Phi_c, _ = swiglu_forward(H_c, I)
    return H_c, Phi_c


def pruned_backward_recompute(inp, quotas, scores=None):
    """The pruned backward of a forward that kept x and phi_sq = ||phi_u||^2 instead of h and phi:
    score from the norms, select, compact dY_c and X_c, recompute H_c and Phi_c for the kept rows,
    then the grouped backward and the return to token order.  inp holds topk_idx, alpha, x, g,
    phi_sq [T,k], w_gate_up, w_down.  `scores` overrides the selection scores as in pruned_backward.
    Pinned: with quota = load it equals torch fp64 autograd of the explicit forward; on inputs whose
    h and phi are the exact fp64 forward of x it equals pruned_backward (tests/test_oracle.py)."""
    idx = _np(inp["topk_idx"])
    T, k = idx.shape
    E = _np(inp["w_down"]).shape[0]
    R_u = lrm_scores_from_norms(_np(inp["alpha"]), _np(inp["g"]), _np(inp["phi_sq"]))
    sel_scores = R_u if scores is None else _np(scores)
    seg, kept, rop = select(idx, sel_scores, quotas, E)
    a = np.asarray(_np(inp["alpha"])).reshape(-1)[kept].astype(np.float64)
    t = kept // k
    dY_c = a[:, None] * np.asarray(_np(inp["g"]))[t].astype(np.float64)
    X_c = np.asarray(_np(inp["x"]))[t].astype(np.float64)
    H_c, Phi_c = recompute_saved_state(kept, idx, _np(inp["x"]), _np(inp["w_gate_up"]), k)
    dWgu, dWd, dH_c, dX_c = expert_backward(seg, dY_c, X_c, H_c, Phi_c,
                                            _np(inp["w_gate_up"]), _np(inp["w_down"]))
    dX = scatter_dx(rop, dX_c, T, k)
    return {"scores": R_u, "seg_offsets": seg, "kept_pair": kept, "row_of_pair": rop,
            "dY_c": dY_c, "X_c": X_c, "H_c": H_c, "Phi_c": Phi_c,
            "dH_c": dH_c, "dX_c": dX_c, "dw_gate_up": dWgu, "dw_down": dWd, "dx": dX}


def unpruned_backward(inp):
    """The ordinary expert backward over every routed pair (quota = load)."""
    idx = _np(inp["topk_idx"])
    E = _np(inp["w_down"]).shape[0]
    loads = expert_loads(idx, E)
    return pruned_backward(inp, loads)


def masked_backward(inp, quotas):
    """Full-shape backward: every routed pair is processed, dropped pairs' gradient rows
    are zero-masked instead of removed (the articles' 'selection without compaction')."""
    idx = _np(inp["topk_idx"])
    T, k = idx.shape
    E = _np(inp["w_down"]).shape[0]
    R_u = lrm_scores(_np(inp["alpha"]), _np(inp["g"]), _np(inp["phi"]))
    _, _, rop = select(idx, R_u, quotas, E)
    loads = expert_loads(idx, E)
    seg_all, all_pairs, rop_all = select(idx, R_u, loads, E)
    dY, X, Hh, Phi = compact(all_pairs, _np(inp["alpha"]), _np(inp["g"]), _np(inp["x"]),
                             _np(inp["h"]), _np(inp["phi"]), k)
    dropped = rop[all_pairs] < 0
    dY[dropped] = 0.0
    dWgu, dWd, dH, dX_rows = expert_backward(seg_all, dY, X, Hh, Phi,
                                             _np(inp["w_gate_up"]), _np(inp["w_down"]))
    dX = scatter_dx(rop_all, dX_rows, T, k)
    return {"dw_gate_up": dWgu, "dw_down": dWd, "dx": dX}


def _np(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if a.dtype.is_floating_point:
            a = a.double()
        return a.numpy()
    return np.asarray(a)
