"""Python binding of include/lrm.h: the same entry points, taking torch CUDA tensors.

Argument marshalling only (shapes, dtypes, pointers, the current stream); every step of
the pruned backward runs in liblrm.so's kernels.  There is no CPU path: a missing
library, a CPU tensor or a failed status raises.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib as L


class LrmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        name = L.STATUS_NAMES.get(code, str(code))
        text = L.load().lrm_status_string(code).decode()
        super().__init__(f"{where}: {name} ({text})")


def _ok(code: int, where: str):
    if code != L.LRM_OK:
        raise LrmError(code, where)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return L.LRM_BF16
    if t.dtype == torch.float32:
        return L.LRM_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _cuda(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _opt(t, name, dtype=None):
    return None if t is None else _cuda(t, name, dtype)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def lrm_workspace_size(T: int, k: int, E: int, H: int, I: int, dtype: torch.dtype) -> int:
    out = C.c_size_t(0)
    dt = L.LRM_BF16 if dtype == torch.bfloat16 else L.LRM_F32
    _ok(L.load().lrm_workspace_size(T, k, E, H, I, dt, C.byref(out)), "lrm_workspace_size")
    return int(out.value)


def lrm_plan_quotas(topk_idx, E, kind, num=0, den=1, cap=0, explicit=None, loads=None, quotas=None,
                    dev_status=None):
    """kind: "ratio" (num/den), "cap" (cap) or "explicit" (explicit int32 [E] tensor)."""
    T, k = topk_idx.shape
    dev = topk_idx.device
    loads = torch.empty(E, dtype=torch.int32, device=dev) if loads is None else loads
    quotas = torch.empty(E, dtype=torch.int32, device=dev) if quotas is None else quotas
    kinds = {"ratio": L.LRM_QUOTA_RATIO, "cap": L.LRM_QUOTA_CAP, "explicit": L.LRM_QUOTA_EXPLICIT}
    _ok(L.load().lrm_plan_quotas(_cuda(topk_idx, "topk_idx", torch.int32), T, k, E, kinds[kind], num, den, cap,
                                 _opt(explicit, "explicit", torch.int32), _cuda(loads, "loads", torch.int32),
                                 _cuda(quotas, "quotas", torch.int32), _opt(dev_status, "dev_status", torch.int32),
                                 _stream()), "lrm_plan_quotas")
    return loads, quotas


def lrm_score(alpha, g, phi, scores=None, dev_status=None):
    T, H = g.shape
    k, I = phi.shape[-2], phi.shape[-1]
    if phi.numel() != T * k * I or alpha.numel() != T * k:
        raise ValueError("alpha [T,k], g [T,H], phi [T,k,I] expected")
    scores = torch.empty(T * k, dtype=torch.float32, device=g.device) if scores is None else scores
    _ok(L.load().lrm_score(_cuda(alpha, "alpha", torch.float32), _cuda(g, "g"), _cuda(phi, "phi", g.dtype), T, k,
                           H, I, _dt(g), _cuda(scores, "scores", torch.float32),
                           _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_score")
    return scores


def lrm_score_norms(alpha, g, phi_sq, scores=None, dev_status=None):
    """LRM score from the forward's ||phi_u||^2 (phi_sq fp32 [T,k] or [T*k]); phi is not read."""
    T, H = g.shape
    k = alpha.numel() // max(T, 1) if T > 0 else alpha.shape[-1]
    if phi_sq.numel() != alpha.numel():
        raise ValueError("alpha and phi_sq must both hold T*k values")
    scores = torch.empty(T * k, dtype=torch.float32, device=g.device) if scores is None else scores
    _ok(L.load().lrm_score_norms(_cuda(alpha, "alpha", torch.float32), _cuda(g, "g"),
                                 _cuda(phi_sq, "phi_sq", torch.float32), T, k, H, _dt(g),
                                 _cuda(scores, "scores", torch.float32), _opt(dev_status, "dev_status", torch.int32),
                                 _stream()), "lrm_score_norms")
    return scores


def lrm_route(logits, k, kind, num=0, den=1, cap=0, explicit=None, topk_idx=None, alpha=None, loads=None,
              quotas=None, ws=None, dev_status=None):
    """Router top-k + softmax weights + loads + quotas in one launch.  logits fp32 [T,E].
    Returns topk_idx int32 [T,k], alpha fp32 [T,k], loads int32 [E], quotas int32 [E]."""
    T, E = logits.shape
    dev = logits.device
    i32 = dict(dtype=torch.int32, device=dev)
    topk_idx = torch.empty(T, k, **i32) if topk_idx is None else topk_idx
    alpha = torch.empty(T, k, dtype=torch.float32, device=dev) if alpha is None else alpha
    loads = torch.empty(E, **i32) if loads is None else loads
    quotas = torch.empty(E, **i32) if quotas is None else quotas
    ws = torch.empty(4 * (E + 1), dtype=torch.uint8, device=dev) if ws is None else ws
    kinds = {"ratio": L.LRM_QUOTA_RATIO, "cap": L.LRM_QUOTA_CAP, "explicit": L.LRM_QUOTA_EXPLICIT}
    _ok(L.load().lrm_route(_cuda(logits, "logits", torch.float32), T, E, k, kinds[kind], num, den, cap,
                           _opt(explicit, "explicit", torch.int32), _cuda(topk_idx, "topk_idx", torch.int32),
                           _cuda(alpha, "alpha", torch.float32), _cuda(loads, "loads", torch.int32),
                           _cuda(quotas, "quotas", torch.int32), _cuda(ws, "ws"), ws.numel(),
                           _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_route")
    return topk_idx, alpha, loads, quotas


def lrm_swiglu_forward(h, phi=None, phi_sq=None, norms=True):
    """phi = SiLU(gate) * up of rows h [..., 2I] (gate first), plus ||phi||^2 per row when norms."""
    I = h.shape[-1] // 2
    P = h.numel() // (2 * I)
    phi = torch.empty(*h.shape[:-1], I, dtype=h.dtype, device=h.device) if phi is None else phi
    if norms and phi_sq is None:
        phi_sq = torch.empty(h.shape[:-1], dtype=torch.float32, device=h.device)
    _ok(L.load().lrm_swiglu_forward(_cuda(h, "h"), P, I, _dt(h), _cuda(phi, "phi", h.dtype),
                                    _opt(phi_sq if norms else None, "phi_sq", torch.float32), _stream()),
        "lrm_swiglu_forward")
    return phi, (phi_sq if norms else None)


def lrm_score_mode(alpha, g, phi, mode, scores=None, dev_status=None):
    """mode: "lrm", "grad_sq" (||g_t||^2) or "grad_abs" (||g_t||_1); phi gives k and I."""
    T, H = g.shape
    k, I = phi.shape[-2], phi.shape[-1]
    modes = {"lrm": L.LRM_SCORE_LRM, "grad_sq": L.LRM_SCORE_GRAD_SQ, "grad_abs": L.LRM_SCORE_GRAD_ABS}
    scores = torch.empty(T * k, dtype=torch.float32, device=g.device) if scores is None else scores
    _ok(L.load().lrm_score_mode(_opt(alpha, "alpha", torch.float32), _cuda(g, "g"), _opt(phi, "phi", g.dtype), T, k,
                                H, I, _dt(g), modes[mode], _cuda(scores, "scores", torch.float32),
                                _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_score_mode")
    return scores


def lrm_select(topk_idx, scores, quotas, E, cap=None, seg_offsets=None, kept_pair=None, row_of_pair=None,
               ws=None, dev_status=None):
    T, k = topk_idx.shape
    P = T * k
    dev = topk_idx.device
    cap = P if cap is None else int(cap)
    seg_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if seg_offsets is None else seg_offsets
    kept_pair = torch.empty(max(cap, 1), dtype=torch.int32, device=dev) if kept_pair is None else kept_pair
    row_of_pair = torch.empty(P, dtype=torch.int32, device=dev) if row_of_pair is None else row_of_pair
    if ws is None:
        ws = torch.empty(lrm_workspace_size(T, k, E, 8, 8, torch.float32), dtype=torch.uint8, device=dev)
    _ok(L.load().lrm_select(_cuda(topk_idx, "topk_idx", torch.int32), _cuda(scores, "scores", torch.float32),
                            _cuda(quotas, "quotas", torch.int32), T, k, E, cap,
                            _cuda(seg_offsets, "seg_offsets", torch.int32), _cuda(kept_pair, "kept_pair", torch.int32),
                            _cuda(row_of_pair, "row_of_pair", torch.int32), _cuda(ws, "ws"), ws.numel(),
                            _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_select")
    return seg_offsets, kept_pair, row_of_pair


def lrm_compact(row_of_pair, alpha, g, x, h, phi, cap, dy_c=None, x_c=None, h_c=None, phi_c=None, dy_only=False,
                dev_status=None, x_only=False, k=None, I=None):
    """dy_only: write only dy_c (the compaction-free variant; x_c, h_c, phi_c are returned as None).
    x_only: write dy_c and x_c (h and phi may be None: the variant that recomputes them; k and I
    must then be given)."""
    T, H = g.shape
    if phi is not None:
        k, I = phi.shape[-2], phi.shape[-1]
    elif k is None or I is None:
        raise ValueError("k and I are needed when phi is not given")
    dev, dt = g.device, g.dtype
    rows = max(int(cap), 1)
    dy_c = torch.empty(rows, H, dtype=dt, device=dev) if dy_c is None else dy_c
    if dy_only:
        x_c = h_c = phi_c = None
    else:
        x_c = torch.empty(rows, H, dtype=dt, device=dev) if x_c is None else x_c
        if x_only:
            h_c = phi_c = None
        else:
            h_c = torch.empty(rows, 2 * I, dtype=dt, device=dev) if h_c is None else h_c
            phi_c = torch.empty(rows, I, dtype=dt, device=dev) if phi_c is None else phi_c
    _ok(L.load().lrm_compact(_cuda(row_of_pair, "row_of_pair", torch.int32), _cuda(alpha, "alpha", torch.float32),
                             _cuda(g, "g"), _opt(x, "x", dt), _opt(h, "h", dt), _opt(phi, "phi", dt), T, k, H, I,
                             _dt(g), int(cap), _cuda(dy_c, "dy_c", dt), _opt(x_c, "x_c", dt),
                             _opt(h_c, "h_c", dt), _opt(phi_c, "phi_c", dt),
                             _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_compact")
    return dy_c, x_c, h_c, phi_c


def lrm_grouped_backward(seg_offsets, dy_c, x_c, h_c, phi_c, w_gate_up, w_down, cap, dw_gate_up=None,
                         dw_down=None, dh_c=None, dx_c=None, ws=None, flags=L.LRM_GEMM_DEFAULT, dev_status=None,
                         row_dot=None):
    """row_dot: optional fp32 [cap] output (dphi . phi of each retained row, for lrm_router_grad)."""
    E, H, I = w_down.shape
    dev, dt = w_down.device, w_down.dtype
    rows = max(int(cap), 1)
    dw_gate_up = torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev) if dw_gate_up is None else dw_gate_up
    dw_down = torch.empty(E, H, I, dtype=torch.float32, device=dev) if dw_down is None else dw_down
    dh_c = torch.empty(rows, 2 * I, dtype=dt, device=dev) if dh_c is None else dh_c
    dx_c = torch.empty(rows, H, dtype=dt, device=dev) if dx_c is None else dx_c
    if ws is None:
        ws_rows = int(cap) if row_dot is not None else 0
        ws = torch.empty(lrm_workspace_size(ws_rows, 1, E, H, I, dt), dtype=torch.uint8, device=dev)
    _ok(L.load().lrm_grouped_backward(
        _cuda(seg_offsets, "seg_offsets", torch.int32), _cuda(dy_c, "dy_c", dt), _cuda(x_c, "x_c", dt),
        _cuda(h_c, "h_c", dt), _cuda(phi_c, "phi_c", dt), _cuda(w_gate_up, "w_gate_up", dt),
        _cuda(w_down, "w_down", dt), E, H, I, _dt(w_down), int(cap),
        _cuda(dw_gate_up, "dw_gate_up", torch.float32), _cuda(dw_down, "dw_down", torch.float32),
        _cuda(dh_c, "dh_c", dt), _cuda(dx_c, "dx_c", dt), _opt(row_dot, "row_dot", torch.float32),
        _cuda(ws, "ws"), ws.numel(), int(flags),
        _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_grouped_backward")
    return dw_gate_up, dw_down, dh_c, dx_c


def lrm_grouped_backward_gather(seg_offsets, kept_pair, k, dy_c, x, h, phi, w_gate_up, w_down, cap,
                                dw_gate_up=None, dw_down=None, dh_c=None, dx_c=None, ws=None,
                                flags=L.LRM_GEMM_DEFAULT, dev_status=None, row_dot=None):
    """Compaction-free grouped backward: x [T,H], h [T,k,2I], phi [T,k,I] read in place via kept_pair."""
    E, H, I = w_down.shape
    dev, dt = w_down.device, w_down.dtype
    rows = max(int(cap), 1)
    dw_gate_up = torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev) if dw_gate_up is None else dw_gate_up
    dw_down = torch.empty(E, H, I, dtype=torch.float32, device=dev) if dw_down is None else dw_down
    dh_c = torch.empty(rows, 2 * I, dtype=dt, device=dev) if dh_c is None else dh_c
    dx_c = torch.empty(rows, H, dtype=dt, device=dev) if dx_c is None else dx_c
    if ws is None:
        ws_rows = int(cap) if row_dot is not None else 0
        ws = torch.empty(lrm_workspace_size(ws_rows, 1, E, H, I, dt), dtype=torch.uint8, device=dev)
    _ok(L.load().lrm_grouped_backward_gather(
        _cuda(seg_offsets, "seg_offsets", torch.int32), _cuda(kept_pair, "kept_pair", torch.int32), x.shape[0], int(k),
        _cuda(dy_c, "dy_c", dt), _cuda(x, "x", dt), _cuda(h, "h", dt), _cuda(phi, "phi", dt),
        _cuda(w_gate_up, "w_gate_up", dt), _cuda(w_down, "w_down", dt), E, H, I, _dt(w_down), int(cap),
        _cuda(dw_gate_up, "dw_gate_up", torch.float32), _cuda(dw_down, "dw_down", torch.float32),
        _cuda(dh_c, "dh_c", dt), _cuda(dx_c, "dx_c", dt), _opt(row_dot, "row_dot", torch.float32),
        _cuda(ws, "ws"), ws.numel(), int(flags), _opt(dev_status, "dev_status", torch.int32), _stream()),
        "lrm_grouped_backward_gather")
    return dw_gate_up, dw_down, dh_c, dx_c


def lrm_recompute_forward(seg_offsets, x_c, w_gate_up, cap, h_c=None, phi_c=None, ws=None, flags=L.LRM_GEMM_DEFAULT,
                          dev_status=None):
    """h_c = W_gate_up[e] x_c and phi_c = SiLU(gate) * up for the retained rows (the saved forward
    state recomputed from x).  Returns (h_c [cap,2I], phi_c [cap,I])."""
    E, I2, H = w_gate_up.shape
    I = I2 // 2
    dev, dt = w_gate_up.device, w_gate_up.dtype
    rows = max(int(cap), 1)
    h_c = torch.empty(rows, 2 * I, dtype=dt, device=dev) if h_c is None else h_c
    phi_c = torch.empty(rows, I, dtype=dt, device=dev) if phi_c is None else phi_c
    if ws is None:
        ws = torch.empty(lrm_workspace_size(0, 1, E, H, I, dt), dtype=torch.uint8, device=dev)
    _ok(L.load().lrm_recompute_forward(_cuda(seg_offsets, "seg_offsets", torch.int32), _cuda(x_c, "x_c", dt),
                                       _cuda(w_gate_up, "w_gate_up", dt), E, H, I, _dt(w_gate_up), int(cap),
                                       _cuda(h_c, "h_c", dt), _cuda(phi_c, "phi_c", dt), _cuda(ws, "ws"), ws.numel(),
                                       int(flags), _opt(dev_status, "dev_status", torch.int32), _stream()),
        "lrm_recompute_forward")
    return h_c, phi_c


def lrm_router_grad(row_of_pair, alpha, row_dot, T, k, cap, dalpha=None):
    """dL/dalpha [T*k] fp32 of the retained pairs (0 for dropped ones) from lrm_grouped_backward's row_dot."""
    dalpha = torch.empty(T * k, dtype=torch.float32, device=alpha.device) if dalpha is None else dalpha
    _ok(L.load().lrm_router_grad(_cuda(row_of_pair, "row_of_pair", torch.int32), _cuda(alpha, "alpha", torch.float32),
                                 _opt(row_dot, "row_dot", torch.float32), T, k, int(cap),
                                 _cuda(dalpha, "dalpha", torch.float32), _stream()), "lrm_router_grad")
    return dalpha


def lrm_scatter_dx(row_of_pair, dx_c, T, k, dx=None, cap=None, dev_status=None):
    """cap: rows of dx_c that row_of_pair may name (default: all of dx_c's rows)."""
    H = dx_c.shape[1]
    cap = dx_c.shape[0] if cap is None else int(cap)
    if cap > dx_c.shape[0]:
        raise ValueError(f"cap {cap} exceeds the {dx_c.shape[0]} rows of dx_c")
    dx = torch.empty(T, H, dtype=dx_c.dtype, device=dx_c.device) if dx is None else dx
    _ok(L.load().lrm_scatter_dx(_cuda(row_of_pair, "row_of_pair", torch.int32), _cuda(dx_c, "dx_c"), T, k, H,
                                _dt(dx_c), cap, _cuda(dx, "dx", dx_c.dtype),
                                _opt(dev_status, "dev_status", torch.int32), _stream()), "lrm_scatter_dx")
    return dx


class PrunedBackward:
    """The whole pruned expert backward for one fixed problem size, with every buffer
    allocated once (device memory from torch).  `run` queues score -> select -> compact ->
    grouped backward -> scatter on the current stream; no host synchronisation.

    cap defaults to T*k, which can never overflow; a caller that knows sum(min(quota, load))
    may pass it to shrink the compacted buffers.  router_grad=True also produces dL/dalpha of
    every pair (`dalpha`, fp32 [T*k]; 0 for dropped pairs).
    compaction: "materialised" (the pages' physical compaction of dY, x, h, phi), "gather" (only dY
    is compacted; x, h, phi rows are read in place) or "recompute" (the forward kept x and
    ||phi_u||^2 only: dY and x are compacted and h, phi are recomputed for the retained rows)."""

    def __init__(self, T, k, E, H, I, dtype=torch.bfloat16, device="cuda", cap=None, flags=L.LRM_GEMM_DEFAULT,
                 router_grad=False, compaction="materialised"):
        if compaction not in ("materialised", "gather", "recompute"):
            raise ValueError("compaction: 'materialised' (the pages' physical compaction), 'gather' or 'recompute'")
        self.T, self.k, self.E, self.H, self.I = T, k, E, H, I
        self.dtype, self.flags, self.router_grad = dtype, flags, router_grad
        self.gather = compaction == "gather"
        self.recompute = compaction == "recompute"
        self.cap = T * k if cap is None else int(cap)
        dev = torch.device(device)
        rows = max(self.cap, 1)
        i32 = dict(dtype=torch.int32, device=dev)
        self.scores = torch.empty(T * k, dtype=torch.float32, device=dev)
        self.seg_offsets = torch.empty(E + 1, **i32)
        self.kept_pair = torch.empty(rows, **i32)
        self.row_of_pair = torch.empty(max(T * k, 1), **i32)
        self.dy_c = torch.empty(rows, H, dtype=dtype, device=dev)
        # the compaction-free variant keeps x, h, phi where they are
        self.x_c = None if self.gather else torch.empty(rows, H, dtype=dtype, device=dev)
        self.h_c = None if self.gather else torch.empty(rows, 2 * I, dtype=dtype, device=dev)
        self.phi_c = None if self.gather else torch.empty(rows, I, dtype=dtype, device=dev)
        self.dh_c = torch.empty(rows, 2 * I, dtype=dtype, device=dev)
        self.dx_c = torch.empty(rows, H, dtype=dtype, device=dev)
        self.dw_gate_up = torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev)
        self.dw_down = torch.empty(E, H, I, dtype=torch.float32, device=dev)
        self.dx = torch.empty(T, H, dtype=dtype, device=dev)
        self.ws = torch.empty(lrm_workspace_size(T, k, E, H, I, dtype), dtype=torch.uint8, device=dev)
        self.dev_status = torch.zeros(1, **i32)
        self.row_dot = torch.empty(rows, dtype=torch.float32, device=dev) if router_grad else None
        self.dalpha = torch.empty(max(T * k, 1), dtype=torch.float32, device=dev) if router_grad else None

    def run(self, inp, quotas):
        """inp: dict with topk_idx [T,k] int32, alpha [T,k] fp32, x, g [T,H], h [T,k,2I], phi [T,k,I],
        w_gate_up [E,2I,H], w_down [E,H,I] (CUDA), and optionally phi_sq fp32 [T,k] (||phi_u||^2 from
        lrm_swiglu_forward; the score then reads it instead of phi).  quotas: int32 [E] (CUDA).
        compaction="recompute" needs phi_sq and neither h nor phi."""
        if self.recompute:
            return self._run_recompute(inp, quotas)
        if inp.get("phi_sq") is not None:  # the forward handed over ||phi_u||^2
            lrm_score_norms(inp["alpha"], inp["g"], inp["phi_sq"], scores=self.scores, dev_status=self.dev_status)
        else:
            lrm_score(inp["alpha"], inp["g"], inp["phi"], scores=self.scores, dev_status=self.dev_status)
        lrm_select(inp["topk_idx"], self.scores, quotas, self.E, cap=self.cap, seg_offsets=self.seg_offsets,
                   kept_pair=self.kept_pair, row_of_pair=self.row_of_pair, ws=self.ws, dev_status=self.dev_status)
        lrm_compact(self.row_of_pair, inp["alpha"], inp["g"], inp["x"], inp["h"], inp["phi"], self.cap,
                    dy_c=self.dy_c, x_c=self.x_c, h_c=self.h_c, phi_c=self.phi_c, dy_only=self.gather,
                    dev_status=self.dev_status)
        if self.gather:
            lrm_grouped_backward_gather(self.seg_offsets, self.kept_pair, self.k, self.dy_c, inp["x"], inp["h"],
                                        inp["phi"], inp["w_gate_up"], inp["w_down"], self.cap,
                                        dw_gate_up=self.dw_gate_up, dw_down=self.dw_down, dh_c=self.dh_c,
                                        dx_c=self.dx_c, ws=self.ws, flags=self.flags, dev_status=self.dev_status,
                                        row_dot=self.row_dot)
        else:
            lrm_grouped_backward(self.seg_offsets, self.dy_c, self.x_c, self.h_c, self.phi_c, inp["w_gate_up"],
                                 inp["w_down"], self.cap, dw_gate_up=self.dw_gate_up, dw_down=self.dw_down,
                                 dh_c=self.dh_c, dx_c=self.dx_c, ws=self.ws, flags=self.flags,
                                 dev_status=self.dev_status, row_dot=self.row_dot)
        lrm_scatter_dx(self.row_of_pair, self.dx_c, self.T, self.k, dx=self.dx, cap=self.cap,
                       dev_status=self.dev_status)
        if self.router_grad:
            lrm_router_grad(self.row_of_pair, inp["alpha"], self.row_dot, self.T, self.k, self.cap,
                            dalpha=self.dalpha)
        return self

    def _run_recompute(self, inp, quotas):
        if inp.get("phi_sq") is None:
            raise ValueError("compaction='recompute' scores from phi_sq (||phi_u||^2 of the forward)")
        lrm_score_norms(inp["alpha"], inp["g"], inp["phi_sq"], scores=self.scores, dev_status=self.dev_status)
        lrm_select(inp["topk_idx"], self.scores, quotas, self.E, cap=self.cap, seg_offsets=self.seg_offsets,
                   kept_pair=self.kept_pair, row_of_pair=self.row_of_pair, ws=self.ws, dev_status=self.dev_status)
        lrm_compact(self.row_of_pair, inp["alpha"], inp["g"], inp["x"], None, None, self.cap, dy_c=self.dy_c,
                    x_c=self.x_c, x_only=True, k=self.k, I=self.I, dev_status=self.dev_status)
        lrm_recompute_forward(self.seg_offsets, self.x_c, inp["w_gate_up"], self.cap, h_c=self.h_c, phi_c=self.phi_c,
                              ws=self.ws, flags=self.flags, dev_status=self.dev_status)
        lrm_grouped_backward(self.seg_offsets, self.dy_c, self.x_c, self.h_c, self.phi_c, inp["w_gate_up"],
                             inp["w_down"], self.cap, dw_gate_up=self.dw_gate_up, dw_down=self.dw_down,
                             dh_c=self.dh_c, dx_c=self.dx_c, ws=self.ws, flags=self.flags,
                             dev_status=self.dev_status, row_dot=self.row_dot)
        lrm_scatter_dx(self.row_of_pair, self.dx_c, self.T, self.k, dx=self.dx, cap=self.cap,
                       dev_status=self.dev_status)
        if self.router_grad:
            lrm_router_grad(self.row_of_pair, inp["alpha"], self.row_dot, self.T, self.k, self.cap,
                            dalpha=self.dalpha)
        return self

    def outputs(self):
        return {"scores": self.scores, "seg_offsets": self.seg_offsets, "kept_pair": self.kept_pair,
                "row_of_pair": self.row_of_pair, "dy_c": self.dy_c, "x_c": self.x_c, "h_c": self.h_c,
                "phi_c": self.phi_c, "dh_c": self.dh_c, "dx_c": self.dx_c, "dw_gate_up": self.dw_gate_up,
                "dw_down": self.dw_down, "dx": self.dx, "dev_status": self.dev_status,
                "row_dot": self.row_dot, "dalpha": self.dalpha}


class HostPipeline:
    """The pruned backward over batches held in pinned host memory.

    Two device copies of the per-step inputs (topk_idx, alpha, x, g, h, phi and the quotas) are
    kept: while step i computes on the current stream, step i+1's inputs travel host -> device on
    a copy stream into the other copy, so transfers overlap compute.  After every step
    its result (dX and seg_offsets) is copied back to pinned host buffers and the host waits for
    it.  The weights stay on the device.  All compute runs in liblrm.so's kernels (through
    PrunedBackward); this class only orders copies with CUDA events."""

    NAMES = ("topk_idx", "alpha", "x", "g", "h", "phi")

    def __init__(self, pb: PrunedBackward, w_gate_up, w_down):
        self.pb = pb
        self.w_gate_up, self.w_down = w_gate_up, w_down
        self.copy_stream = torch.cuda.Stream(device=w_down.device)
        self.sets = [None, None]
        self.quotas = [None, None]
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.free = [torch.cuda.Event(), torch.cuda.Event()]
        self.dx_host = torch.empty(pb.dx.shape, dtype=pb.dx.dtype).pin_memory()
        self.seg_host = torch.empty(pb.seg_offsets.shape, dtype=torch.int32).pin_memory()

    def _upload(self, slot, host_inp, host_quotas):
        if self.sets[slot] is None:
            self.sets[slot] = {n: torch.empty(host_inp[n].shape, dtype=host_inp[n].dtype,
                                              device=self.w_down.device) for n in self.NAMES}
            self.quotas[slot] = torch.empty(host_quotas.shape, dtype=torch.int32, device=self.w_down.device)
        with torch.cuda.stream(self.copy_stream):
            self.copy_stream.wait_event(self.free[slot])  # the step that last used this slot is done
            for n in self.NAMES:
                self.sets[slot][n].copy_(host_inp[n], non_blocking=True)
            self.quotas[slot].copy_(host_quotas, non_blocking=True)
            self.ready[slot].record(self.copy_stream)

    def run(self, batches, on_result=None):
        """batches: a list of (host_inputs dict, host_quotas int32 [E]) in pinned memory.
        Returns the retained row count of each step (read from the step's seg_offsets).
        on_result(i, dx_host, seg_offsets_host), if given, sees each step's result on the host
        (the buffers are reused by the next step)."""
        retained = []
        if not batches:
            return retained
        cur = torch.cuda.current_stream()
        self._upload(0, *batches[0])
        for i in range(len(batches)):
            slot = i & 1
            if i + 1 < len(batches):
                self._upload(slot ^ 1, *batches[i + 1])
            cur.wait_event(self.ready[slot])
            inp = dict(self.sets[slot], w_gate_up=self.w_gate_up, w_down=self.w_down)
            self.pb.run(inp, self.quotas[slot])
            self.free[slot].record(cur)
            self.dx_host.copy_(self.pb.dx, non_blocking=True)
            self.seg_host.copy_(self.pb.seg_offsets, non_blocking=True)
            cur.synchronize()
            retained.append(int(self.seg_host[-1]))
            if on_result is not None:
                on_result(i, self.dx_host, self.seg_host)
        return retained
