"""Shared helpers of the tests: build/load the library, run the CUDA path, compare with the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import workloads as W

TOL = {"f32": 1e-5, "bf16": 1e-2}


def ensure_built():
    from pruned_expert_backward_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def rel_fro(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    d = np.linalg.norm(want)
    n = np.linalg.norm(got - want)
    if d == 0:
        return 0.0 if n == 0 else float("inf")
    return float(n / d)


def to_np(t):
    t = t.detach().cpu()
    return (t.double() if t.dtype.is_floating_point else t.long()).numpy()


def gpu_quotas(inp, wl):
    import pruned_expert_backward_gb300 as lrm
    kind, num, den, cap, expl = W.quota_policy(wl)
    ex = None if expl is None else torch.tensor(expl, dtype=torch.int32, device=inp["topk_idx"].device)
    return lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, kind, num, den, cap, explicit=ex)


def run_cuda_path(wl, seed=0, flags=0, quotas=None, cap=None, device="cuda", router_grad=False):
    import pruned_expert_backward_gb300 as lrm
    inp = W.generate(wl, device, seed=seed)
    loads, q = gpu_quotas(inp, wl)
    if quotas is not None:
        q = torch.as_tensor(np.asarray(quotas), dtype=torch.int32, device=device)
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, device=device, cap=cap,
                            flags=flags, router_grad=router_grad)
    pb.run(inp, q)
    torch.cuda.synchronize()
    return inp, loads, q, pb


def check_selection_bit_exact(inp, q, pb, E):
    """Oracle selection run on the GPU's own fp32 scores must match the GPU bit for bit."""
    idx = to_np(inp["topk_idx"])
    gpu_scores = pb.scores.cpu().numpy()
    seg, kept, rop = oracle.select(idx, gpu_scores, to_np(q), E)
    R = int(seg[-1])
    assert np.array_equal(to_np(pb.seg_offsets), seg)
    assert np.array_equal(to_np(pb.kept_pair)[:R], kept)
    assert np.array_equal(to_np(pb.row_of_pair)[: idx.size], rop)
    return seg, kept, rop


def check_selection_vs_fp64(inp, q, pb, E, rtol=1e-5):
    """Against fp64 scores: equal kept counts, and any disagreement only at the cutoff."""
    idx = to_np(inp["topk_idx"]).reshape(-1)
    R64 = oracle.lrm_scores(to_np(inp["alpha"]), to_np(inp["g"]), to_np(inp["phi"])).reshape(-1)
    seg64, kept64, _ = oracle.select(idx, R64, to_np(q), E)
    seg = to_np(pb.seg_offsets)
    assert np.array_equal(seg, seg64)
    kept = to_np(pb.kept_pair)
    for e in range(E):
        a = set(kept[seg[e]:seg[e + 1]].tolist())
        b = set(kept64[seg64[e]:seg64[e + 1]].tolist())
        diff = a ^ b
        if not diff:
            continue
        cut = min(R64[list(b)]) if b else 0.0
        for u in diff:
            assert abs(R64[u] - cut) <= rtol * cut, (e, u, R64[u], cut)
