"""Seeded synthetic workloads for the LRM-pruned MoE expert backward.

This module feeds BOTH the CUDA path and the oracle and therefore holds none of the
pruned backward's arithmetic (no score, no selection, no compaction, no gradient).
It draws the router logits, activations, upstream gradients and expert weights, and
runs the ordinary, unpruned SwiGLU expert forward that produces the state a
backward pass consumes (the routed pairs, their weights alpha, the pre-activations
h = [gate; up] and the down-projection input phi = SiLU(gate) * up).

Shapes follow the LRMoE articles' workloads ("LRMoE: Trimming Backward Work in
Memory-Bound MoE Training", section "What the measurements show": Qwen3-30B-A3B and
GLM4.5-106B-A12B MoE layers, sequence 8192 x microbatch 4 per GPU, BF16). No
weights or dataset exist here; random values of the same shapes stand in for them.

Pair layout is token-major: pair u = t * k + j is token t's j-th routed choice.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    H: int          # hidden size
    I: int          # expert intermediate size
    E: int          # experts
    k: int          # routed experts per token
    dtype: str      # "f32" or "bf16": storage type of x, g, h, phi and the weights
    zipf_s: float   # expert popularity skew of the router bias
    g_std: float    # std of the upstream gradient g
    quota: tuple    # ("ratio", num, den) | ("cap", c) | ("explicit", (q_0, ..., q_{E-1}))
    topk_idx: tuple = field(default=None)  # hand-built routing (T*k expert ids), else drawn

    @property
    def P(self) -> int:
        return self.T * self.k

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def _cap(T, k, E, frac_num=7, frac_den=10):
    # fixed per-expert row budget ceil(0.7 * T * k / E), exact integer arithmetic
    return (frac_num * T * k + frac_den * E - 1) // (frac_den * E)


WORKLOADS = {
    # tiny fp32 layer the oracle finishes in well under a second
    "tiny_f32": Workload("tiny_f32", 512, 256, 128, 8, 2, "f32", 1.0, 1.0, ("ratio", 8, 10)),
    # the articles' load example: loads [4, 2, 3] cut to quotas [3, 1, 2]
    "load_example": Workload("load_example", 9, 16, 8, 3, 1, "f32", 0.0, 1.0, ("explicit", (3, 1, 2)),
                             topk_idx=(0, 1, 2, 0, 2, 0, 1, 2, 0)),
    # Qwen3-30B-A3B-shaped layer, one 8192-token sequence, drop 20%
    "qwen3_t8k_d20": Workload("qwen3_t8k_d20", 8192, 2048, 768, 128, 8, "bf16", 1.0, 1e-3, ("ratio", 8, 10)),
    # Qwen3-30B-A3B-shaped layer at seq 8192 x microbatch 4, drop 0 / 20 / 30 %
    "qwen3_t32k_d0": Workload("qwen3_t32k_d0", 32768, 2048, 768, 128, 8, "bf16", 1.0, 1e-3, ("ratio", 1, 1)),
    "qwen3_t32k_d20": Workload("qwen3_t32k_d20", 32768, 2048, 768, 128, 8, "bf16", 1.0, 1e-3, ("ratio", 8, 10)),
    "qwen3_t32k_d30": Workload("qwen3_t32k_d30", 32768, 2048, 768, 128, 8, "bf16", 1.0, 1e-3, ("ratio", 7, 10)),
    # GLM4.5-106B-A12B-shaped routed-expert layer, drop 20 %
    "glm45_t32k_d20": Workload("glm45_t32k_d20", 32768, 4096, 1408, 128, 8, "bf16", 1.0, 1e-3, ("ratio", 8, 10)),
    # a smaller case of the GLM4.5-shaped layer for counter captures that replay each kernel many
    # times: the same H, I and k and the same mean retained rows per expert (8192 tokens over 32
    # experts), about 5 GB on the device
    "glm45_shape_t8k_e32": Workload("glm45_shape_t8k_e32", 8192, 4096, 1408, 32, 8, "bf16", 1.0, 1e-3,
                                    ("ratio", 8, 10)),
    # overload stress: Zipf 1.5 skew, fixed row budget per expert
    "qwen3_t64k_zipf15_cap": Workload("qwen3_t64k_zipf15_cap", 65536, 2048, 768, 128, 8, "bf16", 1.5, 1e-3,
                                      ("cap", _cap(65536, 8, 128))),
}


def small_workload(name, T, H, I, E, k, dtype="bf16", zipf_s=1.0, g_std=1e-3, quota=("ratio", 8, 10)):
    """An ad-hoc workload (parity tests at sizes spanning several tiles and a ragged tail)."""
    return Workload(name, T, H, I, E, k, dtype, zipf_s, g_std, quota)


def _randn(gen, shape, device, std=1.0):
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def generate(wl: Workload, device="cpu", seed: int = 0) -> dict:
    """Draw one seeded batch for `wl` on `device`.

    Draw order: router noise [T,E], x [T,H], g [T,H], W_gate_up [E,2I,H], W_down [E,H,I].
    Returns a dict of tensors on `device`:
      topk_idx int32 [T,k], alpha fp32 [T,k], x [T,H], g [T,H], h [T,k,2I] (gate first),
      phi [T,k,I], w_gate_up [E,2I,H], w_down [E,H,I] (the last six in wl.dtype), and the fp32
      router logits [T,E] the top-k was taken from (noise + bias; plain noise for an explicit routing).
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    dt = wl.torch_dtype

    # Router: logits N(0,1) plus log of Zipf(s) popularity (expert 0 hottest); the
    # top-k biased logits choose the experts and their softmax gives alpha.
    noise = _randn(gen, (T, E), dev)
    logits = noise
    if wl.topk_idx is not None:
        topk_idx = torch.tensor(wl.topk_idx, dtype=torch.int64, device=dev).view(T, k)
        chosen = torch.gather(noise, 1, topk_idx)
    else:
        w = torch.arange(1, E + 1, device=dev, dtype=torch.float64).pow(-wl.zipf_s)
        bias = torch.log(w / w.sum()).to(torch.float32)
        logits = noise + bias
        chosen, topk_idx = torch.topk(logits, k, dim=1, largest=True, sorted=True)
    alpha = torch.softmax(chosen, dim=1).to(torch.float32).contiguous()

    x = _randn(gen, (T, H), dev).to(dt)
    g = _randn(gen, (T, H), dev, wl.g_std).to(dt)
    w_gate_up = _randn(gen, (E, 2 * I, H), dev, 1.0 / math.sqrt(H)).to(dt)
    w_down = _randn(gen, (E, H, I), dev, 1.0 / math.sqrt(I)).to(dt)

    # Unpruned SwiGLU expert forward, computed in fp32 from the stored values and
    # rounded to the storage type: h_u = W_gate_up[e] x_t, phi_u = SiLU(gate_u) * up_u.
    h = torch.empty(T * k, 2 * I, device=dev, dtype=dt)
    flat_idx = topk_idx.reshape(-1)
    tok = torch.arange(T * k, device=dev) // k
    for e in range(E):
        sel = torch.nonzero(flat_idx == e).flatten()
        if sel.numel() == 0:
            continue
        xe = x.index_select(0, tok.index_select(0, sel))
        if dt == torch.float32:
            he = xe.double() @ w_gate_up[e].double().t()
        else:
            he = xe @ w_gate_up[e].t()  # bf16 operands, fp32 accumulation, bf16 result
        h.index_copy_(0, sel, he.to(dt))
    hf = h.float()
    gate, up = hf[:, :I], hf[:, I:]
    phi = (torch.nn.functional.silu(gate) * up).to(dt)

    return {
        "topk_idx": topk_idx.to(torch.int32).contiguous(),
        "alpha": alpha,
        "x": x.contiguous(),
        "g": g.contiguous(),
        "h": h.view(T, k, 2 * I).contiguous(),
        "phi": phi.view(T, k, I).contiguous(),
        "w_gate_up": w_gate_up.contiguous(),
        "w_down": w_down.contiguous(),
        "logits": logits.contiguous(),
    }


def quota_policy(wl: Workload):
    """The workload's quota rule as (kind, num, den, cap, explicit_list)."""
    q = wl.quota
    if q[0] == "ratio":
        return ("ratio", q[1], q[2], 0, None)
    if q[0] == "cap":
        return ("cap", 0, 0, q[1], None)
    return ("explicit", 0, 0, 0, list(q[1]))
