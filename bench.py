#!/usr/bin/env python3
"""Throughput of the LRM-pruned MoE expert backward on GB300: retained pairs/s.

One step = one pass of the whole hot path (score -> select -> compact -> grouped SwiGLU
expert backward -> scatter dX) over one batch of seeded synthetic input that is already
resident in HBM.  Default workload: the largest single-GPU configuration, the
GLM4.5-106B-A12B-shaped routed-expert layer at the articles' per-GPU batch (sequence
8192 x microbatch 4): T=32768, H=4096, I=1408, E=128, top-8, bf16, drop 20 %
(quota = ceil(0.8 * load)).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--workload NAME] [--no-cpu-baseline] [--no-extras]
Under torchrun (N > 1) every rank runs an independent batch (weak scaling, no collective on
the data path; a barrier brackets the timed region and the slowest rank's time is used).

--impl reference times the fp64 CPU oracle (the plain restatement of the method) on the
host cores, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "retained pairs/s through pruned expert backward; % of BF16 TC / HBM roofline"
UNIT = "pairs/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def quota_text(wl):
    q = wl.quota
    if q[0] == "ratio":
        return f"ceil({q[1]}/{q[2]} * load_e)"
    if q[0] == "cap":
        return f"min(load_e, {q[1]})"
    return f"explicit {list(q[1])}"


# ------------------------------------------------------------------ byte / flop models ----
def algorithmic(wl, R, T_any):
    """Bytes (or flops) each stage must move (or do).  b = element bytes; R retained rows;
    T_any tokens with at least one kept pair (compaction reads g_t, x_t once per such token)."""
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    P = T * k
    b = 2 if wl.dtype == "bf16" else 4
    return {
        "score": {"bytes": T * H * b + P * I * b + 4 * P + 4 * P},
        "select": {"bytes": 4 * P * 2 + 4 * P * 2 + 4 * P + 4 * R + 4 * (E + 1)},
        "compact": {"bytes": T_any * 2 * H * b + R * 3 * I * b + R * (2 * H + 3 * I) * b + 4 * P + 4 * P},
        "grouped": {"flops": 12 * H * I * R,
                    "bytes": R * (H + I) * b + 4 * E * H * I            # dW_down
                    + R * H * b + E * H * I * b + 2 * R * 2 * I * b     # dphi + SwiGLU
                    + R * (2 * I + H) * b + 8 * E * I * H               # dW_gate_up
                    + R * 2 * I * b + 2 * E * I * H * b + R * H * b},   # dX_c
        "scatter": {"bytes": R * H * b + T * H * b + 4 * P},
    }


# ------------------------------------------------------------------ ranks -----------------
def aggregate_over_ranks(ms, retained, dist=None, device="cpu"):
    """Whole-job view of one timed region: the slowest rank's milliseconds and the retained
    pairs of all ranks (each rank runs its own batch; no data moves between ranks)."""
    if dist is None:
        return float(ms), float(retained)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    r = torch.tensor([float(retained)], dtype=torch.float64, device=device)
    dist.all_reduce(r)
    return float(t.item()), float(r.item())


def pairs_per_second(retained_total, steps, ms):
    return retained_total * steps / (ms / 1e3)


# ------------------------------------------------------------------ clocks ----------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"lrm_clocks_{os.getpid()}.csv")
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ traffic record --------
def recorded_traffic(kernel_stage, workload):
    """DRAM bytes per call of a stage from the committed ncu record, if one was taken on this
    workload and on the current source of that kernel (the record stores a hash of the kernel's
    source file).  None otherwise: a record of another workload or of older code says nothing
    about this run."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        m = re.match(r"\s*stage=(\S+)\s+workload=(\S+)\s+source=(\S+)\s+sha=(\S+)\s+dram_bytes=(\d+)", line)
        if not m or m.group(1) != kernel_stage or m.group(2) != workload:
            continue
        src = os.path.join(ROOT, m.group(3))
        if not os.path.exists(src):
            return None
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != m.group(4):
            return None
        return {"workload": m.group(2), "bytes": int(m.group(5))}
    return None


# ------------------------------------------------------------------ oracle timing ---------
def oracle_inputs(inp):
    """The workload's tensors as numpy arrays for the oracle, floating point widened to fp64 where
    the tensors live (the widening is input preparation, not the oracle's work)."""
    return {n: (v.double() if v.dtype.is_floating_point else v).cpu().numpy()
            for n, v in inp.items() if n != "logits"}


class OracleSample:
    """The fp64 oracle on a bounded sample of a workload: a subset S of the experts.  One call runs
    the whole oracle (score, selection, compaction, expert backward, return to token order) on the
    tokens routed to an expert of S, with the quotas of the other experts set to 0.  An expert's
    selection and backward depend on its own pairs and rows only, so every retained row of S costs
    the oracle what it costs in the whole workload; the tokens' other pairs are scored too.  S takes
    experts in proportion to the retained rows they hold (see __init__) until one call takes about
    the target time; when one expert alone takes longer, its quota is cut to the rows that fit (its
    top rows by score: the same work per row)."""

    def __init__(self, wl, npi):
        import oracle
        self.oracle, self.wl, self.npi = oracle, wl, npi
        kind, num, den, cap, expl = W.quota_policy(wl)
        self.loads, self.quotas = oracle.plan_quotas(npi["topk_idx"], wl.E, kind, num, den, cap, expl)
        kept = np.minimum(np.maximum(self.quotas, 0), self.loads)
        # experts in the order of the retained rows they hold: the i-th pick is the expert that
        # holds the row at quantile vdc(i) (van der Corput: 1/2, 1/4, 3/4, 1/8, ...) of all retained
        # rows, so a sample of any size weighs experts by their share of the work
        ends = np.cumsum(kept)
        total = int(ends[-1]) if len(ends) else 0
        order, seen, i = [], set(), 1
        while total > 0 and len(seen) < int(np.count_nonzero(kept)) and i < 64 * wl.E:
            v, f, n = 0.0, 0.5, i
            while n:
                v += f * (n & 1)
                n >>= 1
                f *= 0.5
            e = int(np.searchsorted(ends, v * total, side="right"))
            if e < wl.E and kept[e] > 0 and e not in seen:
                seen.add(e)
                order.append(e)
            i += 1
        order += [e for e in range(wl.E) if e not in seen and kept[e] > 0]
        order += [e for e in range(wl.E) if kept[e] == 0]
        self.order = order
        self.kept = kept
        self.cum_rows = np.concatenate([[0], np.cumsum(kept[self.order])])
        self.n, self.frac = wl.E, 1.0
        self._sub = {}

    def quotas_for(self, n, frac=1.0):
        q = np.zeros_like(self.quotas)
        sel = self.order[:n]
        q[sel] = self.quotas[sel]
        if frac < 1.0 and n == 1:
            e = sel[0]
            q[e] = max(1, int(min(self.quotas[e], self.loads[e]) * frac))
        return q

    def inputs_for(self, n):
        """The tokens with a pair routed to one of the first n experts of the order (input
        preparation, outside the timed call)."""
        if n not in self._sub:
            idx = np.asarray(self.npi["topk_idx"])
            tok = np.nonzero(np.isin(idx, np.asarray(self.order[:n], dtype=idx.dtype)).any(axis=1))[0]
            sub = {}
            for name, v in self.npi.items():
                sub[name] = v if name in ("w_gate_up", "w_down") else np.ascontiguousarray(v[tok])
            self._sub = {n: (sub, int(tok.shape[0]))}
        return self._sub[n]

    def rows(self, n=None, frac=None):
        n = self.n if n is None else n
        frac = self.frac if frac is None else frac
        return int(np.minimum(np.maximum(self.quotas_for(n, frac), 0), self.loads).sum())

    def run(self, n=None, min_s=0.0, frac=None):
        """One oracle call on the first n experts of the order (repeated until min_s seconds have
        passed, for samples that take milliseconds); returns (kept rows, seconds per call)."""
        n = self.n if n is None else n
        frac = self.frac if frac is None else frac
        q = self.quotas_for(n, frac)
        sub, _ = self.inputs_for(n)
        reps, t0 = 0, time.perf_counter()
        while True:
            out = self.oracle.pruned_backward(sub, q)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= min_s:
                return int(out["seg_offsets"][-1]), dt / reps

    def calibrate(self, target_s, rounds=4):
        """Pick |S| (and, for one expert, the share of its rows) so that one call takes about
        target_s, from the measured cost per retained row, refined over a few calls (the cost of a
        row depends on its expert's size and on the tokens that come with it)."""
        def timed(n, frac=1.0):  # the faster of two calls: host timings are noisy
            r, t = self.run(n, frac=frac)
            return r, min(t, self.run(n, frac=frac)[1])

        n, frac = 1, 1.0
        self.run(n, frac=frac)  # warm-up: the first call also pays for thread start and page faults
        r, t = timed(n)
        for _ in range(rounds):
            if t > 1.5 * target_s and n == 1:
                frac = max(frac * target_s / t, 1.0 / max(1, int(self.kept[self.order[0]])))
                r, t = timed(1, frac)
                continue
            c = t / max(r, 1)
            m = 1
            while m < self.wl.E and c * self.cum_rows[m + 1] <= target_s:
                m += 1
            if m == n or frac < 1.0:
                break
            n = m
            r, t = timed(n)
            if t > 1.5 * target_s and n > 1:
                n = max(1, n // 2)
                r, t = timed(n)
        self.n, self.frac = n, frac
        return n

    def describe(self):
        _, ntok = self.inputs_for(self.n)
        share = "" if self.frac >= 1.0 else f" (its top {self.frac:.0%} by score)"
        return (f"fp64 numpy oracle on the {ntok} of {self.wl.T} tokens routed to {self.n} of {self.wl.E} "
                f"experts: score and selection of their {ntok * self.wl.k} pairs, backward of the "
                f"{self.rows()} retained rows of those experts{share}, per call")


_BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NVPL_BLAS_NUM_THREADS")


def oracle_baseline(wl, inp, target_s=12.0, single_target_s=6.0):
    """cpu_baseline of the bench line: the oracle on the host cores (all threads of numpy's BLAS pool),
    then, in a child process whose BLAS pool is held to one thread, the same on one thread; each on
    a sample sized to about its target time."""
    smp = OracleSample(wl, oracle_inputs(inp))
    smp.calibrate(target_s)
    R, dt = smp.run(min_s=1.0)
    out = {"value": round(R / dt, 1), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
           "sample": f"{smp.describe()} ({dt:.1f} s)"}
    del smp
    env = dict(os.environ, **{v: "1" for v in _BLAS_THREAD_VARS})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-thread", "--workload", wl.name,
                        "--oracle-target-s", str(single_target_s)], env=env, capture_output=True, text=True)
    try:
        out["single_thread"] = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        out["single_thread"] = {"unavailable": (r.stderr.strip().splitlines() or ["no output"])[-1][:200]}
    return out


def oracle_single_thread(wl, target_s):
    """Child process of oracle_baseline (started with every BLAS pool held to one thread)."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    smp = OracleSample(wl, oracle_inputs(W.generate(wl, dev, seed=0)))
    smp.calibrate(target_s)
    R, dt = smp.run(min_s=1.0)
    print(json.dumps({"value": round(R / dt, 1), "unit": UNIT, "cores": 1,
                      "sample": f"{smp.describe()} ({dt:.1f} s)"}), flush=True)


def cpu_threads():
    """Threads of numpy's BLAS pool: threadpoolctl's answer where it is installed, else the thread
    count the environment fixes, else every core (the BLAS libraries' default)."""
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    for v in _BLAS_THREAD_VARS:
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


# ------------------------------------------------------------------ main -------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="glm45_t32k_d20", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--simt", action="store_true", help="CUDA-core GEMMs instead of tcgen05 (comparison only)")
    ap.add_argument("--oracle-single-thread", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-target-s", type=float, default=6.0, help=argparse.SUPPRESS)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the widened rows timed after the headline step (router gradient, compaction-free, "
                         "forward-side steps, ablation scores)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = W.WORKLOADS[args.workload]

    if args.oracle_single_thread:
        return oracle_single_thread(wl, args.oracle_target_s)
    if args.impl == "reference":
        return reference_arm(args, wl, rank, world)

    import pruned_expert_backward_gb300 as lrm
    from pruned_expert_backward_gb300 import _lib

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    inp = W.generate(wl, dev, seed=rank)
    kind, num, den, cap, expl = W.quota_policy(wl)
    ex = None if expl is None else torch.tensor(expl, dtype=torch.int32, device=dev)
    loads, quotas = lrm.lrm_plan_quotas(inp["topk_idx"], wl.E, kind, num, den, cap, explicit=ex)
    flags = _lib.LRM_GEMM_FORCE_SIMT if (args.simt or wl.dtype == "f32") else _lib.LRM_GEMM_DEFAULT
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, device=dev, flags=flags)
    stream = torch.cuda.current_stream()

    stages = ["score", "select", "compact", "grouped", "scatter"]

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        lrm.lrm_score(inp["alpha"], inp["g"], inp["phi"], scores=pb.scores, dev_status=pb.dev_status)
        if evs is not None:
            evs[1].record(stream)
        lrm.lrm_select(inp["topk_idx"], pb.scores, quotas, wl.E, cap=pb.cap, seg_offsets=pb.seg_offsets,
                       kept_pair=pb.kept_pair, row_of_pair=pb.row_of_pair, ws=pb.ws, dev_status=pb.dev_status)
        if evs is not None:
            evs[2].record(stream)
        lrm.lrm_compact(pb.row_of_pair, inp["alpha"], inp["g"], inp["x"], inp["h"], inp["phi"], pb.cap,
                        dy_c=pb.dy_c, x_c=pb.x_c, h_c=pb.h_c, phi_c=pb.phi_c, dev_status=pb.dev_status)
        if evs is not None:
            evs[3].record(stream)
        lrm.lrm_grouped_backward(pb.seg_offsets, pb.dy_c, pb.x_c, pb.h_c, pb.phi_c, inp["w_gate_up"],
                                 inp["w_down"], pb.cap, dw_gate_up=pb.dw_gate_up, dw_down=pb.dw_down,
                                 dh_c=pb.dh_c, dx_c=pb.dx_c, ws=pb.ws, flags=flags, dev_status=pb.dev_status)
        if evs is not None:
            evs[4].record(stream)
        lrm.lrm_scatter_dx(pb.row_of_pair, pb.dx_c, wl.T, wl.k, dx=pb.dx, cap=pb.cap, dev_status=pb.dev_status)
        if evs is not None:
            evs[5].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = int(pb.dev_status.item())
    if st != 0:
        raise SystemExit(f"device status {st} after warm-up")
    R = int(pb.seg_offsets[-1].item())
    rop = pb.row_of_pair.view(wl.T, wl.k)
    T_any = int((rop >= 0).any(dim=1).sum().item())

    # The timed steps carry no events between the stages: an event recorded between two kernels
    # of the chain stops the next one from launching while the previous one drains.  The stage
    # breakdown comes from a second pass of the same steps with an event at every stage boundary.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clk = clocks.stop()
    total_ms, R_total = aggregate_over_ranks(t_start.elapsed_time(t_end), R, pg, dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    stage_ms = {s: 0.0 for s in stages}
    for e in evs:
        for j, s in enumerate(stages):
            stage_ms[s] += e[j].elapsed_time(e[j + 1])
    stage_ms = {s: v / args.steps for s, v in stage_ms.items()}
    pass_step_ms = sorted(e[0].elapsed_time(e[len(stages)]) for e in evs)
    ms_per_step = total_ms / args.steps
    value = pairs_per_second(R_total, args.steps, total_ms)

    # ---- end-to-end through the public API with pinned host buffers ------------------------
    e2e = end_to_end(args, wl, inp, quotas, pb, step, stream, R_total, pg, dev)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    pk = peaks()
    alg = algorithmic(wl, R, T_any)
    stage_info = {}
    for s in stages:
        ms = stage_ms[s]
        d = {"ms": round(ms, 4)}
        if "bytes" in alg[s]:
            gbs = alg[s]["bytes"] / (ms / 1e3) / 1e9
            d.update({"alg_bytes": alg[s]["bytes"], "GB/s": round(gbs, 1),
                      "frac_hbm": round(gbs / pk["hbm_gbs"], 4)})
        if "flops" in alg[s]:
            tf = alg[s]["flops"] / (ms / 1e3) / 1e12
            d.update({"alg_flops": alg[s]["flops"], "TFLOP/s": round(tf, 1),
                      "frac_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 4)})
        stage_info[s] = d
    # the memory-bound stages together (score, selection, compaction, scatter): their bytes over their
    # summed time, against the same HBM bar as each of them
    mem = [s for s in stages if s != "grouped"]
    mem_ms = sum(stage_ms[s] for s in mem)
    mem_bytes = sum(alg[s]["bytes"] for s in mem)
    mem_gbs = mem_bytes / (mem_ms / 1e3) / 1e9
    memory_stages = {"stages": mem, "ms": round(mem_ms, 4), "alg_bytes": mem_bytes, "GB/s": round(mem_gbs, 1),
                     "frac_hbm": round(mem_gbs / pk["hbm_gbs"], 4)}
    dom = max(stages, key=lambda s: stage_ms[s])
    tr = recorded_traffic(dom, wl.name)
    # the binding roofline of the dominant stage is the one whose ideal time is longer
    t_hbm = alg[dom]["bytes"] / (pk["hbm_gbs"] * 1e9)
    t_tc = alg[dom].get("flops", 0) / (pk["bf16_tflops_sustained"] * 1e12) if wl.dtype == "bf16" else 0.0
    if t_tc > t_hbm:
        ach = alg[dom]["flops"] / (stage_ms[dom] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": f"lrm_grouped_backward ({dom})", "achieved": round(ach, 2),
                "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops_sustained"], 4),
                "peak_kind": f"bf16 dense, sustained, {pk['source']}"}
    else:
        ach = alg[dom]["bytes"] / (stage_ms[dom] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": f"lrm_grouped_backward ({dom})" if dom == "grouped" else dom,
                "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "peak_kind": f"HBM copy, {pk['source']}"}
    roof["ideal_ms"] = {"hbm": round(t_hbm * 1e3, 4), "tensor": round(t_tc * 1e3, 4)}
    roof["traffic"] = tr["bytes"] if tr else None
    if tr:
        roof["traffic_workload"] = tr["workload"]

    nxt = None if args.no_extras else next_rows(args, wl, inp, quotas, flags, dev, stream, ms_per_step, pk)
    launches = pb_launches(wl, flags)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "pairs": wl.P, "retained_pairs": R, "quota": quota_text(wl), "zipf_s": wl.zipf_s,
                   "gemm": "simt" if flags else "tcgen05", "parallelism": f"replicas{world}" if world > 1 else "1gpu",
                   "l2": "no flush: every step streams > 1 GB (inputs, compacted buffers, weights, fp32 dW) "
                         "through a 129 MB L2"},
        "roofline": roof,
        "stages": stage_info,
        "memory_stages": memory_stages,
        "stages_pass": {"ms_per_step": round(sum(stage_ms.values()), 4),
                        "step_ms_median": round(pass_step_ms[len(pass_step_ms) // 2], 4),
                        "step_ms_min": round(pass_step_ms[0], 4),
                        "how": "a second pass of the same steps with an event at every stage boundary"},
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "next_rows": nxt,
    }
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = oracle_baseline(wl, inp)
    print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


def _event_ms(fn, n, stream):
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def _graph_ms(fn, n, stream, reps=20):
    """Per-call device time of a short launch sequence: `reps` calls captured in one CUDA graph,
    replayed n times (host launch overhead would otherwise dominate microsecond kernels)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (n * reps)


def next_rows(args, wl, inp, quotas, flags, dev, stream, ms_step, pk):
    """Widened rows, timed apart from the headline step (same inputs, same stream): the step with
    the routing-weight gradient added (fused dphi . phi parts, their ordered sum, and the division /
    return to pair order), the forward-side steps (router with quotas, SwiGLU with row norms, score
    from norms) and the gradient-only ablation scores."""
    import pruned_expert_backward_gb300 as lrm
    n = max(10, min(args.steps, 50))
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, device=dev, flags=flags,
                            router_grad=True)
    ms_rg = _event_ms(lambda: pb.run(inp, quotas), n, stream)
    ms_rk = _graph_ms(lambda: lrm.lrm_router_grad(pb.row_of_pair, inp["alpha"], pb.row_dot, wl.T, wl.k, pb.cap,
                                                  dalpha=pb.dalpha), n, stream)
    st = int(pb.dev_status.item())
    R = int(pb.seg_offsets[-1].item())
    del pb
    b = 2 if wl.dtype == "bf16" else 4
    out = {"router_grad": {"ms_per_step": round(ms_rg, 4), "added_ms": round(ms_rg - ms_step, 4),
                           "router_grad_kernel_ms": round(ms_rk, 4), "steps": n, "dev_status": st}}
    # compaction-free variant: only dy_c is compacted; x / h / phi rows are gathered by index
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, device=dev, flags=flags,
                            compaction="gather")
    ms_g = _event_ms(lambda: pb.run(inp, quotas), n, stream)
    out["compaction_free"] = {"ms_per_step": round(ms_g, 4), "value": round(R / (ms_g / 1e3), 1), "unit": UNIT,
                              "vs_materialised": round(ms_step / ms_g, 4), "steps": n,
                              "dev_status": int(pb.dev_status.item())}
    del pb
    # recompute variant: the forward kept x and ||phi_u||^2 only; the retained rows' h and phi are
    # recomputed from x (one more var-M GEMM) instead of being compacted from saved state
    _, phi_sq = lrm.lrm_swiglu_forward(inp["h"])
    lean = {nm: v for nm, v in inp.items() if nm not in ("h", "phi")}
    lean["phi_sq"] = phi_sq
    pb = lrm.PrunedBackward(wl.T, wl.k, wl.E, wl.H, wl.I, dtype=wl.torch_dtype, device=dev, flags=flags,
                            compaction="recompute")
    ms_r = _event_ms(lambda: pb.run(lean, quotas), n, stream)
    b_el = 2 if wl.dtype == "bf16" else 4
    out["recompute"] = {"ms_per_step": round(ms_r, 4), "value": round(R / (ms_r / 1e3), 1), "unit": UNIT,
                        "vs_materialised": round(ms_step / ms_r, 4), "steps": n,
                        "extra_flops": 4 * wl.H * wl.I * R,
                        "forward_state_not_kept_bytes": wl.P * 3 * wl.I * b_el - 4 * wl.P,
                        "dev_status": int(pb.dev_status.item())}
    del pb, lean, phi_sq
    scores = torch.empty(wl.P, dtype=torch.float32, device=dev)

    def hbm(ms, by):
        gbs = by / (ms / 1e3) / 1e9
        return {"ms": round(ms, 4), "alg_bytes": by, "GB/s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}

    # forward-side steps: router top-k with loads and quotas in one launch, SwiGLU activation that
    # also emits ||phi||^2, and the score from those norms (phi not re-read)
    kind, num, den, cap, expl = W.quota_policy(wl)
    ex = None if expl is None else torch.tensor(expl, dtype=torch.int32, device=dev)
    ws = torch.empty(4 * (wl.E + 1), dtype=torch.uint8, device=dev)
    r_out = [torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev),
             torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev),
             torch.empty(wl.E, dtype=torch.int32, device=dev), torch.empty(wl.E, dtype=torch.int32, device=dev)]
    ms = _graph_ms(lambda: lrm.lrm_route(inp["logits"], wl.k, kind, num, den, cap, explicit=ex, topk_idx=r_out[0],
                                         alpha=r_out[1], loads=r_out[2], quotas=r_out[3], ws=ws), n, stream)
    out["route_with_quotas"] = hbm(ms, 4 * wl.T * wl.E + 8 * wl.P + 8 * wl.E)
    out["route_with_quotas"]["matches_generator_routing"] = bool(torch.equal(r_out[0], inp["topk_idx"]))
    phi = torch.empty_like(inp["phi"])
    phi_sq = torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev)
    ms = _graph_ms(lambda: lrm.lrm_swiglu_forward(inp["h"], phi=phi, phi_sq=phi_sq), n, stream)
    out["swiglu_forward_with_norms"] = hbm(ms, wl.P * 3 * wl.I * b + 4 * wl.P)
    ms = _graph_ms(lambda: lrm.lrm_swiglu_forward(inp["h"], phi=phi, norms=False), n, stream)
    out["swiglu_forward_without_norms"] = hbm(ms, wl.P * 3 * wl.I * b)
    ms = _graph_ms(lambda: lrm.lrm_score_norms(inp["alpha"], inp["g"], phi_sq, scores=scores), n, stream)
    out["score_from_norms"] = hbm(ms, wl.T * wl.H * b + 12 * wl.P)
    for name in ("grad_sq", "grad_abs"):
        ms = _graph_ms(lambda: lrm.lrm_score_mode(inp["alpha"], inp["g"], inp["phi"], name, scores=scores), n,
                       stream)
        by = wl.T * wl.H * b + 4 * wl.P
        out[f"score_{name}"] = {"ms": round(ms, 4), "alg_bytes": by,
                                "GB/s": round(by / (ms / 1e3) / 1e9, 1),
                                "frac_hbm": round(by / (ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
    return out


def pb_launches(wl, flags):
    """Kernels this library launches per step (memsets excluded)."""
    sel = (5 if wl.P >= 131072 else 4) if wl.P > 0 else 1  # the row scatter runs from 131072 pairs on
    grouped = 4 if flags else 5  # SIMT: 4 GEMMs; tcgen05: tile-plan kernel + 4 GEMMs
    return 1 + sel + 1 + grouped + 1


def end_to_end(args, wl, inp, quotas, pb, step, stream, R_total, pg, dev):
    """Same metric through the public API (HostPipeline): every step's inputs come from pinned
    host memory (copied on a copy stream, overlapping the previous step's compute) and every
    step's result (dX and the segment offsets) is read back to the host before the next step."""
    import pruned_expert_backward_gb300 as lrm
    names = lrm.HostPipeline.NAMES
    host = {n: inp[n].cpu().pin_memory() for n in names}
    host_q = quotas.cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + host_q.numel() * 4
    d2h = pb.dx.numel() * pb.dx.element_size() + pb.seg_offsets.numel() * 4
    steps = max(3, min(args.steps, 20))
    pipe = lrm.HostPipeline(pb, inp["w_gate_up"], inp["w_down"])
    pipe.run([(host, host_q)] * 3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    got = pipe.run([(host, host_q)] * steps)
    b.record(stream)
    torch.cuda.synchronize()
    assert all(r == got[0] for r in got)
    ms, _ = aggregate_over_ranks(a.elapsed_time(b), 0, pg, dev)
    return {"value": round(pairs_per_second(R_total, steps, ms), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 4),
            "path": "HostPipeline: pinned host inputs, H2D on a copy stream overlapping the previous step, "
                    "dX + seg_offsets read back every step; the fp32 weight gradients stay on the device "
                    "(the optimizer step that consumes them runs there)"}


def reference_arm(args, wl, rank, world):
    """fp64 CPU oracle on the host cores: each step is one oracle call on a bounded sample of the
    workload (OracleSample; the sample is sized before the warm-up steps to about 4 s per call, or
    to 150 s over all steps when that is less)."""
    if rank != 0:
        return
    # inputs drawn with the same generator, on the GPU where there is one (drawing the largest
    # workloads on the host takes minutes); the oracle itself runs on the host only
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = W.generate(wl, dev, seed=0)
    smp = OracleSample(wl, oracle_inputs(inp))
    del inp
    # per call about 4 s, less when many steps are asked for, so that the run ends in a few minutes
    smp.calibrate(min(4.0, max(0.25, 150.0 / max(1, args.steps + args.warmup))))
    for _ in range(max(0, args.warmup - 2)):
        smp.run()
    t0 = time.perf_counter()
    R = 0
    for _ in range(args.steps):
        R, _ = smp.run()
    dt = time.perf_counter() - t0
    value = R * args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "quota": quota_text(wl), "sample_experts": smp.n, "sample_rows": smp.rows()},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": smp.describe()},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
