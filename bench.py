#!/usr/bin/env python
"""Benchmark of the latent-MoE block on GB300: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one full block call (pre-norm, router, top-k, permutation, pooler,
pool norm, gate/up + SwiGLU, down, combine, unpooler, post-norm + residual)
over one batch of T synthetic tokens with the weights resident in HBM.  With
N > 1 (torchrun) every rank runs an independent replica on its own tokens
(the block is token-independent: no exchange on the data path); the time is
the max over ranks and ``value`` counts the tokens of all ranks.

``--impl reference`` times the fp64 CPU oracle (test infrastructure, a
deliberately slow reference) on the host cores over a bounded token sample of
the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "latent-MoE block tokens/s (BF16, NVFP4) at Muse shape; % of tensor/HBM roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------ distributed
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


# ------------------------------------------------------------------ roofline
def stage_costs(w: workloads.Workload, counts: np.ndarray):
    """Algorithmic bytes and FLOPs of each stage of one call (weights counted once per
    expert that receives at least one row; activations read/written once)."""
    T, D, L, E, I, k = w.T, w.D, w.L, w.E, w.I, w.k
    R = T * k
    used = int(np.count_nonzero(counts))
    bf, f4 = 2, 4
    xb = 4 if w.act == "f32" else 2
    # bytes per element of the pooler/expert/unpooler weights and of their activation operands:
    # bf16, or NVFP4 = half a byte of code + one E4M3 byte per 16 elements
    wb = 0.5625 if w.weights == "nvfp4" else 2
    ab = 0.5625 if w.weights == "nvfp4" else 2
    c = {
        "prenorm": (T * D * xb + T * 2 * D * bf + (T * D * ab if w.weights == "nvfp4" else 0), 0),
        "router": (E * D * bf + T * 2 * D * bf + T * E * f4, 2 * T * E * 2 * D),
        "pooler": (L * D * wb + T * D * ab + T * L * f4, 2 * T * L * D),
        "gate_up": (used * 2 * I * L * wb + R * L * ab + R * I * ab, 2 * R * L * 2 * I),
        "down": (used * L * I * wb + R * I * ab + R * L * f4, 2 * R * I * L),
        "unpooler": (D * L * wb + T * L * ab + T * D * f4, 2 * T * D * L),
        "combine": (R * L * f4 + T * L * ab, 0),
        "postnorm": (T * D * (xb + f4 + 4), 0),
    }
    return {kk: (int(b), f) for kk, (b, f) in c.items()}, used


FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense FP4 / BF16 tensor ratio of GB300


def roofline(stage: str, dur_ms: float, costs: dict, pk: dict, pk_kind: str, sustained: bool,
             fp4: bool = False):
    nbytes, flops = costs[stage]
    hbm = pk["hbm_gbs"]
    tf = pk["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    fp4 = fp4 and stage not in ("router",)
    if fp4:
        tf = round(tf * FP4_OVER_BF16, 1)
    t_hbm = nbytes / (hbm * 1e9)
    t_tc = flops / (tf * 1e12) if flops else 0.0
    if t_tc > t_hbm:
        ach = flops / (dur_ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": stage, "achieved": round(ach, 2), "peak": tf, "unit": "TFLOP/s",
                "frac": round(ach / tf, 4),
                "peak_source": f"{pk_kind} bf16_tflops{'_sustained' if sustained else ''}"
                               + (" x 6 (nominal fp4/bf16 ratio)" if fp4 else ""),
                "algorithmic_flop": flops, "traffic": None}
    ach = nbytes / (dur_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": stage, "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(ach / hbm, 4), "peak_source": f"{pk_kind} hbm_gbs",
            "algorithmic_bytes": nbytes, "traffic": None}


def measured_traffic(stage: str, w: workloads.Workload, units: int):
    """DRAM bytes (read + write) per launch of the dominant kernel, scaled from the ncu capture
    recorded in profiles/traffic.json by the units this launch processes; None when no capture
    covers this kernel in this regime or the kernel source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    regime = "decode" if w.T <= 512 else "prefill"
    table = json.load(open(path))
    # a capture of this very workload (full size, one pass of the DRAM counters) first, else
    # one of the same regime scaled by the units
    rec = table.get(f"{stage}/{w.name}") or table.get(f"{stage}/{w.weights}/{regime}")
    if rec is None:
        return None
    src = os.path.join(ROOT, rec["kernel_source"])
    if hashlib.md5(open(src, "rb").read()).hexdigest() != rec["kernel_source_md5"]:
        return None
    return int(rec["traffic_per_unit"] * units)


# ------------------------------------------------------------------ oracle timing
def oracle_sample_inputs(w: workloads.Workload, tokens, inp=None) -> workloads.BlockInputs:
    """Host-resident inputs for the sampled tokens: their x rows, the dense weights, and
    only the experts these tokens route to (expert stacks as dicts keyed by expert id).
    Values come from the seeded generator: copied from ``inp`` (device) when given, else
    regenerated on the host."""
    import oracle
    cpu = lambda t: tuple(u.cpu() for u in t) if isinstance(t, tuple) else t.cpu()  # noqa: E731
    if inp is not None:
        g = {n: getattr(inp, n).cpu() for n in ("g_pre", "g_pool", "g_expert", "g_post")}
        dense = {n: cpu(getattr(inp, n)) for n in ("W_router", "W_pool", "W_unpool")}
        bias = None if inp.router_bias is None else inp.router_bias.cpu()
    else:
        g = workloads.gammas(w)
        nv = w.weights == "nvfp4"
        dense = {"W_router": workloads.dense_weight(w, "W_router")}
        for n in ("W_pool", "W_unpool"):
            dense[n] = workloads.nvfp4_weight(w, n) if nv else workloads.dense_weight(w, n)
        bias = workloads.zipf_bias(w) if w.routing == "zipf" else None
    x = workloads.x_tensor(w, rows=tokens)
    if w.routing == "hot4":
        sel = workloads.forced_routing(w)[tokens].numpy()
    else:
        xn = oracle.rms_norm(x.double().numpy(), g["g_pre"].double().numpy(), w.eps)
        lg = xn @ dense["W_router"].double().numpy().T
        if bias is not None:
            lg = lg + bias.double().numpy()
        sel = oracle.top_k(lg, w.k)
    experts = sorted({int(e) for e in sel.reshape(-1)})
    stacks = {}
    for n in ("W_gate", "W_up", "W_down"):
        if inp is not None:
            src = getattr(inp, n)
            if isinstance(src, tuple):
                stacks[n] = ({e: src[0][e].cpu() for e in experts}, {e: src[1][e].cpu() for e in experts},
                             src[2].cpu())
            else:
                stacks[n] = {e: src[e].cpu() for e in experts}
        elif w.weights == "nvfp4":
            parts = {e: workloads.nvfp4_weight(w, n, expert=e) for e in experts}
            s = torch.full((w.E,), float(next(iter(parts.values()))[2][0]), dtype=torch.float32)
            stacks[n] = ({e: p[0] for e, p in parts.items()}, {e: p[1] for e, p in parts.items()}, s)
        else:
            stacks[n] = {e: workloads.dense_weight(w, n, expert=e) for e in experts}
    forced = workloads.forced_routing(w)[tokens] if w.routing == "hot4" else None
    return workloads.BlockInputs(w=w, x=x, **dense, **stacks, **g, router_bias=bias, forced_idx=forced)


def oracle_resident(w: workloads.Workload, n_tokens: int, inp=None):
    """(params, x, forced) for the first n_tokens of w with every routed expert already
    widened to fp64: the oracle's inputs resident in its own format, as the GPU arm's
    weights are resident in HBM before its timed region."""
    import oracle
    tokens = list(range(n_tokens))
    sample = oracle_sample_inputs(w, tokens, inp=inp)
    P = oracle.params_from_inputs(sample)
    for n in ("W_gate", "W_up", "W_down"):
        keys = getattr(sample, n)[0].keys() if isinstance(getattr(sample, n), tuple) else getattr(sample, n).keys()
        mats = {e: np.array(getattr(P, n)[e]) for e in keys}
        setattr(P, n, oracle.ExpertStack(lambda e, m=mats: m[int(e)], w.E))
    x = sample.x.double().numpy()
    forced = None if sample.forced_idx is None else sample.forced_idx.numpy()
    return P, x, forced


def time_oracle(w: workloads.Workload, n_tokens: int, inp=None, min_seconds: float = 0.0,
                repeats: int = 1, keep: bool = False):
    """Per-call seconds of the fp64 oracle on the first n_tokens of w; repeats the call
    at least ``repeats`` times and until ``min_seconds`` of oracle time have passed.  With keep,
    also (P, x, forced, out, trace) of the last call."""
    import oracle
    P, x, forced = oracle_resident(w, n_tokens, inp=inp)
    times = []
    ref = tr = None
    while len(times) < repeats or sum(times) < min_seconds:
        tr = oracle.Trace() if keep else None
        t0 = time.perf_counter()
        ref = oracle.forward_batched(x, P, w.k, forced_idx=forced, trace=tr)
        times.append(time.perf_counter() - t0)
    return (times, (P, x, forced, ref, tr)) if keep else times


def pick_workload(args) -> workloads.Workload:
    name = "decode_bf16" if args.workload == "all" else args.workload
    return workload_of(name, args.tokens or None, args.experts)


def replica_x(w: workloads.Workload, rank: int, device="cpu"):
    """Tokens of replica `rank`: rows [rank*T, (rank+1)*T) of one long seeded batch (the block is
    token-independent, so replicas exchange nothing)."""
    return workloads.x_tensor(w, device, first_token=rank * w.T)


# ------------------------------------------------------------------ our arm
# Default run: the decode BF16 step (T = 128) is the headline line; the other workloads of the
# block (BF16 prefill with Zipf routing, NVFP4 prefill, NVFP4 hot-expert decode at T = 1..512)
# follow as records under "workloads", each measured the same way.  Workloads of one weight
# dtype share one set of device-resident weights.
ALL_PLAN = [("decode_bf16", None), ("prefill_bf16_zipf", None), ("prefill_nvfp4", None)] + \
    [("decode_nvfp4_hot", t) for t in workloads.DECODE_SWEEP_T]


def plan_of(args):
    if args.workload == "all":
        return ALL_PLAN
    return [(args.workload, args.tokens or None)]


def workload_of(name: str, T, experts: int = 0) -> workloads.Workload:
    import dataclasses
    w = workloads.WORKLOADS[name]
    if T:
        w = w.with_tokens(T)
    if experts:
        w = dataclasses.replace(w, E=experts, name=f"{w.name}@E{experts}")
    return w


def inputs_sharing_weights(w: workloads.Workload, base: workloads.BlockInputs, dev, first_token: int):
    """Inputs of workload w (its x, router bias, forced routing) with the weights of ``base``
    (same seed and shapes, so the same values)."""
    import dataclasses
    return dataclasses.replace(
        base, w=w, x=workloads.x_tensor(w, dev, first_token=first_token),
        router_bias=workloads.zipf_bias(w, dev) if w.routing == "zipf" else None,
        forced_idx=workloads.forced_routing(w, dev) if w.routing == "hot4" else None)


def topk_margins(blk, cfg, w, bias=None):
    """GPU-side routing statistics from the workspace of the last call (host post-processing
    of the kernels' own logits and ids): tokens whose k-th and (k+1)-th logits differ by < 1e-3
    (near ties: another selection would be as legitimate), and tokens with two selected experts
    whose logits differ by < 1e-3 (their order may legitimately swap)."""
    import latent_mixture_experts_router_gb300 as lm
    lay = lm.lmoe_get_workspace_layout(cfg)
    ld = (w.E + 31) // 32 * 32
    lg = blk._ws[lay["logits"]:lay["logits"] + 4 * w.T * ld].view(torch.float32).view(w.T, ld)[:, :w.E]
    if bias is not None:   # the top-k kernel adds the bias (fp32) to the stored logits
        lg = lg + bias.view(1, -1)
    lg = lg.double().cpu().numpy()
    srt = -np.sort(-lg, axis=1)
    near = int(np.sum(srt[:, w.k - 1] - srt[:, w.k] < 1e-3)) if w.k < w.E else 0
    gap = srt[:, :w.k - 1] - srt[:, 1:w.k]
    band = int(np.sum(np.any(gap < 1e-3, axis=1))) if w.k > 1 else 0
    rec = {"near_tie_tokens": near, "in_band_order_tokens": band, "tokens": w.T,
           "source": "GPU fp32 logits of the timed workload; the oracle-graded counts (exact, near "
                     "ties, order swaps, bad) are printed by tests/test_gpu_fullsize.py"}
    if w.routing == "hot4":
        rec["note"] = "routing forced (4 hot experts); the margins describe the router's own logits"
    return rec


def block_bytes(w, used: int) -> float:
    """Algorithmic bytes of one step: the weights of the `used` experts and the dense weights
    (NVFP4: 0.5 + 1/16 bytes per weight), the router, x read and out (fp32) written."""
    T, D, L, E, I = w.T, w.D, w.L, w.E, w.I
    wb = 0.5625 if w.weights == "nvfp4" else 2
    xb = 4 if w.act == "f32" else 2
    return used * 3 * L * I * wb + 2 * D * L * wb + E * D * 2 + T * D * xb + T * D * 4


def block_roofline(w, costs, used, ms_step, pk, pk_kind, sustained, clk=None):
    """The whole step against the block's own bound (SURVEY-style algorithmic bytes: unique
    weights touched + x read + out written; FLOPs of every contraction).  A tensor-bound step
    also reports its fraction of the burst peak and of the burst peak scaled to the median SM
    clock of the timed region (the peak was measured at the maximum clock)."""
    nbytes = block_bytes(w, used)
    flops = sum(f for _, f in costs.values())
    hbm = pk["hbm_gbs"]
    tf = pk["bf16_tflops_sustained" if sustained else "bf16_tflops"] * (FP4_OVER_BF16 if w.weights == "nvfp4" else 1)
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tf * 1e12)
    t = ms_step * 1e-3
    if t_tc > t_hbm:
        rec = {"bound": "tensor", "frac": round(t_tc / t, 4), "achieved_tflops": round(flops / t / 1e12, 1),
               "peak_tflops": round(tf, 1), "algorithmic_flop": int(flops),
               "peak_source": f"{pk_kind} bf16_tflops{'_sustained' if sustained else ''}"
                              + (" x 6" if w.weights == "nvfp4" else "")}
        burst = pk["bf16_tflops"] * (FP4_OVER_BF16 if w.weights == "nvfp4" else 1)
        rec["frac_of_burst"] = round(flops / t / 1e12 / burst, 4)
        mhz, mx = (clk or {}).get("sm_mhz"), (clk or {}).get("sm_max_mhz") or pk.get("sm_max_mhz")
        if mhz and mx:
            rec["frac_of_burst_at_median_clock"] = round(flops / t / 1e12 / (burst * mhz / mx), 4)
            rec["median_sm_mhz"] = mhz
        return rec
    return {"bound": "hbm", "frac": round(t_hbm / t, 4), "achieved_gbs": round(nbytes / t / 1e9, 1),
            "peak_gbs": hbm, "algorithmic_bytes": int(nbytes), "peak_source": f"{pk_kind} hbm_gbs"}


def workload_config(w: workloads.Workload, counts: np.ndarray, ws: int) -> dict:
    """The `config` object of a line: the workload and what one step streams (both arms)."""
    costs, used = stage_costs(w, counts)
    return {"workload": w.name, "T_per_gpu": w.T, "d_model": w.D, "d_latent": w.L, "n_experts": w.E,
            "d_ff": w.I, "top_k": w.k, "routing": w.routing, "weights": w.weights,
            "experts_touched": used, "parallelism": f"replicas x{ws} (token-independent, no exchange)",
            "l2": "inputs larger than L2: each step streams "
                  f"{sum(b for b, _ in costs.values()) / 1e9:.2f} GB (129 MB L2)"}


def measure(args, ws, rank, local, w, blk, inp, cpu_tokens: int, cpu_seconds: float):
    """One workload: stage pass, timed pass, dominant-kernel pass, end-to-end pass; the record
    (rank 0) or None."""
    import latent_mixture_experts_router_gb300 as lm
    dev = torch.device(f"cuda:{local}")
    T = w.T
    cfg = blk.config(T, w.act, "f32")
    blk.workspace(cfg)
    out = torch.empty(T, w.D, dtype=torch.float32, device=dev)
    ex = {}
    if inp.router_bias is not None:
        ex["router_bias"] = inp.router_bias
    if inp.forced_idx is not None:
        ex["forced_idx"] = inp.forced_idx
    if getattr(args, "single_token_path", 0):
        ex["single_token_path"] = args.single_token_path
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        if evs is not None:
            blk.forward(inp.x, out=out, stage_events=evs, **ex)
        else:
            blk.forward(inp.x, out=out, **ex)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, word = lm.lmoe_check_status(cfg, blk._ws)
    assert st == 0, f"device status {st} ({word:#x})"
    lay = lm.lmoe_get_workspace_layout(cfg)
    counts = blk._ws[lay["counts"]:lay["counts"] + 4 * w.E].view(torch.int32).cpu().numpy()
    margins = topk_margins(blk, cfg, w, inp.router_bias)

    # ---- stage breakdown (untimed pass): an event at every stage boundary, which serialises
    #      the launches; it gives the stage table and picks the dominant kernel
    n_bd = max(3, min(args.steps, 20))
    bd = [[torch.cuda.Event(enable_timing=True) for _ in range(lm.NUM_STAGE_EVENTS)] for _ in range(n_bd)]
    for i in range(n_bd):
        step(bd[i])
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in bd)
                for i, name in enumerate(lm.STAGES)}
    costs, used = stage_costs(w, counts)
    # the expert pair (lmoe_expert_pair): gate/up and down in one kernel, which the gate_up stage
    # spans (the down stage is empty); its bytes are both GEMMs'
    pair = lm.lmoe_expert_pair(cfg)
    if pair:
        costs["expert_pair"] = tuple(a + b for a, b in zip(costs["gate_up"], costs["down"]))
        stage_ms["expert_pair"] = stage_ms["gate_up"] + stage_ms["down"]
        del costs["gate_up"], costs["down"]
    dom = max((s for s in costs if s in stage_ms), key=lambda s: stage_ms[s])
    di = lm.STAGES.index("gate_up" if dom == "expert_pair" else dom)

    # ---- timed region (device): K whole steps, nothing recorded between the kernels
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    n0 = lm.lmoe_kernel_launches()
    barrier(ws)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    launches = lm.lmoe_kernel_launches() - n0
    ms = t_start.elapsed_time(t_end)
    ms_max = allreduce_max(ms, ws)

    # ---- the dominant kernel, timed live in a second pass of K steps right after: events on
    #      the launching stream around that kernel only.  An event between two kernels turns off
    #      their launch overlap, which is why the headline pass above records none.  A step that
    #      ran as one kernel (one token with NVFP4 weights: the single-token kernel, which stage
    #      events turn back into the kernel chain) is timed by events around each call.
    single = (T == 1 and w.weights == "nvfp4" and getattr(args, "single_token_path", 0) == 1
              and launches == 2 * args.steps)
    rcosts = dict(costs)
    if single:
        dom = "single_token_kernel"
        rcosts[dom] = (block_bytes(w, used), sum(f for _, f in costs.values()))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    else:
        evs = [[torch.cuda.Event(enable_timing=True) if j in (di, di + 1) else None
                for j in range(lm.NUM_STAGE_EVENTS)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    k_start = torch.cuda.Event(enable_timing=True)
    k_end = torch.cuda.Event(enable_timing=True)
    k_start.record(stream)
    for i in range(args.steps):
        if single:
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        else:
            step(evs[i])
    k_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    if single:
        dom_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    else:
        dom_ms = statistics.mean(e[di].elapsed_time(e[di + 1]) for e in evs)
    ms_kpass = k_start.elapsed_time(k_end) / args.steps

    # ---- end to end through the host-I/O entry point: pinned x in, pinned out back
    x_host = inp.x.cpu().pin_memory()
    out_host = torch.empty(T, w.D, dtype=torch.float32).pin_memory()
    ws_io = torch.zeros(lm.lmoe_workspace_size_host_io(cfg), dtype=torch.uint8, device=dev)
    W = blk.W

    def step_io():
        lm.latent_moe_forward_host_io_ex(cfg, x_host, W["W_router"], W["W_pool"], W["g_pool"], W["W_gate"],
                                         W["W_up"], W["W_down"], W["g_expert"], W["W_unpool"], W["g_pre"],
                                         W["g_post"], w.k, out_host, ws_io, **ex)

    # router bias and forced routing stay device-resident routing controls; x and out go
    # through pinned host memory every step
    for _ in range(max(2, args.warmup // 2)):
        step_io()
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step_io()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms_io = allreduce_max(e0.elapsed_time(e1), ws)
    # the parity sample: one more step on the timed path, the output and top-k of its first
    # tokens kept for the oracle (rank 0, with the CPU baseline)
    par = None
    if rank == 0 and not args.no_cpu_baseline:
        step()
        torch.cuda.synchronize()
        n_par = max(1, min(cpu_tokens, T))
        lay_p = lm.lmoe_get_workspace_layout(cfg)
        par = (out[:n_par].double().cpu().numpy(),
               blk._ws[lay_p["topk_idx"]:lay_p["topk_idx"] + 4 * n_par * w.k].view(torch.int32)
               .view(n_par, w.k).cpu().numpy())
    e2e = {"value": round(ws * T * args.steps / (ms_io * 1e-3), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()),
           "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size()),
           "ms_per_step": round(ms_io / args.steps, 4), "path": "latent_moe_forward_host_io_ex"}
    del ws_io, x_host, out_host, out

    if rank != 0:
        return None
    pk, pk_kind = peaks()
    total_flops = sum(f for _, f in costs.values())
    ms_step = ms_max / args.steps
    capped = bool(clk and "sw_power_cap" in clk.get("reasons", []))
    rec = {
        "value": round(ws * T * args.steps / (ms_max * 1e-3), 1), "unit": "tokens/s",
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "dtype": "nvfp4" if w.weights == "nvfp4" else "bf16",
        "config": workload_config(w, counts, ws),
        "tflops": round(total_flops / (ms_step * 1e-3) / 1e12, 2),
        "block_roofline": block_roofline(w, costs, used, ms_step, pk, pk_kind, capped, clk),
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stage_ms_note": f"separate pass of {n_bd} steps, an event at every stage boundary"
                         + ("; gate/up and down ran as one kernel (the expert pair), which the gate_up stage "
                            "spans (down empty); expert_pair = their sum" if pair else "")
                         + (" (the stage kernels: events at the stage boundaries select the kernel chain; "
                            "the timed steps ran the single-token path "
                            f"{getattr(args, 'single_token_path', 0)} of lmoe_ex.single_token_path)"
                            if T == 1 and w.weights == "nvfp4" and getattr(args, "single_token_path", 0) != 2 else ""),
        # a kernel that ran under the power cap is held against the sustained tensor peak (the
        # measured one of a seconds-long GEMM loop under the same cap), else the burst peak
        "roofline": {**roofline(dom, dom_ms, rcosts, pk, pk_kind, sustained=capped, fp4=w.weights == "nvfp4"),
                     "traffic": measured_traffic(dom, w, used),
                     "timing": (f"CUDA events on the launching stream around each call (the single-token "
                                f"kernel and the kernel that clears its status words), {args.steps} steps timed "
                                "right after the headline pass" if single else
                                f"CUDA events on the launching stream around the kernel, {args.steps} steps "
                                "timed right after the headline pass (that pass records no events: an "
                                "event between two kernels turns off their launch overlap)"),
                     "step_ms_with_kernel_events": round(ms_kpass, 4)},
        "routing": margins,
        "gpu_launches": int(launches), "clocks": clk, "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        from oracle.compare import TOL_BF16, TOL_NVFP4, compare_block
        n_tok = max(1, min(cpu_tokens, w.T))
        times, (P_o, x_o, forced_o, ref_o, tr_o) = time_oracle(w, n_tok, inp=inp, min_seconds=cpu_seconds, keep=True)
        tol = TOL_NVFP4 if w.weights == "nvfp4" else TOL_BF16
        pr = compare_block(par[0], par[1], x_o, P_o, w.k, tol, tr=tr_o, ref=ref_o, forced_idx=forced_o)
        rec["parity"] = {
            "tokens": pr.tokens, "topk_exact": pr.idx_exact, "near_tie": pr.near_tie_tokens,
            "order_swaps": pr.order_swaps, "quant_boundary": pr.quant_boundary_tokens,
            "bad_topk": len(pr.bad_idx_tokens), "max_abs_err": float(f"{pr.max_abs_err:.4e}"),
            "ref_rms": float(f"{pr.ref_rms:.4e}"),
            "max_abs_err_over_rms": float(f"{pr.max_abs_err / max(pr.ref_rms, 1e-30):.4e}"), "tolerance": tol,
            "ok": bool(pr.ok),
            "source": f"the first {pr.tokens} tokens of the timed workload: the output and top-k of one more "
                      "step on the timed path against the fp64 oracle, under the rules of oracle/compare.py "
                      "(near ties and in-band order swaps re-graded; NVFP4 rounding-boundary alternatives)"}
        t = sum(times)
        rec["cpu_baseline"] = {"value": round(n_tok * len(times) / t, 3), "unit": "tokens/s",
                               "cores": os.cpu_count(), "kind": "oracle",
                               "sample": f"first {n_tok} tokens of {w.name} through the fp64 oracle (numpy "
                                         f"BLAS, routed experts pre-widened to fp64), {len(times)} calls, "
                                         f"{t:.1f} s"}
    return rec


def run_ours(args, ws, rank, local):
    import gc

    import latent_mixture_experts_router_gb300 as lm
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    recs = []
    base = {}   # weight dtype -> (inputs holding the weights, block)
    t0 = time.perf_counter()
    for i, (name, T) in enumerate(plan_of(args)):
        w = workload_of(name, T, args.experts)
        key = w.weights
        if key not in base:
            for k_old in list(base):   # one weight set resident at a time
                del base[k_old]
            gc.collect()
            torch.cuda.empty_cache()
            inp = workloads.make_inputs(w, dev)
            if ws > 1:
                inp.x = workloads.x_tensor(w, dev, first_token=rank * w.T)
            blk = lm.LatentMoEBlock(inp.W_router, inp.W_pool, inp.g_pool, inp.W_gate, inp.W_up, inp.W_down,
                                    inp.g_expert, inp.W_unpool, inp.g_pre, inp.g_post, w.k, w.eps,
                                    weight_dtype=w.weights)
            base[key] = (inp, blk)
        else:
            inp = inputs_sharing_weights(w, base[key][0], dev, rank * w.T)
            blk = base[key][1]
        headline = i == 0
        # the headline's oracle sample takes ~10 s; the other records' a few seconds each
        n_cpu = args.cpu_tokens if args.cpu_tokens else ({"tiny_fp32": 64}.get(w.name.split("@")[0], 8)
                                                         if headline else 2)
        rec = measure(args, ws, rank, local, w, blk, inp, n_cpu, 10.0 if headline else 3.0)
        if rec is not None:
            recs.append(rec)
        del inp
        torch.cuda.empty_cache()
    if rank != 0:
        return None
    head = recs[0]
    line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
            "data": "synthetic (seeded counter-based generator; random-init weights of the Muse layer shapes)"}
    line.update({k: v for k, v in head.items() if k not in line and k not in ("steps", "warmup")})
    line["gpu_launches"] = sum(r["gpu_launches"] for r in recs[:1])
    if len(recs) > 1:
        line["workloads"] = {r["config"]["workload"]: r for r in recs[1:]}
        line["workloads_note"] = ("the block's other workloads, measured after the headline one in the "
                                  "same run and the same way (each record: K device-timed steps, "
                                  "dominant kernel, end-to-end host-I/O figure, clocks, oracle baseline, parity "
                                  "of the first tokens against the oracle)")
    line["bench_wall_s"] = round(time.perf_counter() - t0, 1)
    return line


# ------------------------------------------------------------------ reference arm
def host_routing_counts(w: workloads.Workload) -> np.ndarray:
    """Rows per expert of the workload's routing, from the oracle's router on the host (the
    reference arm's config, which names the same workload as the GPU arm's)."""
    import oracle
    if w.routing == "hot4":
        sel = workloads.forced_routing(w).numpy()
    else:
        g = workloads.gammas(w)
        xn = oracle.rms_norm(workloads.x_tensor(w).double().numpy(), g["g_pre"].double().numpy(), w.eps)
        lg = xn @ workloads.dense_weight(w, "W_router").double().numpy().T
        if w.routing == "zipf":
            lg = lg + workloads.zipf_bias(w).double().numpy()
        sel = oracle.top_k(lg, w.k)
    return np.bincount(np.asarray(sel).reshape(-1), minlength=w.E)


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    w = pick_workload(args)
    n_tok = max(1, args.cpu_tokens)
    times = time_oracle(w, n_tok, repeats=args.warmup + args.steps)[args.warmup:]
    dt = sum(times)
    v = round(n_tok * args.steps / dt, 3)
    sample = (f"each step: the first {n_tok} of the workload's {w.T} tokens ({w.name}) through the fp64 "
              f"oracle (numpy BLAS on the host cores); weights of the routed experts generated on the host "
              f"and widened to fp64 before timing; tokens/s of that sample")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator; random-init weights of the Muse layer shapes)",
            "config": workload_config(w, host_routing_counts(w), ws),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all", choices=["all"] + sorted(workloads.WORKLOADS),
                    help="all (default): the decode BF16 headline plus every other workload as records")
    ap.add_argument("--tokens", type=int, default=0, help="override T of the workload")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (smaller profiling cases; the benchmark line uses the workload's E)")
    ap.add_argument("--cpu-tokens", type=int, default=None,
                    help="oracle sample size in tokens (default: ~10-30 s of CPU work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single-token-path", type=int, default=0, choices=[0, 1, 2],
                    help="NVFP4 at T = 1: 0 pre/post kernels around the expert GEMMs (default), 1 the whole "
                         "block as one kernel, 2 the stage kernels (lmoe_ex.single_token_path)")
    args = ap.parse_args()
    ws, rank, local = dist_init()
    if args.impl == "reference" and args.cpu_tokens is None:   # bounded host memory
        args.cpu_tokens = {"tiny_fp32": 64}.get(args.workload, 4)
    if args.impl == "reference":
        args.steps = 3 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        line = run_reference(args, ws, rank)
    else:
        args.steps = 20 if args.steps is None else args.steps
        args.warmup = 5 if args.warmup is None else args.warmup
        line = run_ours(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
