"""Benchmark of the single-GPU MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T] [--alpha A]
                    [--impl ours|reference] [--no-sweep] [--no-cpu]

One step = one moe_forward_ex over one batch of T tokens (router + top-k,
permute, fused gate+up GEMM, down GEMM, combine), inputs and weights already
resident in HBM.  Prints ONE JSON line.  The default workload is the
Mixtral-8x7B-shaped layer (H=4096, F=14336, E=8, top-2) at T=4096; the
other token counts of that layer (1, 32, 128, 512) are timed in the same run
and reported under "sweep".

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer forward has no exchange step); the time is the max over ranks and
the value the tokens of all ranks divided by it.

--impl reference times the CPU oracle (float64 numpy) on the host cores on
bounded samples of the same workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth.workloads import SKEW_ALPHAS, T_SWEEP  # noqa: E402

METRIC = "MoE layer fwd tokens/s on 1 GB300; % of max(HBM, bf16 tensor) roofline"
NOMINAL_HBM = 8.0e12       # B/s, the layer roofline's denominators
NOMINAL_BF16 = 2.25e15     # FLOP/s
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ("route", "permute", "gate_up_gemm", "down_gemm", "combine")


# ----------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running;
    the summary's clock is the median over the samples taken under load
    (power draw above half the largest seen)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        rows, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm = float(parts[1])
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = float("nan")
            rows.append((sm, pw))
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        pmax = max((p for _, p in rows if p == p), default=float("nan"))
        loaded = [sm for sm, p in rows if pmax == pmax and p == p and p >= 0.5 * pmax] or [sm for sm, _ in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded)}


def make_cfg(moe, wl, d):
    return moe.MoeConfig.make(score=wl.score, renormalize=wl.renormalize, route_scale=wl.route_scale,
                              n_group=wl.n_group, topk_group=wl.topk_group, group_topn=wl.group_topn,
                              logit_bias=d.get("logit_bias"), ws_gate=d.get("ws_gate"), ws_up=d.get("ws_up"),
                              ws_down=d.get("ws_down"), w_shared_gate=d.get("w_shared_gate"),
                              activation=wl.activation)


def stage_algorithmic(wl, active: int):
    """Algorithmic FLOPs and bytes of each stage of one forward: what the
    stage must compute and move at minimum given its inputs and outputs
    (x_perm and h bf16, the expert outputs y fp16)."""
    T, H, F, E, k = wl.T, wl.H, wl.F, wl.E, wl.k
    Tk = T * k
    out = {
        "route": (2.0 * T * H * E, T * H * 2.0 + E * H * 2.0 + Tk * 8.0),
        "permute": (0.0, T * H * 2.0 + Tk * H * 2.0 + Tk * 12.0),
        "gate_up_gemm": (Tk * 4.0 * H * F, active * 4.0 * H * F + Tk * H * 2.0 + Tk * F * 2.0),
        "down_gemm": (Tk * 2.0 * H * F, active * 2.0 * H * F + Tk * F * 2.0 + Tk * H * 2.0),
        "combine": (0.0, Tk * H * 2.0 + T * H * 2.0 + Tk * 8.0),
    }
    if wl.F_shared:
        Fs = wl.F_shared
        f, b = out["gate_up_gemm"]
        out["gate_up_gemm"] = (f + T * 4.0 * H * Fs, b + 4.0 * H * Fs + T * H * 2.0 + T * Fs * 2.0)
        f, b = out["down_gemm"]
        out["down_gemm"] = (f + T * 2.0 * H * Fs, b + 2.0 * H * Fs + T * Fs * 2.0 + T * H * 2.0)
        f, b = out["combine"]
        out["combine"] = (f, b + T * H * 2.0)
    return out


def max_over_ranks(ms: float, world: int) -> float:
    """The job's time: the slowest replica's (all-reduce MAX over the ranks of
    the default process group; the group is gloo, so this runs on the host)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, T: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every replica processes T tokens per step."""
    return world * T * steps / (ms / 1e3)


def workload_overrides(args) -> dict:
    """Per-run changes to the named layer shape: the Zipf exponent, and a
    reduced expert count (--experts) that keeps H, F, k and the routing
    variant (groups of E / n_group experts) for small profiling captures; the
    label names the expert count, so such a line is never the headline."""
    kw = {} if args.alpha is None else {"alpha": args.alpha}
    if args.activation is not None:
        kw["activation"] = args.activation
    if args.experts is not None:
        base = synth.workload(args.workload)
        if args.experts < base.k or args.experts % base.n_group != 0:
            raise SystemExit(f"--experts must be >= k={base.k} and a multiple of n_group={base.n_group}")
        kw["E"] = args.experts
    return kw


def sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_layer_06_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and this workload; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {})
    if e.get("sources_sha") == sources_sha() and e.get("workload") == workload:
        return e.get("dram_bytes_per_launch")
    return None


# ----------------------------------------------------------------------------- our arm

# Every (layer, T, alpha) point of the five layer shapes, timed in the same
# run as the headline, in this order (one layer's weights on the device at a time).
CONFIG_ORDER = ("deepseek", "mixtral", "qwen2", "skew", "tiny")


def config_points():
    pts = []
    for name in CONFIG_ORDER:
        for a in (SKEW_ALPHAS if name == "skew" else (None,)):
            for T in T_SWEEP[name]:
                pts.append((name, T, a))
    return pts


def to_device(torch, inp):
    d = {}
    for name, a in inp.items():
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        d[name] = t.cuda().view(torch.bfloat16) if a.dtype == np.uint16 else t.cuda()
    return d


def load_workload(torch, wl_all):
    """The layer's tensors on the device (one tensor generated on the host at
    a time and dropped once copied)."""
    d = to_device(torch, synth.make_inputs(wl_all, with_experts=False, with_shared=True))
    for name in ("w_gate", "w_up", "w_down"):
        shape = (wl_all.E, wl_all.F, wl_all.H) if name != "w_down" else (wl_all.E, wl_all.H, wl_all.F)
        stream = {"w_gate": synth.STREAM_WG, "w_up": synth.STREAM_WU, "w_down": synth.STREAM_WD}[name]
        d.update(to_device(torch, {name: synth.normal_bf16(wl_all.seed, stream, shape, std=0.02)}))
    return d


def time_point(moe, torch, d, cfg, wl, K, W, stream, world=1, timed_stages=True, mark_stage=None):
    """K forwards of wl.T tokens back to back (after W warm-up forwards) on
    `stream`, timed with CUDA events around the K forwards.  Inside that timed
    region the library records events only around stage `mark_stage` (when
    given), whose duration per forward is then measured over the timed region
    itself; any other event between kernels would break the launch overlap
    between them.  The full per-stage split comes from a separate pass of K
    forwards with events between all stages."""
    import torch.distributed as dist
    T = wl.T
    x = d["x"][:T]
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(moe.moe_workspace_bytes(cfg, T, wl.H, wl.F, wl.E, wl.k), dtype=torch.uint8, device="cuda")

    def fwd():
        moe.moe_forward_ex(x, d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg, out=out,
                           workspace=ws)

    for _ in range(W):
        fwd()
    st, raw = moe.moe_device_error()
    if st != 0:
        raise RuntimeError(f"device error {moe.moe_status_string(st)} {raw:#x}")
    # active experts of this batch (for the compulsory-byte roofline)
    idx, _, _ = moe.moe_route(x, d["w_router"], wl.k, cfg)
    active = int(torch.unique(idx).numel())
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = None
    if mark_stage is not None:
        marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a_, b_ in marks:  # create the CUDA events before the timed region
            a_.record(stream)
            b_.record(stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        if marks is not None:
            row = [None] * 6
            row[mark_stage], row[mark_stage + 1] = marks[i]
            moe.moe_set_trace_events(row)
        fwd()
    stop.record(stream)
    torch.cuda.synchronize()
    if marks is not None:
        moe.moe_set_trace_events(None)
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(stop)
    res = {"T": T, "ms_total": ms, "active_experts": active, "wl": wl}
    if marks is not None:
        res["marked_stage_ms"] = float(np.mean([a_.elapsed_time(b_) for a_, b_ in marks]))
    if timed_stages:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
        for row in ev:  # create the CUDA events before the traced pass
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        for i in range(K):
            moe.moe_set_trace_events(ev[i])
            fwd()
        torch.cuda.synchronize()
        moe.moe_set_trace_events(None)
        per = np.array([[ev[i][j].elapsed_time(ev[i][j + 1]) for j in range(5)] for i in range(K)])
        res["stage_ms"] = dict(zip(STAGES, per.mean(axis=0).tolist()))
    st, raw = moe.moe_device_error()
    if st != 0:
        raise RuntimeError(f"device error {moe.moe_status_string(st)} {raw:#x}")
    del out, ws
    return res


def point_summary(r, K):
    w = r["wl"]
    ms = r["ms_total"] / K
    tr = max(w.flops() / NOMINAL_BF16, w.compulsory_bytes(r["active_experts"]) / NOMINAL_HBM)
    out = {"workload": w.label, "T": w.T, "tokens_per_s": w.T / (ms / 1e3), "us_per_step": ms * 1e3,
           "layer_roofline_us": tr * 1e6, "layer_roofline_frac": tr / (ms / 1e3),
           "active_experts": r["active_experts"], "steps": K}
    if w.alpha is not None:
        out["alpha"] = w.alpha
    if "stage_ms" in r:
        out["stages_us"] = {k2: v * 1e3 for k2, v in r["stage_ms"].items()}
    return out


def skew_slowdown(configs):
    """Per T of the skew layer: time per forward at alpha = 2 over alpha = 0."""
    by = {(c["T"], c.get("alpha")): c["us_per_step"] for c in configs if c["workload"].startswith("skew")}
    res = {}
    for (T, a), us in sorted(by.items()):
        if a == 2.0 and (T, 0.0) in by:
            res[str(T)] = us / by[(T, 0.0)]
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist

    import mixture_experts_layer_06_gb300 as moe

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo", init_method="env://")
    torch.cuda.set_device(local)
    moe.load_library()
    stream = torch.cuda.current_stream()

    kw = workload_overrides(args)
    T_main = args.T if args.T is not None else max(T_SWEEP[args.workload])
    T_all = max([T_main] + list(T_SWEEP[args.workload]))
    wl_all = synth.workload(args.workload, T=T_all, **kw)
    d = load_workload(torch, wl_all)
    cfg = make_cfg(moe, wl_all, d)

    pk, pk_kind = peaks()
    # the stage split of the headline batch (a traced pass), then its timed
    # region with events around the dominant stage only
    split = time_point(moe, torch, d, cfg, wl_all.with_T(T_main), args.steps, args.warmup, stream, world)
    dom_i = max(range(len(STAGES)), key=lambda j: split["stage_ms"][STAGES[j]])
    # clocks over the headline batch's timed forwards and its end-to-end leg
    clocks = ClockSampler(local).__enter__()
    try:
        main = time_point(moe, torch, d, cfg, wl_all.with_T(T_main), args.steps, 3, stream, world,
                          timed_stages=False, mark_stage=dom_i)
        main["stage_ms"] = split["stage_ms"]
    except BaseException:
        clocks.__exit__(None, None, None)
        raise

    ms_main = max_over_ranks(main["ms_total"], world)
    wl = main["wl"]
    ms_step = ms_main / args.steps
    value = job_tokens_per_s(world, T_main, args.steps, ms_main)

    # layer roofline (nominal denominators) for this batch
    flops = wl.flops()
    cbytes = wl.compulsory_bytes(main["active_experts"])
    t_roof = max(flops / NOMINAL_BF16, cbytes / NOMINAL_HBM)

    # end to end through the public API with host buffers
    try:
        e2e = run_e2e(moe, torch, d, cfg, wl, args, stream)
    finally:
        clocks.__exit__(None, None, None)
    clk = clocks.summary()

    # dominant kernel roofline (measured peaks)
    stage_ms = main["stage_ms"]
    alg = stage_algorithmic(wl, main["active_experts"])
    dom = STAGES[dom_i]
    f_dom, b_dom = alg[dom]
    sec = main["marked_stage_ms"] / 1e3  # measured over the timed region
    intensity = f_dom / b_dom
    # The bf16 peak that matches the clocks seen in the timed region: the
    # burst figure while the GPU ran at full clock, the sustained one once the
    # power cap had pulled the clock down.
    capped = "sw_power_cap" in clk.get("reasons", [])
    bf16 = pk["bf16_tflops_sustained"] if capped else pk["bf16_tflops"]
    ridge = bf16 * 1e12 / (pk["hbm_gbs"] * 1e9)
    if intensity >= ridge:
        roof = {"bound": "tensor", "achieved": f_dom / sec / 1e12, "peak": bf16, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": b_dom / sec / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    kind = ("sustained" if capped else "burst") + " bf16 matmul"
    roof["peak_source"] = f"{pk_kind} ({kind if roof['bound'] == 'tensor' else 'copy'})"
    roof["kernel"] = dom
    roof["duration_us"] = main["marked_stage_ms"] * 1e3
    roof["timing"] = "CUDA events around this stage in every timed forward (the only events inside the timed region)"
    roof["traffic"] = recorded_traffic(dom, wl.label)
    roof["algorithmic"] = {"flops_per_launch": f_dom, "bytes_per_launch": b_dom,
                           "intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge}
    gpu_launches = moe.moe_forward_launches(cfg, wl.T, wl.H, wl.F, wl.E, wl.k) * args.steps

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(wl, budget_s=args.cpu_seconds)

    # every point of the five layer shapes, in the same run
    configs, decode = [], []
    headline_key = (args.workload, T_main, wl.alpha)
    if not args.no_sweep and not kw.get("E") and not kw.get("activation"):
        loaded = (args.workload, wl.alpha)
        for name, T, a in config_points():
            if (name, T, a) == headline_key:
                configs.append(dict(point_summary(main, args.steps), headline=True))
                continue
            if (name, a) != loaded:
                del d
                torch.cuda.empty_cache()
                wl_all = synth.workload(name, T=max(T_SWEEP[name]), **({} if a is None else {"alpha": a}))
                d = load_workload(torch, wl_all)
                cfg = make_cfg(moe, wl_all, d)
                loaded = (name, a)
            K = max(args.steps, 50) if T <= 32 else max(args.steps, 20) if T <= 512 else args.steps
            r = time_point(moe, torch, d, cfg, wl_all.with_T(T), K, args.warmup, stream, world)
            configs.append(point_summary(r, K))
            if name == "mixtral" and T == max(T_SWEEP[name]) and not args.no_decode:
                decode = run_decode(moe, torch, d, cfg, wl_all, stream)

    esweep = run_expert_sweep(moe, torch, args, stream) if args.expert_sweep else None
    sched = ablation = None
    if args.schedule_ablation or args.fusion_ablation:
        if (wl_all.name, wl_all.alpha) != (args.workload, wl.alpha):
            del d
            torch.cuda.empty_cache()
            wl_all = synth.workload(args.workload, T=T_all, **kw)
            d = load_workload(torch, wl_all)
            cfg = make_cfg(moe, wl_all, d)
        Ts = sorted(set([T_main] + list(T_SWEEP[args.workload])))
        if args.schedule_ablation:
            sched = run_schedule_ablation(moe, torch, d, cfg, wl_all, Ts, stream, args.steps)
        if args.fusion_ablation:
            ablation = run_fusion_ablation(moe, torch, d, cfg, wl_all, Ts, stream, args.steps)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) x, N(0,0.02) weights, bf16)",
        "config": {"workload": wl.label, "T": wl.T, "H": wl.H, "F": wl.F, "E": wl.E, "k": wl.k,
                   "routing": f"{wl.score}, renormalize={wl.renormalize}, scale={wl.route_scale}",
                   "parallelism": f"replicas x{world}",
                   "l2": f"no flush: the {cbytes / 1e9:.2f} GB of compulsory weight traffic per step exceeds "
                         f"the 126 MB L2"},
        "layer_roofline": {"t_roofline_us": t_roof * 1e6, "frac": t_roof / (ms_step / 1e3),
                           "flops": flops, "compulsory_bytes": cbytes, "active_experts": main["active_experts"],
                           "denominators": "nominal 8 TB/s HBM, 2.25 PFLOP/s dense bf16"},
        "roofline": roof,
        "stages_ms": stage_ms,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": gpu_launches,
        "configs": configs,
        "skew_alpha2_over_alpha0_time": skew_slowdown(configs),
        "decode": decode,
    }
    if esweep is not None:
        line["expert_sweep"] = esweep
    if ablation is not None:
        line["fusion_ablation"] = ablation
    if sched is not None:
        line["schedule_ablation"] = sched
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_fusion_ablation(moe, torch, d, cfg, wl_all, Ts, stream, steps):
    """The fused gate+up GEMM against the unfused form (two GEMMs with bf16
    g, u in HBM, then the element-wise activation), on the routed experts of
    the batch: route and permute once, then time each FFN over `steps`
    back-to-back calls.  intermediate_bytes counts the HBM traffic of the
    per-row intermediates (bf16): fused writes and reads h (4 rows F); unfused
    also writes and reads g and u (12 rows F)."""
    res = []
    for T in Ts:
        wl = wl_all.with_T(T)
        x = d["x"][:T]
        idx, _, _ = moe.moe_route(x, d["w_router"], wl.k, cfg)
        _, offsets, _, _, x_perm = moe.moe_permute(idx, x, wl.E)
        rows = T * wl.k
        args = (x_perm, offsets, d["w_gate"], d["w_up"], d["w_down"])
        out = {}
        for name, fn in (("fused", lambda: moe.moe_expert_ffn(*args, activation=wl.activation)),
                         ("unfused", lambda: moe.moe_expert_ffn_unfused(*args, activation=wl.activation))):
            for _ in range(3):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            out[name] = a.elapsed_time(b) * 1e3 / steps
        st, raw = moe.moe_device_error()
        if st != 0:
            raise RuntimeError(f"device error {moe.moe_status_string(st)} {raw:#x}")
        res.append({"T": T, "rows": rows, "fused_us": out["fused"], "unfused_us": out["unfused"],
                    "unfused_over_fused": out["unfused"] / out["fused"],
                    "intermediate_bytes": {"fused": 4 * rows * wl.F, "unfused": 12 * rows * wl.F},
                    "scope": "routed experts: gate+up and down GEMMs (+ element-wise pass when unfused)"})
    return res


def run_schedule_ablation(moe, torch, d, cfg, wl_all, Ts, stream, steps, block_m=64):
    """The persistent, device-scheduled grouped FFN against the pages'
    schedule (expert counts read back to the host with a synchronisation,
    fixed block_m token tiles, one CTA per tile), on the routed experts of the
    batch; each timed over `steps` back-to-back calls."""
    res = []
    for T in Ts:
        wl = wl_all.with_T(T)
        x = d["x"][:T]
        idx, _, _ = moe.moe_route(x, d["w_router"], wl.k, cfg)
        counts, offsets, _, _, x_perm = moe.moe_permute(idx, x, wl.E)
        args = (x_perm, offsets, d["w_gate"], d["w_up"], d["w_down"])
        out = {}
        for name, fn in (("persistent", lambda: moe.moe_expert_ffn(*args)),
                         ("static", lambda: moe.moe_expert_ffn_static(*args, block_m=block_m))):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()  # wall clock: the static schedule synchronises with the host
            for _ in range(steps):
                fn()
            torch.cuda.synchronize()
            out[name] = (time.perf_counter() - t0) * 1e6 / steps
        st, raw = moe.moe_device_error()
        if st != 0:
            raise RuntimeError(f"device error {moe.moe_status_string(st)} {raw:#x}")
        c = counts.cpu()
        res.append({"T": T, "persistent_us": out["persistent"], "static_us": out["static"],
                    "static_over_persistent": out["static"] / out["persistent"], "block_m": block_m,
                    "active_experts": int((c > 0).sum()), "max_rows_per_expert": int(c.max()),
                    "timing": "host wall clock per call, back-to-back, both arms"})
    return res


DECODE_T = (1, 2, 4, 8, 16, 32)
ESWEEP_T = (128, 512)


def run_expert_sweep(moe, torch, args, stream):
    """The expert-count sweep: E experts of width F = 8 * 14336 / E (constant
    expert parameters), H = 4096, top-2, at the token counts of ESWEEP_T;
    device time per forward over args.steps back-to-back forwards."""
    from synth.workloads import EXPERT_SWEEP_E, expert_sweep
    res = []
    for E in EXPERT_SWEEP_E:
        wl_all = expert_sweep(E, max(ESWEEP_T))
        d = load_workload(torch, wl_all)
        cfg = make_cfg(moe, wl_all, d)
        for T in ESWEEP_T:
            wl = wl_all.with_T(T)
            x = d["x"][:T]
            out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
            ws = torch.empty(moe.moe_workspace_bytes(cfg, T, wl.H, wl.F, wl.E, wl.k), dtype=torch.uint8,
                             device="cuda")

            def fwd():
                moe.moe_forward_ex(x, d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg, out=out,
                                   workspace=ws)

            for _ in range(args.warmup):
                fwd()
            idx, _, _ = moe.moe_route(x, d["w_router"], wl.k, cfg)
            active = int(torch.unique(idx).numel())
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(args.steps):
                fwd()
            b.record(stream)
            torch.cuda.synchronize()
            st, raw = moe.moe_device_error()
            if st != 0:
                raise RuntimeError(f"device error {moe.moe_status_string(st)} {raw:#x}")
            us = a.elapsed_time(b) * 1e3 / args.steps
            tr = max(wl.flops() / NOMINAL_BF16, wl.compulsory_bytes(active) / NOMINAL_HBM)
            res.append({"workload": wl.label, "E": E, "F": wl.F, "T": T, "us_per_step": us,
                        "tokens_per_s": T / (us / 1e6), "layer_roofline_frac": tr / (us / 1e6),
                        "active_experts": active})
        del d
        torch.cuda.empty_cache()
    return res


def run_decode(moe, torch, d, cfg, wl_all, stream, reps=200):
    """Decode-sized batches: the forward launched eagerly on one stream and
    the same forward captured once in a CUDA graph and replayed.  Reports
    device time per forward for both (CUDA events around `reps` back-to-back
    forwards), the host time to issue one eager forward, and checks that the
    replay writes the same bits as the eager call."""
    res = []
    for T in (t for t in DECODE_T if t <= d["x"].shape[0]):
        wl = wl_all.with_T(T)
        x = d["x"][:T]
        out = torch.empty((T, wl.H), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(moe.moe_workspace_bytes(cfg, T, wl.H, wl.F, wl.E, wl.k), dtype=torch.uint8, device="cuda")

        def fwd():
            moe.moe_forward_ex(x, d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg, out=out,
                               workspace=ws)

        for _ in range(3):
            fwd()
        torch.cuda.synchronize()
        ref = out.clone()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fwd()
        b.record(stream)
        torch.cuda.synchronize()
        eager_us = a.elapsed_time(b) * 1e3 / reps
        n_host = 32  # few enough that the launch queue never fills
        t0 = time.perf_counter()
        for _ in range(n_host):
            fwd()
        host_us = (time.perf_counter() - t0) * 1e6 / n_host
        torch.cuda.synchronize()

        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fwd()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            fwd()
        out.zero_()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        same = bool(torch.equal(out, ref))
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        graph_us = a.elapsed_time(b) * 1e3 / reps
        st, raw = moe.moe_device_error()
        if st != 0:
            raise RuntimeError(f"device error {moe.moe_status_string(st)} {raw:#x}")
        res.append({"T": T, "eager_us": eager_us, "graph_us": graph_us, "host_issue_us": host_us,
                    "graph_bitwise_equal": same,
                    "launches": moe.moe_forward_launches(cfg, T, wl.H, wl.F, wl.E, wl.k)})
        del g
    return res


def run_e2e(moe, torch, d, cfg, wl, args, stream):
    """Same metric through the C ABI with host buffers.  Every step copies its
    x in from pinned host memory and its output back to pinned host memory;
    as in a serving loop the copies run on their own streams, double-buffered,
    so that step i+1's input and step i-1's output move while step i runs."""
    T, H = wl.T, wl.H
    nb = 2
    x_host = [d["x"][:T].cpu().pin_memory() for _ in range(nb)]
    out_host = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    x_dev = [torch.empty_like(d["x"][:T]) for _ in range(nb)]
    out = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(nb)]
    ws = torch.empty(moe.moe_workspace_bytes(cfg, T, H, wl.F, wl.E, wl.k), dtype=torch.uint8, device="cuda")
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        copied = [torch.cuda.Event() for _ in range(n)]
        computed = [torch.cuda.Event() for _ in range(n)]
        drained = [torch.cuda.Event() for _ in range(n)]
        h2d.wait_stream(stream)  # nothing starts before the timing event
        d2h.wait_stream(stream)
        with torch.cuda.stream(h2d):
            x_dev[0].copy_(x_host[0], non_blocking=True)
            copied[0].record(h2d)
        for i in range(n):
            b = i % nb
            if i + 1 < n:  # prefetch the next step's input
                with torch.cuda.stream(h2d):
                    if i >= 1:
                        h2d.wait_event(computed[i - 1])  # its buffer was read by step i-1
                    x_dev[(i + 1) % nb].copy_(x_host[(i + 1) % nb], non_blocking=True)
                    copied[i + 1].record(h2d)
            stream.wait_event(copied[i])
            if i >= nb:
                stream.wait_event(drained[i - nb])  # out buffer b is free again
            moe.moe_forward_ex(x_dev[b], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], wl.k, cfg,
                               out=out[b], workspace=ws, stream=stream)
            computed[i].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[i])
                out_host[b].copy_(out[b], non_blocking=True)
                drained[i].record(d2h)
        stream.wait_event(drained[n - 1])

    run(args.warmup)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(args.steps)
    e.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e)
    nbytes = T * H * 2
    return {"value": T * args.steps / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes, "ms_per_step": ms / args.steps,
            "pipelining": "x in and out copied on side streams, double-buffered, overlapping the forward"}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_inputs(wl):
    """Host inputs for the oracle without the routed experts' weights (those
    are generated one expert at a time by expert_weights)."""
    inp = synth.make_inputs(wl, with_experts=False, with_shared=True)

    def expert_weights(name, e):
        return synth.expert_slice(wl, name, e)
    return inp, expert_weights


def cpu_baseline(wl, budget_s=15.0, sample_tokens=4):
    """The oracle, as it stands, on the host cores: forward_tokens over
    consecutive samples of the batch until about budget_s seconds pass (the
    experts' weights generated per call, as the oracle's expert_weights hook
    allows; generation included in the time)."""
    import oracle

    inp, ew = oracle_inputs(wl)
    t0 = time.perf_counter()
    done = 0
    start = 0
    while time.perf_counter() - t0 < budget_s and done < wl.T:
        toks = np.arange(start, min(start + sample_tokens, wl.T))
        oracle.forward_tokens(inp, wl, toks, expert_weights=ew)
        done += toks.size
        start += toks.size
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done} tokens of the T={wl.T} batch in groups of {sample_tokens} "
                      f"(float64 numpy, OpenBLAS threads for the matmuls), {el:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    kw = workload_overrides(args)
    T = args.T if args.T is not None else max(T_SWEEP[args.workload])
    wl = synth.workload(args.workload, T=T, **kw)
    inp, ew = oracle_inputs(wl)
    n = 4 if wl.E * wl.F * wl.H < 2e10 else 1

    def step(i):
        toks = (np.arange(n) + i * n) % wl.T
        oracle.forward_tokens(inp, wl, toks, expert_weights=ew)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    v = n * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) x, N(0,0.02) weights, bf16)",
            "config": {"workload": wl.label, "T": wl.T, "H": wl.H, "F": wl.F, "E": wl.E, "k": wl.k,
                       "parallelism": "host cores (rank 0 only)"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"each step: {n} tokens of the T={wl.T} batch, float64 numpy oracle"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="deepseek", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--alpha", type=float, default=None)
    ap.add_argument("--activation", default=None, choices=["silu", "gelu"],
                    help="gate activation of the experts (default: the workload's, SiLU)")
    ap.add_argument("--experts", type=int, default=None,
                    help="reduced expert count (same H, F, k, routing) for small profiling captures")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true",
                    help="time only the headline batch (not every point of the five layer shapes)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--schedule-ablation", action="store_true",
                    help="also time the persistent device schedule against host-read counts, fixed 64-row "
                         "tiles and one CTA per tile")
    ap.add_argument("--fusion-ablation", action="store_true",
                    help="also time the fused gate+up GEMM against two GEMMs + an element-wise pass")
    ap.add_argument("--expert-sweep", action="store_true",
                    help="also time the expert-count sweep (E = 8..128, F = 8*14336/E, H = 4096, top-2)")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the eager vs CUDA-graph decode-size timings on the Mixtral-shaped layer (also "
                         "skipped with --no-sweep)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload == "skew" and args.alpha is None:
        args.alpha = 0.0
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
