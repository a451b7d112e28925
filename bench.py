"""Benchmark of the dropless-MoE layer hot path on GB300.

One step = one pass of the whole layer (route -> dispatch -> grouped GEMM1 +
SwiGLU -> [MXFP8 quantise] -> grouped GEMM2 -> combine, plus the backward for
training workloads) over one batch of seeded synthetic input already resident
in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs one independent replica per GPU (one rank per GPU): the layer has no
exchange step on one GPU, so ranks share nothing but a barrier and the
max-over-ranks time; ``value`` is the units all ranks processed / that time.
Launched without torchrun, ``--gpus N`` starts the N ranks itself (torchrun on
127.0.0.1); under torchrun, ``--gpus`` must equal WORLD_SIZE.

The default workload is the largest single-GPU one: the DeepSeek-V3-shaped
layer's forward and backward, whole step graph-captured.  The same line carries
``targets``: the DeepSeek-V3-shaped MXFP8 grouped GEMMs against the FP8 peak and
the dispatch / combine stages of the other layer shapes against the copy
bandwidth, timed in the same process.
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

METRIC = "MoE layer grouped-GEMM TFLOPS & permute/combine GB/s on 1 GB300 vs roofline"
DEFAULT_WORKLOAD = "dsv3-bf16-train"
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about 1.5 s of timed work; reference arm: 3)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the targets leg (MXFP8 GEMMs of the DeepSeek-V3 layer, dispatch / combine of every shape)")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of replays of the step captured in one CUDA graph")
    ap.add_argument("--T", type=int, default=None, help="override tokens (small profiling cases)")
    ap.add_argument("--f", type=int, default=None, help="override expert hidden dim (profiling)")
    ap.add_argument("--E", type=int, default=None, help="override expert count (profiling)")
    ap.add_argument("--router-gemm", action="store_true",
                    help="also time the router GEMM fused with top-k (a seeded W_r) against routing from logits")
    ap.add_argument("--capacity-factor", type=float, default=None,
                    help="also time the capacity-based (drop/pad) forward with C = ceil(CF * T*k / E), the contrast case")
    return ap.parse_args()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def ensure_ranks(args):
    """Make the process count match --gpus: a plain launch with --gpus N > 1 re-runs
    this script under torchrun with N ranks (and exits with its status); a launch
    whose WORLD_SIZE differs from --gpus stops with an error."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world == args.gpus:
        return
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(args.gpus),
               "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
               os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.run(cmd).returncode)
    sys.exit(f"bench.py: --gpus {args.gpus} does not match WORLD_SIZE={world} (one rank per GPU)")


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class Clocks:
    """nvidia-smi sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.p = None
        # raw samples: MOE_CLOCKS_DIR if set (to keep them), else the temp directory
        self.path = os.path.join(os.environ.get("MOE_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.close()
        rows = [r.split(", ") for r in open(self.path).read().strip().splitlines() if r.strip()]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip() == "Active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm

def stage_bytes(w):
    """Algorithmic bytes of the bandwidth stages (each moved once).  The MXFP8
    training dispatch writes both MXFP8 forms of Xp (row-wise codes + scales,
    column-wise codes + scales): x read once, the two outputs written once."""
    s = 4 if w.dtype == "f32" else 2
    if w.dtype == "nvfp4":                      # NVFP4 codes + scales (x read twice: amax, scatter)
        xp_out = w.M * w.d * (0.5 + 1 / 16)
    elif w.dtype == "mxfp8" and w.backward:
        xp_out = w.M * w.d * 2 * (1 + 1 / 32)
    elif w.dtype == "mxfp8":
        xp_out = w.M * w.d * (1 + 1 / 32)
    else:
        xp_out = w.M * w.d * s
    permute = w.T * w.d * s + xp_out + w.T * w.k * 4 * 3 + w.M * 4
    combine = w.M * w.d * s + w.T * w.d * s + w.T * w.k * 8
    return permute, combine


def routing_summary(counts):
    """The per-expert row histogram of one step's routing: largest count, experts
    without rows, median of the others, experts with 1..127 rows, the share of the
    rows taken by the 8 busiest experts, and the padding share of 128-row tiles
    (rows computed past a group's end / rows computed)."""
    import numpy as np
    c = np.asarray(counts, dtype=np.int64)
    total = int(c.sum())
    nonempty = c[c > 0]
    tiled = int((-(-c // 128) * 128).sum())
    return {"max_count": int(c.max()) if c.size else 0,
            "empty_experts": int((c == 0).sum()),
            "median_nonempty": float(np.median(nonempty)) if nonempty.size else 0.0,
            "experts_below_128_rows": int(((c > 0) & (c < 128)).sum()),
            "top8_share": round(float(np.sort(c)[::-1][:8].sum()) / total, 4) if total else 0.0,
            "tile128_padding": round((tiled - total) / tiled, 4) if tiled else 0.0}


GEMM_KERNELS = ("gemm1", "gemm2", "dgrad2", "wgrad2", "dgrad1", "wgrad1")
KERNEL_NAMES = {"gemm1": "grouped GEMM1 (gate+up, fused SwiGLU)", "gemm2": "grouped GEMM2 (down)",
                "dgrad2": "GEMM2 data gradient with fused dSwiGLU", "wgrad2": "GEMM2 weight gradient",
                "dgrad1": "GEMM1 data gradient", "wgrad1": "GEMM1 weight gradient"}


def kernel_work(w, name, e_used):
    """Algorithmic FLOPs and HBM bytes of one launch of a grouped GEMM of the step:
    operands read once (the weights of the experts with tokens), outputs written
    once; the weight gradients write dW of every expert (zeros for empty ones).
    Quantised operands count their codes and scales; NVFP4 codes are half a byte."""
    M, d, f, E = w.M, w.d, w.f, w.E
    s = 4 if w.dtype == "f32" else 2                           # stored activations / gradients
    q = {"mxfp8": 1 + 1 / 32, "nvfp4": 0.5 + 1 / 16}.get(w.dtype, s)   # quantised GEMM operands
    mdf = M * d * f
    if name == "gemm1":
        h_out = M * f * (1 + 1 / 32) if (w.dtype == "mxfp8" and not w.backward) else M * f * s
        gu = M * 2 * f * s if w.backward else 0
        return 4.0 * mdf, e_used * 2 * f * d * q + M * d * q + h_out + gu
    if name == "gemm2":
        return 2.0 * mdf, e_used * d * f * q + M * f * q + M * d * s
    if name == "dgrad2":          # dYp . W2 -> dH, with G|U read and dG|dU written
        return 2.0 * mdf, M * d * q + e_used * d * f * q + M * 2 * f * s * 2
    if name == "wgrad2":
        return 2.0 * mdf, M * f * q + M * d * q + E * d * f * 2
    if name == "dgrad1":
        return 4.0 * mdf, M * 2 * f * q + e_used * 2 * f * d * q + M * d * s
    if name == "wgrad1":
        return 4.0 * mdf, M * d * q + M * 2 * f * q + E * 2 * f * d * 2
    raise KeyError(name)


def dtype_peak(w, pk, burst=True):
    """Tensor peak of the workload's GEMM dtype: the measured bf16 figure (burst or
    sustained) times the nominal dense ratio (fp8 2x, fp4 6x, tf32 0.5x)."""
    base = pk["bf16"] if burst else pk["bf16_sus"]
    return base * {"mxfp8": 2.0, "nvfp4": 6.0, "f32": 0.5}.get(w.dtype, 1.0)


def kernel_roofline(w, name, ms, e_used, pk, brief=False):
    """Achieved rate of one GEMM launch (eager, CUDA events) against the roofline that
    binds it: tensor time of its FLOPs at the dtype's burst peak vs HBM time of its
    algorithmic bytes at the measured copy bandwidth."""
    flops, nbytes = kernel_work(w, name, e_used)
    peak = dtype_peak(w, pk)
    tf = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm_bound = nbytes / (pk["hbm"] * 1e9) > flops / (peak * 1e12)
    if brief:
        return {"ms": round(ms, 4), "tflops": round(tf, 1), "tensor_frac": round(tf / peak, 4),
                "hbm_gbs": round(gbs, 1), "bound": "hbm" if hbm_bound else "tensor"}
    ratio = {"mxfp8": " x2 (fp8 nominal ratio)", "nvfp4": " x6 (fp4 nominal ratio, 13.5 / 2.25 PFLOP/s dense)",
             "f32": " x0.5 (tf32 nominal ratio)"}.get(w.dtype, "")
    common = {"kernel": KERNEL_NAMES[name], "kernel_key": name, "ms": round(ms, 4),
              "flops_per_launch": flops, "bytes_per_launch": round(nbytes), "experts_with_tokens": e_used,
              "tensor_frac_sustained": round(tf / dtype_peak(w, pk, burst=False), 4)}
    if hbm_bound:
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm"], 4), "peak_source": f"{pk['source']} copy bandwidth",
                "tensor_tflops": round(tf, 1), "tensor_frac": round(tf / peak, 4), **common}
    return {"bound": "tensor", "achieved": round(tf, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
            "frac": round(tf / peak, 4), "peak_source": f"{pk['source']} bf16 burst{ratio}",
            "hbm_gbs": round(gbs, 1), **common}


def kernel_traffic(name, workload):
    """DRAM bytes per launch of a GEMM kernel from the committed ncu summary
    (profiles/<kernel>_traffic_<workload>.txt), or None when there is none or the GEMM
    source has changed since the counters were taken."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", f"{name}_traffic_{workload}.txt")
    if not os.path.exists(prof):
        return None
    fields = dict(l.split(None, 1) for l in open(prof).read().splitlines()
                  if l.strip() and not l.startswith("#") and len(l.split(None, 1)) == 2)
    src = os.path.join(ROOT, "ragged_grouped_gemm_topk_gb300", "csrc", "gemm.cu")
    if fields.get("gemm_cu_sha256", "").strip() != hashlib.sha256(open(src, "rb").read()).hexdigest():
        return None
    try:
        return int(fields["dram_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


def run_ours(args, world, rank, local):
    import torch
    import ragged_grouped_gemm_topk_gb300 as pkg
    from ragged_grouped_gemm_topk_gb300 import build as pbuild
    from ragged_grouped_gemm_topk_gb300 import workloads as W

    pbuild.build()
    w = W.BY_NAME[args.workload]
    if args.T or args.f or args.E:
        w = w.scaled(T=args.T, f=args.f, E=args.E,
                     name=f"{w.name}-T{args.T or w.T}-f{args.f or w.f}-E{args.E or w.E}")
    dev = torch.device("cuda", torch.cuda.current_device())
    x = W.make_x(w, dev)
    W1, W2 = W.make_w1(w, dev), W.make_w2(w, dev)
    lg_h = W.make_logits(w)
    lg = torch.from_numpy(lg_h).to(dev)
    dy = W.make_dy(w, dev) if w.backward else None
    layer = pkg.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype=w.dtype, renormalize=w.renormalize,
                         training=w.backward)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        """One layer step.  With ``ev`` (a list), an event is recorded on the stream
        after each kernel group and appended as (name, event): the eager
        diagnostic pass; without it nothing but the kernels is enqueued."""
        def mark(name):
            if ev is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                ev.append((name, e))
        hook = mark if ev is not None else None
        mark("start")
        layer.route(lg)
        mark("route")
        layer.dispatch(x)
        mark("dispatch")
        layer.expert_mlp(mark=hook)
        mark("gemm2")
        layer.combine()
        mark("combine")
        if w.backward:
            layer.backward(dy, lg, mark=hook)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # Headline: the whole step (no host reads, device-side counts) captured once in
    # a CUDA graph and replayed; --eager times plain launches instead.
    run_step = step
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            step()
        run_step = graph.replay
    for _ in range(args.warmup):
        run_step()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.steps is None:
        # enough steps for ~1.5 s of timed work (several clock samples), same on every rank
        t_a.record(stream)
        run_step()
        t_b.record(stream)
        torch.cuda.synchronize()
        est = max_over_ranks(t_a.elapsed_time(t_b), world)
        args.steps = int(min(5000, max(20, math.ceil(1500.0 / max(est, 1e-3)))))
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0 = time.perf_counter()
    t_a.record(stream)
    for _ in range(args.steps):
        run_step()
    t_b.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    clk = clocks.stop()
    # Per-kernel breakdown: eager launches with events between the kernel groups (a
    # diagnostic pass after the timed region, at the clocks that load sustains).
    n_diag = min(args.steps or 20, 50)
    evs = []
    for _ in range(n_diag):
        ev = []
        step(ev)
        evs.append(ev)
    torch.cuda.synchronize()
    if int(layer.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.dev_status.item())}")
    kern = {}
    for ev in evs:
        for (_, e0), (name, e1) in zip(ev[:-1], ev[1:]):
            kern[name] = kern.get(name, 0.0) + e0.elapsed_time(e1) / n_diag
    per = {k: kern[k] for k in ("route", "dispatch", "gemm1", "gemm2", "combine")}
    bwd_names = [n for n, _ in evs[0]][6:] if w.backward else []
    per["backward"] = sum(kern[n] for n in bwd_names)
    per["step"] = sum(evs[i][0][1].elapsed_time(evs[i][-1][1]) for i in range(n_diag)) / n_diag
    ms = max_over_ranks(t_a.elapsed_time(t_b) / args.steps, world)
    flops = w.fwd_flops * (3 if w.backward else 1)
    value = world * flops / (ms * 1e-3) / 1e12
    pk = peaks()
    counts_h = layer.counts.cpu().numpy()             # read after the timed region
    e_used = int((counts_h > 0).sum())
    # the dominant GEMM of the step and the roofline that binds it: tensor time of its
    # FLOPs at the dtype's burst peak (the kernels are timed in a short eager pass)
    # against HBM time of its algorithmic bytes at the measured copy bandwidth
    gemms = {n: kern[n] for n in GEMM_KERNELS if n in kern}
    dom = max(gemms, key=gemms.get)
    roof = kernel_roofline(w, dom, gemms[dom], e_used, pk)
    kernels = {n: kernel_roofline(w, n, t, e_used, pk, brief=True) for n, t in gemms.items()}
    perm_b, comb_b = stage_bytes(w)
    g_disp, g_comb = graph_stage_ms(w, layer, x)
    launches = layer.launches_per_forward() + (layer.launches_per_backward() if w.backward else 0)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"f32": "tf32", "bf16": "bf16", "mxfp8": "mxfp8-e4m3", "nvfp4": "nvfp4-e2m1"}[w.dtype],
        "data": "synthetic (seeded; no dataset or trained weights)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "f": w.f,
                   "M_rows": w.M, "backward": w.backward,
                   "timing": "eager launches" if args.eager else "whole step captured in one CUDA graph, replayed",
                   "l2": l2_note(W1, W2),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "stages_ms": {k: round(v, 4) for k, v in per.items()},   # eager pass, events between stages
        "kernels_ms": {k: round(v, 4) for k, v in kern.items()},
        "routing": routing_summary(counts_h),
        "route_gbs": round((w.T * w.E * 4 + w.T * w.k * 8) / (max(per["route"], 1e-6) * 1e-3) / 1e9, 1),
        "permute_gbs": round(perm_b / (g_disp * 1e-3) / 1e9, 1),
        "combine_gbs": round(comb_b / (g_comb * 1e-3) / 1e9, 1),
        "bandwidth_stages": {
            "timing": "each stage replayed 20x in one CUDA graph (programmatic dependent launch between "
                      "replays, as inside the step's graph) over rotating input/output buffer sets larger "
                      "than L2 in total; eager = the stage between events in the eager pass",
            "dispatch_ms": round(g_disp, 4), "combine_ms": round(g_comb, 4),
            "dispatch_ms_eager": round(per["dispatch"], 4), "combine_ms_eager": round(per["combine"], 4),
            "hbm_frac_permute_eager": round(perm_b / (per["dispatch"] * 1e-3) / 1e9 / pk["hbm"], 4),
            "hbm_frac_combine_eager": round(comb_b / (per["combine"] * 1e-3) / 1e9 / pk["hbm"], 4)},
        "roofline": {**roof, "traffic": kernel_traffic(dom, w.name),
                     "hbm_frac_permute": round(perm_b / (g_disp * 1e-3) / 1e9 / pk["hbm"], 4),
                     "hbm_frac_combine": round(comb_b / (g_comb * 1e-3) / 1e9 / pk["hbm"], 4)},
        "gemm_kernels": kernels,
        "clocks": clk,
        "gpu_launches": launches * args.steps,
        "wall_s_timed": round(wall, 3),
    }
    if args.router_gemm:
        line["router_gemm"] = router_leg(w, x, lg, layer, pk)
    if args.capacity_factor is not None:
        line["capacity_contrast"] = capacity_leg(w, x, lg, layer, W1, W2, args.capacity_factor, ms)
    if not (args.no_targets or args.T or args.f or args.E):
        line["targets"] = targets_leg(pk, w, layer, x)
    if not args.no_e2e:
        line["e2e"] = e2e(args, w, layer, x, lg_h, dy, world, flops)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=12.0)
    return line


def stage_fns(w, layer, x, nbuf):
    """The dispatch and the combine of a layer shape over nbuf rotating sets of their
    input and output buffers (set 0 is the layer's own input): disp(i), comb(i).
    comb(i) reads the dispatch map disp(i) wrote, so disp(i) runs first."""
    import torch
    import ragged_grouped_gemm_topk_gb300 as pkg
    dev = x.device
    M, d = w.M, w.d
    xs = [x] + [x.clone() for _ in range(nbuf - 1)]
    i32 = dict(dtype=torch.int32, device=dev)
    maps = [dict(offsets=torch.empty(w.E + 1, **i32), dest_row=torch.empty(w.T, w.k, **i32),
                 src_pair=torch.empty(M, **i32)) for _ in range(nbuf)]
    u8 = dict(dtype=torch.uint8, device=dev)
    if w.dtype == "nvfp4":
        outs = [dict(codes=torch.empty(M, d // 2, **u8), scales=torch.empty(M, d // 16, **u8),
                     tensor_scale=torch.empty(2, dtype=torch.float32, device=dev)) for _ in range(nbuf)]
        def disp(i):
            pkg.moe_permute_nvfp4(xs[i], layer.topk_idx, layer.counts, w.E, workspace=layer.workspace,
                                  dev_status=layer.dev_status, **maps[i], **outs[i])
    elif w.dtype == "mxfp8":
        outs = [dict(xp=torch.empty(M, d, **u8), xp_scales=torch.empty(M, d // 32, **u8)) for _ in range(nbuf)]
        if w.backward:               # training: and the column-wise form, gathered from x
            q = [dict(codes=torch.empty(M, d, **u8),
                      scales=torch.empty(((M + 127) // 128 + w.E) * (d // 128), 512, **u8)) for _ in range(nbuf)]
        def disp(i):
            pkg.moe_permute(xs[i], layer.topk_idx, layer.counts, w.E, xp_dtype="mxfp8", workspace=layer.workspace,
                            dev_status=layer.dev_status, **maps[i], **outs[i])
            if w.backward:
                pkg.moe_quantize_mxfp8_gathered(xs[i], maps[i]["src_pair"], maps[i]["offsets"], w.E, w.k, axis=2,
                                                dev_status=layer.dev_status, **q[i])
    else:
        outs = [dict(xp=torch.empty(M, d, dtype=x.dtype, device=dev)) for _ in range(nbuf)]
        def disp(i):
            pkg.moe_permute(xs[i], layer.topk_idx, layer.counts, w.E, workspace=layer.workspace,
                            dev_status=layer.dev_status, **maps[i], **outs[i])
    yps = [layer.yp] + [layer.yp.clone() for _ in range(nbuf - 1)]
    ys = [torch.empty(w.T, d, dtype=layer.yp.dtype, device=dev) for _ in range(nbuf)]
    def comb(i):   # the dispatch map that disp(i) wrote (run disp first)
        pkg.moe_unpermute_combine(yps[i], maps[i]["dest_row"], layer.topk_w, out=ys[i], dev_status=layer.dev_status)
    return disp, comb, nbuf


def graph_stage_ms(w, layer, x, reps=20):
    """Device time of the dispatch and the combine stage as the step's graph runs them:
    each stage captured `reps` times in one CUDA graph (consecutive launches chained by
    programmatic dependent launch) over rotating sets of its input and output buffers,
    so that the sets together exceed L2 and every replay reads cold data."""
    import torch
    es = x.element_size()
    set_bytes = w.T * w.d * es + w.M * w.d * es
    nbuf = max(2, int(math.ceil(3 * L2_BYTES / set_bytes)))
    nbuf = min(nbuf, reps)
    disp, comb, nbuf = stage_fns(w, layer, x, nbuf)

    def timed(fn):
        for i in range(nbuf):                    # warm: every buffer set once, outside capture
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn(0)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for r in range(reps):
                fn(r % nbuf)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    t_d, t_c = timed(disp), timed(comb)
    if int(layer.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(layer.dev_status.item())} after the stage graphs")
    return t_d, t_c


def _launch_ms(fn, reps=10, warm=2, flush=None):
    """Median device time of single launches of fn (CUDA events around each call on
    the current stream), optionally after writing a buffer larger than L2."""
    import torch
    for _ in range(warm):
        fn()
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def _stand_in(w, dev, lg):
    """Routing state and buffers of a layer shape without its expert weights (for
    timing the dispatch and the combine alone)."""
    import types
    import torch
    import ragged_grouped_gemm_topk_gb300 as pkg
    i32 = dict(dtype=torch.int32, device=dev)
    store = torch.float32 if w.dtype == "f32" else torch.bfloat16
    L = types.SimpleNamespace(
        topk_idx=torch.empty(w.T, w.k, **i32), topk_w=torch.empty(w.T, w.k, dtype=torch.float32, device=dev),
        counts=torch.empty(w.E, **i32), dest_row=torch.empty(w.T, w.k, **i32),
        workspace=torch.empty(pkg.moe_permute_workspace_size(w.T, w.k, w.E), dtype=torch.uint8, device=dev),
        dev_status=torch.zeros(1, **i32),
        yp=(torch.randn(w.M, w.d, device=dev) * 0.1).to(store))
    pkg.moe_route_topk(lg, w.k, w.renormalize, topk_idx=L.topk_idx, topk_w=L.topk_w, counts=L.counts,
                       dev_status=L.dev_status)
    return L


def targets_leg(pk, main_w, main_layer, main_x):
    """The stated targets, timed in this process: the DeepSeek-V3-shaped MXFP8 layer's
    two grouped GEMMs (single eager launches, median of 10; FLOPs 4*M*d*f and
    2*M*d*f) against the FP8 tensor peak (2x the measured bf16 burst figure, and the
    nominal 4.5 PFLOP/s), the whole forward of that layer (graph replays), and the
    dispatch and combine of every bf16 / MXFP8 layer shape against the copy
    bandwidth, as the step's graph runs them and as single eager launches after an
    L2 flush."""
    import torch
    import ragged_grouped_gemm_topk_gb300 as pkg
    from ragged_grouped_gemm_topk_gb300 import workloads as W
    dev = main_x.device
    out = {}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    w = W.BY_NAME["dsv3-mxfp8"]
    x = W.make_x(w, dev)
    lg = torch.from_numpy(W.make_logits(w)).to(dev)
    W1, W2 = W.make_w1(w, dev), W.make_w2(w, dev)
    L = pkg.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype="mxfp8", renormalize=w.renormalize)
    del W1, W2
    L.route(lg)
    L.dispatch(x)
    g1 = lambda: pkg.moe_grouped_gemm_fwd_mxfp8_out(L.xq, L.W1q, L.offsets, epi="swiglu", A_scales=L.xs,  # noqa: E731
                                                    B_scales=L.W1s, codes=L.hq, scales=L.hs,
                                                    dev_status=L.dev_status)
    g2 = lambda: pkg.moe_grouped_gemm_fwd(L.hq, L.W2q, L.offsets, A_scales=L.hs, B_scales=L.W2s,  # noqa: E731
                                          out=L.yp, dev_status=L.dev_status)
    t1, t2 = _launch_ms(g1), _launch_ms(g2)
    f1, f2 = 4.0 * w.M * w.d * w.f, 2.0 * w.M * w.d * w.f
    fp8 = 2.0 * pk["bf16"]
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        L.forward(x, lg)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        L.forward(x, lg)
    step_ms = _time_ms(graph.replay, reps=20)
    counts = L.counts.cpu().numpy()
    out["dsv3_mxfp8"] = {
        "gemm1_ms": round(t1, 4), "gemm2_ms": round(t2, 4), "gemm_sum_ms": round(t1 + t2, 4),
        "gemm1_tflops": round(f1 / (t1 * 1e-3) / 1e12, 1), "gemm2_tflops": round(f2 / (t2 * 1e-3) / 1e12, 1),
        "gemm_sum_tflops": round((f1 + f2) / ((t1 + t2) * 1e-3) / 1e12, 1),
        "frac_of_2x_burst_bf16": round((f1 + f2) / ((t1 + t2) * 1e-3) / 1e12 / fp8, 4),
        "frac_of_4500_nominal": round((f1 + f2) / ((t1 + t2) * 1e-3) / 1e12 / 4500.0, 4),
        "gemm1_frac_of_2x_burst_bf16": round(f1 / (t1 * 1e-3) / 1e12 / fp8, 4),
        "gemm2_frac_of_2x_burst_bf16": round(f2 / (t2 * 1e-3) / 1e12 / fp8, 4),
        "target": "GEMM1 + GEMM2 at >= 0.60 of the FP8 tensor peak",
        "peak_tflops_2x_burst_bf16": round(fp8, 1),
        "forward_step_ms_graph": round(step_ms, 4),
        "forward_step_tflops_graph": round(w.fwd_flops / (step_ms * 1e-3) / 1e12, 1),
        "routing": routing_summary(counts),
        "timing": "single eager launches, median of 10 (2 warm-ups); weights larger than L2"}
    bw = {}
    shapes = [(W.BY_NAME["mixtral-bf16"], None), (W.BY_NAME["qwen3-235b-bf16"], None), (w, (L, x)),
              (main_w if main_w.name == "dsv3-bf16-train" else W.BY_NAME["dsv3-bf16-train"],
               (main_layer, main_x) if main_w.name == "dsv3-bf16-train" else None)]
    for ws, have in shapes:
        if have is None:
            xs = W.make_x(ws, dev)
            lgs = torch.from_numpy(W.make_logits(ws)).to(dev)
            Ls = _stand_in(ws, dev, lgs)
        else:
            Ls, xs = have
        perm_b, comb_b = stage_bytes(ws)
        g_d, g_c = graph_stage_ms(ws, Ls, xs)
        disp, comb, _ = stage_fns(ws, Ls, xs, 1)
        e_d = _launch_ms(lambda: disp(0), flush=flush)
        e_c = _launch_ms(lambda: comb(0), flush=flush)
        bw[ws.name] = {"permute_frac": round(perm_b / (g_d * 1e-3) / 1e9 / pk["hbm"], 4),
                       "combine_frac": round(comb_b / (g_c * 1e-3) / 1e9 / pk["hbm"], 4),
                       "permute_frac_eager": round(perm_b / (e_d * 1e-3) / 1e9 / pk["hbm"], 4),
                       "combine_frac_eager": round(comb_b / (e_c * 1e-3) / 1e9 / pk["hbm"], 4),
                       "permute_ms": round(g_d, 4), "combine_ms": round(g_c, 4),
                       "permute_ms_eager": round(e_d, 4), "combine_ms_eager": round(e_c, 4),
                       "permute_bytes": round(perm_b), "combine_bytes": round(comb_b)}
        if int(Ls.dev_status.item()) != 0:
            raise RuntimeError(f"device status {int(Ls.dev_status.item())} in the {ws.name} stages")
    out["bandwidth"] = {**bw, "target": "permute and combine at >= 0.70 of HBM bandwidth",
                        "peak_gbs": pk["hbm"], "peak_source": f"{pk['source']} copy bandwidth",
                        "timing": "graph: the stage replayed 20x in one CUDA graph over rotating buffer sets "
                                  "larger than L2; eager: single launches after an L2 flush, median of 10"}
    return out


def l2_note(W1, W2):
    nbytes = (W1.numel() + W2.numel()) * W1.element_size()
    if nbytes > L2_BYTES:
        return f"inputs larger than L2: {nbytes / 1e9:.2f} GB of expert weights streamed per step"
    return f"inputs smaller than L2 ({nbytes / 1e6:.1f} MB of expert weights, resident between steps; not flushed)"


def _time_ms(fn, reps=20, warm=3):
    """Mean device time of fn over reps calls (CUDA events on the current stream)."""
    import torch
    for _ in range(warm):
        fn()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(s)
    for _ in range(reps):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def router_leg(w, x, lg, layer, pk):
    """The router GEMM fused with the top-k selection (moe_route_topk_gemm, seeded
    W_r [E, d] ~ N(0, 1/d)) against routing from given logits (moe_route_topk):
    device time per call, eager, 20 calls after 3 warm-ups."""
    import torch
    import ragged_grouped_gemm_topk_gb300 as pkg
    from ragged_grouped_gemm_topk_gb300 import workloads as W
    if w.E > 256 or w.k > 8:
        return {"unavailable": "the fused router takes E <= 256 and k <= 8"}
    xr = x if x.dtype in (torch.bfloat16, torch.float32) else x.bfloat16()
    Wr = W.make_matrix(w.E, w.d, seed=1000 * w.seed + 9, dtype=xr.dtype, device=x.device, scale=w.d ** -0.5)
    fused = lambda: pkg.moe_route_topk_gemm(xr, Wr, w.k, w.renormalize, topk_idx=layer.topk_idx,
                                            topk_w=layer.topk_w, counts=layer.counts, dev_status=layer.dev_status)
    t_f = _time_ms(fused)
    t_p = _time_ms(lambda: layer.route(lg))
    # the unfused pair for comparison: the logits by a library GEMM (cuBLAS through
    # torch, bf16 or tf32 out, cast to fp32), then the selection from logits
    lg_out = torch.empty(w.T, w.E, dtype=torch.float32, device=x.device)
    t_g = _time_ms(lambda: lg_out.copy_(torch.matmul(xr, Wr.t())))
    flops = 2.0 * w.T * w.d * w.E
    peak = pk["bf16"] * (0.5 if xr.dtype == torch.float32 else 1.0)
    return {"ms": round(t_f, 4), "tflops": round(flops / (t_f * 1e-3) / 1e12, 1),
            "frac_of_peak": round(flops / (t_f * 1e-3) / 1e12 / peak, 4),
            "route_from_logits_ms": round(t_p, 4), "library_logits_gemm_ms": round(t_g, 4),
            "unfused_ms": round(t_g + t_p, 4), "logits_bytes_not_written": w.T * w.E * 4,
            "timing": "eager, 20 calls; one CTA per 128-token tile x E expert columns (E rounded up to 16), "
                      "or a cluster of 2-4 CTAs per tile splitting the contraction when the tiles leave SMs idle"}


def capacity_leg(w, x, lg, layer, W1, W2, cf, dropless_ms):
    """The capacity-based forward (the pages' contrast to dropless routing): each
    expert keeps its first C = ceil(cf * T*k / E) tokens, is padded to C rows, and
    the two grouped GEMMs run over all E*C rows; eager, 20 steps after 3 warm-ups."""
    import torch
    import ragged_grouped_gemm_topk_gb300 as pkg
    if w.dtype not in ("bf16", "f32") or w.backward:
        return {"unavailable": "capacity mode is built for the bf16 / fp32 forward"}
    C = int(math.ceil(cf * w.M / w.E))
    rows = w.E * C
    dev = x.device
    i32 = dict(dtype=torch.int32, device=dev)
    bufs = {"offsets": torch.empty(w.E + 1, **i32), "dest_row": torch.empty(w.T, w.k, **i32),
            "src_pair": torch.empty(max(rows, 1), **i32), "xp": torch.empty(max(rows, 1), w.d, dtype=x.dtype, device=dev)}
    ws = torch.empty(max(int(pkg.binding._lib.load().moe_permute_capacity_workspace_size(w.T, w.k, w.E)), 16),
                     dtype=torch.uint8, device=dev)
    h = torch.empty(max(rows, 1), w.f, dtype=x.dtype, device=dev)
    yp = torch.empty(max(rows, 1), w.d, dtype=x.dtype, device=dev)
    y = torch.empty(w.T, w.d, dtype=x.dtype, device=dev)

    def step():
        layer.route(lg)
        pkg.moe_permute_capacity(x, layer.topk_idx, layer.counts, w.E, C, workspace=ws,
                                 dev_status=layer.dev_status, **bufs)
        pkg.moe_grouped_gemm_fwd(bufs["xp"][:rows], W1, bufs["offsets"], epi="swiglu", out=h[:rows],
                                 dev_status=layer.dev_status)
        pkg.moe_grouped_gemm_fwd(h[:rows], W2, bufs["offsets"], out=yp[:rows], dev_status=layer.dev_status)
        pkg.moe_unpermute_combine_capacity(yp[:rows], bufs["dest_row"], layer.topk_w, out=y,
                                           dev_status=layer.dev_status)
    t = _time_ms(step)
    dropped = int((bufs["dest_row"] < 0).sum().item())
    kept = w.M - dropped
    return {"capacity_factor": cf, "capacity": C, "computed_rows": rows, "dropless_rows": w.M,
            "dropped_frac": round(dropped / w.M, 4), "padding_frac": round((rows - kept) / max(rows, 1), 4),
            "ms_per_step": round(t, 4), "dropless_ms_per_step": round(dropless_ms, 4),
            "useful_tflops": round(w.fwd_flops * kept / w.M / (t * 1e-3) / 1e12, 1),
            "timing": "eager, 20 steps (route, capacity dispatch, GEMM1 + SwiGLU, GEMM2, combine)"}


def e2e(args, w, layer, x, lg_h, dy, world, flops):
    """Same metric through the public API with host buffers: every step copies that
    step's inputs (x, logits, and dy when training) from pinned host memory and
    reads its result (y, and dx when training) back.  The copies run on a second
    stream with double-buffered device inputs and outputs, so step i's transfers
    overlap the neighbouring steps' kernels; the timed region holds exactly K input
    copies and K output copies and ends when the last output is in host memory.
    The layer calls of each buffer set (forward, and backward when training) are
    captured once in a CUDA graph and replayed per step, as a user runs a layer that
    reads no count on the host (--eager: plain calls instead)."""
    import torch
    train = dy is not None
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    xh = x.cpu().pin_memory()
    lgh = torch.from_numpy(lg_h).pin_memory()
    dyh = dy.cpu().pin_memory() if train else None
    yh = [torch.empty(w.T, w.d, dtype=x.dtype).pin_memory() for _ in range(2)]
    dxh = [torch.empty(w.T, w.d, dtype=x.dtype).pin_memory() for _ in range(2)] if train else None
    xd = [torch.empty_like(x) for _ in range(2)]
    lgd = [torch.empty(lgh.shape, dtype=torch.float32, device=x.device) for _ in range(2)]
    dyd = [torch.empty_like(dy) for _ in range(2)] if train else None
    yd = [torch.empty_like(x) for _ in range(2)]
    dxd = [torch.empty_like(x) for _ in range(2)] if train else None
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def h2d(b):
        with torch.cuda.stream(copy):
            xd[b].copy_(xh, non_blocking=True)
            lgd[b].copy_(lgh, non_blocking=True)
            if train:
                dyd[b].copy_(dyh, non_blocking=True)
            ev_in[b].record(copy)

    def body(b):
        layer.forward(xd[b], lgd[b], out=yd[b])
        if train:
            layer.backward(dyd[b], lgd[b], dx_out=dxd[b])

    calls = [lambda b=b: body(b) for b in range(2)]
    if not args.eager:
        h2d(0)
        h2d(1)
        comp.wait_stream(copy)
        side = torch.cuda.Stream()
        graphs = []
        for b in range(2):
            side.wait_stream(comp)
            with torch.cuda.stream(side):
                body(b)                 # warm, outside the capture
            comp.wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(b)
            graphs.append(g)
        torch.cuda.synchronize()
        calls = [g.replay for g in graphs]

    def run(n):
        h2d(0)
        if n > 1:
            h2d(1)
        for i in range(n):
            b = i % 2
            comp.wait_event(ev_in[b])
            calls[b]()
            ev_done[b].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(ev_done[b])
                yh[b].copy_(yd[b], non_blocking=True)
                if train:
                    dxh[b].copy_(dxd[b], non_blocking=True)
            if i + 2 < n:
                h2d(b)          # after the output copy of buffer b, in copy-stream order
        comp.wait_stream(copy)

    run(max(args.warmup, 2))
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    a.record(comp)
    copy.wait_stream(comp)
    run(args.steps)
    z.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(z) / args.steps, world)
    h2d_b = xh.numel() * xh.element_size() + lgh.numel() * 4 + (dyh.numel() * dyh.element_size() if train else 0)
    d2h_b = yh[0].numel() * yh[0].element_size() + (dxh[0].numel() * dxh[0].element_size() if train else 0)
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOPS",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d_b), "d2h_bytes_per_step": int(d2h_b),
            "overlap": "copies on a second stream, double-buffered",
            "layer_calls": "eager" if args.eager else "captured per buffer set in a CUDA graph, replayed"}


# ----------------------------------------------------------------------------- oracle (CPU) timing

def oracle_sample(w, n_tokens):
    """Inputs for the oracle on a bounded sample: the first n_tokens tokens of the
    workload (their activations and logits).  Only the experts those tokens route
    to are kept (their logit columns and weights): the top-k of every sampled
    token lies inside that set, so routing, weights and outputs are those of the
    full layer.  For timing, every kept expert carries the same seeded weight
    values (a broadcast view, so the host holds one expert's weights)."""
    import numpy as np
    import torch
    from ragged_grouped_gemm_topk_gb300 import workloads as W
    from oracle import moe as om
    lg = W.make_logits(w)[:n_tokens]
    g = torch.Generator().manual_seed(1000 * w.seed + 1)
    x = torch.randn(n_tokens, w.d, generator=g).to(w.torch_dtype).double().numpy()
    idx, _, _ = om.route_topk(lg, w.k, w.renormalize)
    used = np.unique(idx)
    gw = torch.Generator().manual_seed(1000 * w.seed + 2)
    w1 = (torch.randn(2 * w.f, w.d, generator=gw) / w.d ** 0.5).to(w.torch_dtype).double().numpy()
    w2 = (torch.randn(w.d, w.f, generator=gw) / w.f ** 0.5).to(w.torch_dtype).double().numpy()
    W1 = np.broadcast_to(w1, (len(used),) + w1.shape)
    W2 = np.broadcast_to(w2, (len(used),) + w2.shape)
    return x, np.ascontiguousarray(lg[:, used]), W1, W2


def cpu_baseline(w, budget_s=12.0):
    """Time the float64 oracle, as it stands, on a bounded token sample on the
    host cores; report TFLOPS of the algorithmic layer FLOPs it covered."""
    from oracle import moe as om
    cores = len(os.sched_getaffinity(0))
    n = 2
    per_tok = None
    while True:
        x, lg, W1, W2 = oracle_sample(w, n)
        t0 = time.perf_counter()
        fwd = om.layer_forward(x, lg, W1, W2, w.k, w.renormalize, mxfp8_operands=w.dtype == "mxfp8",
                               nvfp4_operands=w.dtype == "nvfp4")
        if w.backward:
            dy = x * 0 + 1.0
            om.layer_backward(fwd, dy, x, lg, W1, W2, w.k, w.renormalize, mxfp8_operands=w.dtype == "mxfp8")
        dt = time.perf_counter() - t0
        per_tok = dt / n
        if dt > budget_s / 3 or n >= w.T:
            break
        n = min(w.T, max(n * 2, int(n * budget_s / 2 / max(dt, 1e-3))))
    flops = w.fwd_flops * (3 if w.backward else 1) * n / w.T
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.T} tokens of {w.name} with the experts they route to "
                      f"(float64 numpy oracle), {dt:.1f} s",
            "s_per_token": per_tok}


def run_reference(args, world, rank):
    """The reference arm: the float64 CPU oracle on the same workload, each step a
    bounded token sample, timed on the host cores (rank 0 only)."""
    from ragged_grouped_gemm_topk_gb300 import workloads as W
    from oracle import moe as om
    w = W.BY_NAME[args.workload]
    if rank != 0:
        return None
    # tokens per step: the training workloads' oracle backward forms dense float64
    # weight gradients of every routed expert, so they take fewer tokens
    n = 4 if (w.backward or w.dtype in ("mxfp8", "nvfp4")) else 16
    x, lg, W1, W2 = oracle_sample(w, n)
    mx = w.dtype == "mxfp8"
    fp4 = w.dtype == "nvfp4"
    for _ in range(args.warmup):
        om.layer_forward(x, lg, W1, W2, w.k, w.renormalize, mxfp8_operands=mx, nvfp4_operands=fp4)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fwd = om.layer_forward(x, lg, W1, W2, w.k, w.renormalize, mxfp8_operands=mx, nvfp4_operands=fp4)
        if w.backward:
            om.layer_backward(fwd, x * 0 + 1.0, x, lg, W1, W2, w.k, w.renormalize, mxfp8_operands=mx)
    dt = (time.perf_counter() - t0) / args.steps
    flops = w.fwd_flops * (3 if w.backward else 1) * n / w.T
    value = flops / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "f": w.f},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": f"{n} of {w.T} tokens per step"},
            "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    ensure_ranks(args)
    world, rank, local = dist_setup(args)
    if args.impl == "reference" and args.steps is None:
        args.steps = 3
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
