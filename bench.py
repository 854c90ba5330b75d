"""Benchmark of the GB300 MoE layer: one JSON line on rank 0.

A step is one whole moe_layer call (router projection, top-k softmax,
init_routing, permutation gather, grouped gate/up + activation, grouped down
projection, shared expert when present, finalize) over one batch of T tokens
already resident in HBM.  Default workload: the largest configured layer that
fits one GPU, the Ling-2.6-1T-style prefill layer (T=16384, D=8192, E=256,
top-8, I=2048, one shared expert of 2048, e4m3 weights with per-column scales,
bf16 activations); the Qwen3-MoE-style prefill layer (T=4096, D=2048, E=128,
top-8, I=768, bf16) is timed in the same run as a secondary line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline]

Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the
layer has no exchange step on one GPU's worth of tokens, so every rank runs
its own batch (weak scaling) and only the timing uses a barrier and a max.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE-layer tokens/s; % of HBM (decode) or tensor (prefill) roofline"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = [os.path.join(ROOT, "mixture_experts_layer_gating_gb300", "csrc", f)
                  for f in ("gemm_sm103.cu", "sm103_ptx.cuh")]


# ------------------------------------------------------------------ helpers
def peaks():
    try:
        p = json.load(open(PEAKS_PATH))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the GEMM kernel sources with comments and whitespace removed, so
    that an edit to a comment does not mark the committed ncu counters stale."""
    h = hashlib.sha1()
    for f in KERNEL_SOURCES:
        src = open(f).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:12]


def profiled_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(PROFILES, f"{kernel_tag}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_hash = re.search(r"kernel_source_sha1:\s*([0-9a-f]+)", txt)
    m_b = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_b or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t_start = time.time()
        else:
            self.t_end = time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = [l for (t, l) in self.lines if self.t_start and self.t_end and self.t_start <= t <= self.t_end + 0.15]
        used = inside if inside else [l for (_, l) in self.lines]
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in used:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[4]))
            except ValueError:
                pass
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons),
                "power_w": statistics.median(pw) if pw else None,
                "samples": len(sm),
                "window": "timed region" if inside else "whole run (timed region shorter than the sampling period)"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle timing
def time_oracle(shape, inp_cpu, n_tokens: int, seed: int = 1):
    """The CPU oracle, as it stands, on the first n_tokens tokens of the batch."""
    import oracle

    sub = dict(inp_cpu)
    sub["x"] = inp_cpu["x"][:n_tokens]
    t0 = time.perf_counter()
    oracle.moe_layer(sub, shape.k, shape.act, shape.renormalize)
    return time.perf_counter() - t0


def cpu_baseline(shape, inp_cpu, budget_s: float = 15.0):
    """Time the oracle, as it stands, on a bounded sample of about budget_s:
    the first n tokens of the batch (n grown until one call takes the budget),
    or the whole batch repeated when one pass is shorter than the budget."""
    n = min(shape.T, 16)
    while True:
        dt = time_oracle(shape, inp_cpu, n)
        if dt >= budget_s or n == shape.T:
            break
        n = int(min(shape.T, n * max(2.0, 0.8 * budget_s / max(dt, 1e-6))))
    reps, total, tokens = 1, dt, n
    while n == shape.T and total < budget_s and reps < 20:
        total += time_oracle(shape, inp_cpu, n)
        tokens += n
        reps += 1
    what = (f"first {n} of {shape.T} tokens" if n < shape.T else f"all {shape.T} tokens x {reps}")
    return {"value": tokens / total, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{what} of {shape.name}: oracle.moe_layer (numpy fp64, per-expert loop, "
                      f"BLAS threads = host cores), {total:.1f} s"}


def router_planes(T: int, E: int, D: int) -> int:
    """Split-K planes of the router projection: the library's rule (a
    function of the shape only), restated for the byte counts below."""
    tiles = ((T + 127) // 128) * ((E + 255) // 256)
    kb = (D + 63) // 64
    ks = max(1, min(8, 148 // max(1, tiles), kb // 4))
    kbs = (kb + ks - 1) // ks
    return (kb + kbs - 1) // kbs


def fused_router(T: int, E: int, D: int, k: int, act_dtype: str, anywhere: bool = False) -> bool:
    """Whether moe_layer runs the router projection and the top-k softmax as
    one kernel: the library's rule (MOE_OPT_FUSED_ROUTING on, its default),
    restated -- bf16 activations, 64 <= E <= 512, E and D multiples of 8,
    k <= 32, not a batch the CUDA-core projection takes (at most 64 tokens
    and 2^25 multiply-adds, slices of D of at most 1024), and a fused grid of
    at least 64 CTAs (not required with `anywhere`: options 2 and 3)."""
    if act_dtype != "bf16" or not 64 <= E <= 512 or E % 8 or D % 8 or k > 32:
        return False
    S = router_planes(T, E, D)
    small = T <= 64 and E % 2 == 0 and T * D * E <= 2 ** 25 and (D + S - 1) // S <= 1024
    # at least 64 CTAs: token tiles of 128 x slices of D (clusters of <= 4) x expert halves
    tiles, nh, kb = (T + 127) // 128, (2 if E > 256 else 1), (D + 63) // 64
    want = max(1, min(4 // nh, 148 // max(1, tiles * nh), kb // 4))
    ck = 1
    while 2 * ck <= want:
        ck *= 2
    return not small and (anywhere or tiles * ck * nh >= 64)


def memory_kernel_bytes(shape, name: str, rows_form_bytes: int, nk: bool = False):
    """Algorithmic bytes of one launch of a memory-bound kernel of the layer
    (every tensor it must read or write, once), or None for the GEMMs.
    rows_form_bytes: bytes per element of the GEMM A rows (2); nk: fp8
    weights stored K-contiguous (h in bf16 rather than fp32)."""
    T, D, E, k, I, Is, R = shape.T, shape.D, shape.E, shape.k, shape.I, shape.I_shared, shape.R
    ab = 4 if shape.act_dtype == "f32" else 2
    S = router_planes(T, E, D)
    bias = shape.zipf > 0
    fp8 = shape.w_dtype == "fp8_e4m3"
    gathered = rows_form_bytes if fp8 else ab  # bytes per element of the permuted rows
    yb = 2 if fp8 else 4  # expert and shared-expert rows: bf16 for fp8 layers, else fp32
    hb = 2 if (fp8 and nk) else 4  # h as the gate/up pass writes it
    nseg_hist = E * 4 * max(1, (R + 1023) // 1024)
    table = {
        "topk_softmax": S * T * E * 4 + (E * 4 if bias else 0) + (T * E * 4 if (S > 1 or bias) else 0) + 8 * T * k,
        # x and W_g read once, logits written, ids and weights written
        "router_topk": T * D * ab + D * E * ab + (E * 4 if bias else 0) + T * E * 4 + 8 * T * k,
        "route_hist": 4 * R + nseg_hist,
        "route_scan_scatter": 4 * R + nseg_hist + 8 * E + 8 * R,
        # ids read twice (histogram, scatter), sorted_rows and dest written
        "route_sort": 8 * R + 8 * R + 8 * E,
        "route_permute": 4 * R + T * D * gathered + R * D * gathered + 8 * R + 8 * E,
        "permute_gather": T * D * gathered + 4 * R + R * D * gathered,
        "finalize": R * D * yb + 4 * R + 4 * T * k + (T * D * yb if Is else 0) + T * D * ab,
        "combine_round": T * D * 4 + (T * D * yb if Is else 0) + T * D * ab,
    }
    rf = rows_form_bytes
    for pre in ("x_to_fp16", "x_to_e4m3x2", "x_to_e4m3"):
        table[pre] = T * D * ab + T * D * rf + 4 * T
    for pre in ("h_to_fp16", "h_to_e4m3x2", "h_to_e4m3"):
        table[pre] = R * I * hb + R * I * rf + 4 * R
        table["shared_" + pre] = T * Is * hb + T * Is * rf + 4 * T
    return table.get(name)


# ------------------------------------------------------------------ arms
def workload_shape(args):
    import dataclasses

    shape = workloads.CONFIGS[args.workload]
    if args.tokens:
        shape = shape.with_tokens(args.tokens)
    if args.experts:
        shape = dataclasses.replace(shape, E=args.experts, name=f"{shape.name}@E{args.experts}")
    return shape


def run_reference(args, world, rank):
    shape = workload_shape(args)
    if rank != 0:
        return
    inp = workloads.make_inputs(shape, seed=0, device="cpu") if not torch.cuda.is_available() else \
        {k: (v.cpu() if isinstance(v, torch.Tensor) else v)
         for k, v in workloads.make_inputs(shape, seed=0, device="cuda").items()}
    # each step: the oracle on a bounded sample so the whole run stays within
    # minutes -- the first n tokens, n doubled from 1 (one call is also the
    # first warm-up) while a call stays under half the per-step target and
    # n < T; the target is --ref-step-s, lowered so that all warm-up and timed
    # steps take about --ref-total-s
    step_s = min(args.ref_step_s, args.ref_total_s / max(1, args.steps + args.warmup))
    if args.ref_tokens:
        n = min(shape.T, args.ref_tokens)
        done = 0
    else:
        n = 1
        dt = time_oracle(shape, inp, n)
        while n < shape.T and dt < 0.5 * step_s:
            n = min(shape.T, 2 * n)
            dt = time_oracle(shape, inp, n)
        done = 1
    for _ in range(max(0, args.warmup - done)):
        time_oracle(shape, inp, n)
    times = [time_oracle(shape, inp, n) for _ in range(args.steps)]
    tot = sum(times)
    value = n * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Gaussian inputs of the workload's shapes)",
        "config": dict(workloads.config_summary(shape), sample_tokens_per_step=n),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"first {n} of {shape.T} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def set_options(moe, args):
    if args.pair_tiles is not None:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, args.pair_tiles)
    if args.gather_a is not None:
        moe.moe_set_option(moe.MOE_OPT_GATHER_A, args.gather_a)
    if args.decode_kernel is not None:
        moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, args.decode_kernel)
    if args.no_pdl:
        moe.moe_set_option(moe.MOE_OPT_PDL, 0)
    if args.serial_shared:
        moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, 0)
    if getattr(args, "shared_fork", None) is not None:
        moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, args.shared_fork)
    if args.fused_combine:
        moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, 1)
    if getattr(args, "b_prefetch", None) is not None:
        moe.moe_set_option(moe.MOE_OPT_B_PREFETCH, args.b_prefetch)
    if getattr(args, "shared_ctas", None) is not None:
        moe.moe_set_option(moe.MOE_OPT_SHARED_CTAS, args.shared_ctas)
    if getattr(args, "dynamic_tiles", None) is not None:
        moe.moe_set_option(moe.MOE_OPT_DYNAMIC_TILES, args.dynamic_tiles)
    if getattr(args, "split_routing", False):
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, 0)
    elif getattr(args, "cluster_sort", False):
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, 3)
    if args.lpt:
        moe.moe_set_option(moe.MOE_OPT_TILE_ORDER, 1)
    if args.shared_in_gemm:
        moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 1)


def pct(v, q):
    """q-th percentile (linear interpolation) of a list."""
    v = sorted(v)
    if not v:
        return None
    pos = (len(v) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (pos - lo)


def gather_mode(shape, opt: int, shared_in_gemm: bool) -> int:
    """Where moe_layer's routed gate/up pass takes its rows for MOE_OPT_GATHER_A
    = opt (the library's rule, restated): 0 = the gather kernel's permuted copy,
    1 = TMA gather4, 2 = cp.async gather warps (bf16 layers); the default (3)
    takes 2 for bf16 layers with at least 32 routed rows per expert, else 0,
    and 0 when the shared expert runs inside the routed GEMMs."""
    if shape.act_dtype == "f32" or opt == 0:
        return 0
    bf16 = shape.w_dtype == "bf16"
    if opt == 1:
        return 1
    if opt == 2:
        return 2 if bf16 else 1
    if shared_in_gemm:
        return 0
    return 2 if (bf16 and shape.R >= 32 * shape.E) else 0


def kernel_names(shape, nk, gather_a=3, a8=False, fused=False, shared_in_gemm=False, fused_routing=True,
                 hist_sort=True):
    """Names of the kernels one moe_layer call launches, in launch order.
    hist_sort=False: MOE_OPT_FUSED_ROUTING 3 (the fused router wherever the
    shape allows, init_routing without its histograms)."""
    fp8 = shape.w_dtype == "fp8_e4m3"
    rows = "e4m3" if a8 else "e4m3x2" if nk else "fp16"  # the A-row form of fp8 layers
    router = ["router_topk"] if fused_routing and fused_router(shape.T, shape.E, shape.D, shape.k,
                                                                shape.act_dtype, not hist_sort) \
        else ["router_gemm", "topk_softmax"]
    names = ([f"x_to_{rows}"] if fp8 else []) + router
    if shape.R <= 8192:  # small batches: init_routing + gather in one kernel
        names += ["route_permute"]
    else:
        # one launch: from the fused router's per-CTA histograms, or as one
        # cluster up to 65536 rows
        one = fused_routing and ((hist_sort and router == ["router_topk"]) or shape.R <= 65536)
        names += ["route_sort"] if one else ["route_hist", "route_scan_scatter"]
        names += ["permute_gather"] if gather_mode(shape, gather_a, shared_in_gemm) == 0 else []
    names += ["w13_gate_up"]
    names += [f"h_to_{rows}"] if fp8 else []
    names += ["w2_down"]
    if shape.I_shared and not shared_in_gemm:
        names += ["shared_w13"] + ([f"shared_h_to_{rows}"] if fp8 else []) + ["shared_w2"]
    names += ["combine_round" if fused else "finalize"]
    return names


def measure(args, world, rank, local, shape, primary: bool, layout: str):
    """Time moe_layer on one workload; returns the fields of a bench line.
    layout: the fp8 weight layout ("kn", "nk", or "nk_a8" for W8A8)."""
    import mixture_experts_layer_gating_gb300 as moe

    dev = torch.device("cuda", local)
    inp = workloads.make_inputs(shape, seed=rank, device=dev, weights_seed=0)
    fp8 = shape.w_dtype == "fp8_e4m3"
    nk = fp8 and layout in ("nk", "nk_a8")
    a8 = fp8 and layout == "nk_a8"
    cfg = moe.config_from_shape(shape, layout if fp8 else "kn")
    ws = moe.alloc_workspace(cfg, device=dev)
    out = torch.empty((shape.T, shape.D), dtype=workloads.torch_dtype(shape.act_dtype), device=dev)
    stream = torch.cuda.current_stream(dev)
    # fp8 weights in the K-contiguous layout: transposed once here, before any
    # timing, as a serving engine does when it loads a checkpoint
    W = {n: inp[n] for n in ("W13", "W2", "W13s", "W2s")}
    if nk:
        W = {n: (None if v is None else moe.pack_weights_nk(v)) for n, v in W.items()}
        torch.cuda.synchronize()
    args_layer = (inp["x"], inp["Wg"], inp["logit_bias"], W["W13"], inp["s13"], W["W2"], inp["s2"],
                  W["W13s"], inp["s13s"], W["W2s"], inp["s2s"])

    def step(x=None):
        a = list(args_layer)
        if x is not None:
            a[0] = x
        moe.moe_layer(cfg, *a, out, ws, stream)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flags = moe.moe_read_device_status(ws)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x}")

    # ---- device-resident timed region: exactly K steps, an event before each
    # (per-step durations for the percentiles), barrier + synchronize around
    def timed_loop(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        barrier(world)
        torch.cuda.synchronize()
        for i in range(n):
            evs[i].record(stream)
            step()
        evs[n].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return evs[0].elapsed_time(evs[n]), [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]

    sampler.mark("start")
    t_ms, per_step = timed_loop(args.steps)
    # percentiles over at least --min-window-ms of steps: the K timed steps,
    # extended by further loops of K steps when they are shorter
    window_ms, window = t_ms, list(per_step)
    while window_ms < args.min_window_ms:
        dt, more = timed_loop(args.steps)
        window_ms += dt
        window += more
    sampler.mark("end")
    t_ms = max_over_ranks(t_ms, world)
    ms_step = t_ms / args.steps
    value = shape.T * world / (t_ms / 1e3 / args.steps)
    step_stats = {"median_ms": pct(window, 50), "p10_ms": pct(window, 10), "p90_ms": pct(window, 90),
                  "mean_ms": sum(window) / len(window), "steps": len(window), "window_ms": window_ms}

    # ---- per-kernel durations (instrumented pass, same work, after the timed region)
    L = moe.moe_layer_launch_count(cfg)
    fused = args.fused_combine and shape.act_dtype == "bf16" and (nk or not fp8)
    gather_opt = 3 if args.gather_a is None else args.gather_a
    in_gemm = (args.shared_in_gemm and shape.I_shared == shape.I and shape.I_shared > 0 and
               shape.act_dtype == "bf16" and (nk or not fp8) and gather_opt in (0, 3))
    names = kernel_names(shape, nk, gather_opt, a8, fused, in_gemm, not args.split_routing,
                         not args.cluster_sort)
    assert len(names) == L
    # the traced steps are enqueued back to back (one synchronisation at the
    # end) so that the device, not the host's launch latency, sets each
    # interval; the first one, enqueued on an idle device, is left out
    per = [[] for _ in range(L)]
    traced = []
    for _ in range(args.steps + 1):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(L + 1)]
        moe.moe_set_trace_events(evs)
        step()
        moe.moe_set_trace_events(None)
        traced.append(evs)
    torch.cuda.synchronize()
    for evs in traced[1:]:
        for i in range(L):
            per[i].append(evs[i].elapsed_time(evs[i + 1]))
    kernels_us = {n: 1e3 * statistics.mean(v) for n, v in zip(names, per)}
    # achieved HBM bandwidth of the memory-bound kernels (routing, gather,
    # row conversions, combine): algorithmic bytes / event-timed duration
    pk_hbm = peaks()["hbm_gbs"]
    memory_kernels = {}
    for n, t_us in kernels_us.items():
        nb = memory_kernel_bytes(shape, n, 1 if a8 else 2, nk)
        if nb is not None and t_us > 0:
            gbs = nb / (t_us * 1e3)
            memory_kernels[n] = {"bytes": nb, "us": t_us, "gbs": gbs, "frac_hbm": gbs / pk_hbm}

    # ---- end to end through the public API with host buffers: every step
    # copies its x from pinned host memory and its out back, on copy streams,
    # double-buffered so that step i's copies overlap the layers of steps i +- 1
    # (as a serving loop would run it)
    x_host = inp["x"].cpu().pin_memory()
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_ready, x_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    for b in range(2):  # every buffer starts free
        x_free[b].record(stream)
        out_free[b].record(stream)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(x_free[b])  # the layer of step i - 2 has read x_dev[b]
            x_dev[b].copy_(x_host, non_blocking=True)
            x_ready[b].record(h2d)
        stream.wait_event(x_ready[b])
        stream.wait_event(out_free[b])  # step i - 2's out has been copied out
        a = list(args_layer)
        a[0] = x_dev[b]
        moe.moe_layer(cfg, *a, out_dev[b], ws, stream)
        x_free[b].record(stream)
        out_ready[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(out_ready[b])
            out_host[b].copy_(out_dev[b], non_blocking=True)
            out_free[b].record(d2h)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(d2h)  # the timed region ends once the last out is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    sampler.stop()

    # ---- roofline of the dominant kernel
    counts = moe.workspace_view(ws, cfg, "counts", (shape.E,), torch.int32).cpu()
    active = int((counts > 0).sum())
    pk = peaks()
    R, D, I = shape.R, shape.D, shape.I
    wb = {"f32": 4, "bf16": 2, "fp8_e4m3": 1}[shape.w_dtype]
    ab = 4 if shape.act_dtype == "f32" else 2
    w13_flops = 2.0 * R * D * 2 * I
    w13_bytes = active * D * 2 * I * wb + R * D * ab + R * I * ab
    w2_flops = 2.0 * R * I * D
    w2_bytes = active * I * D * wb + R * I * ab + R * D * ab
    cand = {"w13_gate_up": (w13_flops, w13_bytes), "w2_down": (w2_flops, w2_bytes)}
    dom = max(cand, key=lambda n: kernels_us[n])
    flops, nbytes = cand[dom]
    t_s = kernels_us[dom] / 1e6
    clocks = sampler.summary()
    # the tensor peak: the burst figure, or the sustained one (a seconds-long
    # GEMM loop under the power cap) when the power cap acted during the timed
    # region, as it does for long tensor-bound steps
    capped = "sw_power_cap" in clocks.get("reasons", [])
    bf16_peak = pk["bf16_tflops_sustained"] if capped else pk["bf16_tflops"]
    # fp8 weights stored K-contiguous run on the e4m3 kind, whose dense peak
    # is twice the 16-bit one (the nominal 4.5 / 2.25 PFLOP/s ratio times the
    # measured bf16 figure); everything else on the 16-bit kinds
    kind_peak = 2 * bf16_peak if nk else bf16_peak
    if a8:  # one-term rows: the rows carry 1 byte per element
        nbytes -= (R * D + R * I) * (ab - 1) if dom == "w13_gate_up" else R * I * (ab - 1)
    t_tensor = flops / (kind_peak * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": flops / t_s / 1e12, "peak": kind_peak, "unit": "TFLOP/s"}
        if nk and not a8:
            roof["peak_kind"] = ("kind::f8f6f4 (e4m3): 2 x the measured bf16 figure; achieved counts "
                                 "the method's multiply-adds once (2 R D 2I for W13), although x and h "
                                 "ride as two e4m3 terms, i.e. two tensor-core products per multiply-add")
            roof["bf16_equivalent_frac"] = (flops / t_s / 1e12) / bf16_peak
        elif a8:
            roof["peak_kind"] = ("kind::f8f6f4 (e4m3): 2 x the measured bf16 figure; W8A8, one "
                                 "tensor-core product per multiply-add")
    else:
        roof = {"bound": "hbm", "achieved": nbytes / t_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the committed ncu summary of this kernel on this workload (W8A8: its own)
    tr = profiled_traffic(dom, (args.workload if primary else shape_key(shape)) + ("_w8a8" if a8 else ""))
    roof.update({"traffic": tr, "kernel": dom, "kernel_us": kernels_us[dom],
                 "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
                 "tensor_frac": (flops / t_s / 1e12) / kind_peak,
                 "hbm_frac": (nbytes / t_s / 1e9) / pk["hbm_gbs"],
                 "peak_source": "%s (MEASURED_PEAKS.json: HBM copy; bf16 %s)" % (
                     pk["source"], "sustained, sw_power_cap seen" if capped else "burst")})
    layer_flops = workloads.layer_flops(shape)
    layer_bytes = workloads.layer_bytes(shape, active_experts=active)
    t_roof = max(layer_flops / (kind_peak * 1e12), layer_bytes / (pk["hbm_gbs"] * 1e9))
    sm_mhz = clocks.get("sm_mhz")

    res = {
        "value": value, "ms_per_step": ms_step, "step_ms": step_stats,
        "dtype": ("f32" if shape.act_dtype == "f32" else "e4m3" if nk else "fp16" if fp8 else "bf16"),
        "layout": layout if fp8 else None,
        "config": dict(workloads.config_summary(shape), parallelism=f"replicas x{world}",
                       l2="inputs larger than L2: %.2f GB of expert weights per step" %
                          (shape.E * workloads.expert_weight_bytes(shape.D, shape.I, shape.w_dtype) / 1e9),
                       active_experts=active,
                       **({"fp8_layout": {
                           "nk": "nk: weights transposed once by moe_pack_weights_nk before timing; "
                                 "e4m3 tensor-core kind, x and h as two e4m3 terms (bf16 activations)",
                           "nk_a8": "nk_a8: W8A8 -- weights as for nk; x and h quantised per row to "
                                    "one e4m3 term with a dynamic scale (changes the result)",
                           "kn": "kn: weights as drawn; expanded to fp16 on chip"}[layout]}
                          if fp8 else {})),
        "roofline": roof,
        "layer_roofline": {"t_roofline_us": t_roof * 1e6, "t_measured_us": ms_step * 1e3,
                           "frac": t_roof / (ms_step / 1e3), "flops": layer_flops, "bytes": layer_bytes,
                           "tensor_peak_tflops": kind_peak},
        # time x median SM clock: the step's length in SM cycles, comparable across clocks
        "mcycles_per_step": (ms_step * 1e-3 * sm_mhz) if sm_mhz else None,
        "kernels_us": kernels_us,
        "memory_kernels": memory_kernels,
        "e2e": {"value": shape.T * world / (e2e_ms / 1e3 / args.steps), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": out_host[0].numel() * out_host[0].element_size(),
                "pipelined": "x and out copies on two copy streams, double-buffered"},
        "gpu_launches": L * args.steps,
        "clocks": clocks,
    }
    cpu_inp = None
    if primary and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_inp = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    del inp, W, args_layer, ws, out, x_dev, out_dev
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if cpu_inp is not None:
        res["cpu_baseline"] = cpu_baseline(shape, cpu_inp, budget_s=args.cpu_budget)
    return res


def shape_key(shape):
    for k, v in workloads.CONFIGS.items():
        if v == shape:
            return k
    return shape.name


def run_ours(args, world, rank, local):
    import mixture_experts_layer_gating_gb300 as moe
    from mixture_experts_layer_gating_gb300 import _build

    if rank == 0 or not os.path.exists(moe.LIB_PATH):
        _build.build()
    barrier(world)
    moe.load_library()
    set_options(moe, args)
    shape = workload_shape(args)
    res = measure(args, world, rank, local, shape, primary=True, layout=args.fp8_layout)
    line = {
        "metric": METRIC, "value": res.pop("value"), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res.pop("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": res.pop("dtype"),
        "data": "synthetic (seeded Gaussian x ~ N(0,1), weights ~ N(0,0.02), random init)",
    }
    line.pop("layout", None)
    line.update(res)
    line.pop("layout", None)
    # secondary workloads of the same run (their own timed regions, after the
    # primary one): NAME or NAME:LAYOUT (fp8 weight layout kn / nk / nk_a8)
    sec = {}
    for item in (args.secondary.split(",") if args.secondary else []):
        name, _, layout = item.partition(":")
        layout = layout or args.fp8_layout
        if not name or (name == args.workload and layout == args.fp8_layout):
            continue
        r = measure(args, world, rank, local, workloads.CONFIGS[name], primary=False, layout=layout)
        sec[item] = {k: r[k] for k in ("value", "ms_per_step", "step_ms", "dtype", "layout", "roofline",
                                        "layer_roofline", "kernels_us", "e2e", "clocks")}
        sec[item]["workload"] = r["config"]["workload"]
    if sec:
        line["secondary"] = sec
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ling_prefill", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--secondary", default="qwen3_prefill,ling_prefill:nk_a8",
                    help="comma-separated workloads (NAME or NAME:FP8_LAYOUT) also timed in the same "
                         "run, each under 'secondary'; empty for none")
    ap.add_argument("--min-window-ms", type=float, default=200.0,
                    help="per-step percentiles cover at least this much device time (the K timed "
                         "steps, repeated when shorter)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="reference arm: tokens per step (0: grown until one step takes ~--ref-step-s)")
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--ref-total-s", type=float, default=150.0,
                    help="reference arm: about this many seconds for all warm-up and timed steps")
    ap.add_argument("--pair-tiles", type=int, nargs="?", const=1, default=None,
                    help="moe_set_option MOE_OPT_PAIR_TILES: 0 never 2-CTA tiles, 1 always (swapped "
                         "tails), 2 always without swapped tails, 3 (default) by rows per group")
    ap.add_argument("--decode-kernel", type=int, default=None, choices=[0, 1, 2, 3],
                    help="moe_set_option MOE_OPT_DECODE_KERNEL (0 off, 1 auto, 2/3 always with 64/16-row tiles)")
    ap.add_argument("--gather-a", type=int, nargs="?", const=1, default=None, choices=[0, 1, 2, 3],
                    help="where the routed gate/up GEMM takes its rows (moe_set_option MOE_OPT_GATHER_A: "
                         "0 = permuted copy, 1 = TMA gather4, 2 = cp.async gather warps for bf16 "
                         "layers, 3 = the library's default rule)")
    ap.add_argument("--fp8-layout", default="nk", choices=["kn", "nk", "nk_a8"],
                    help="fp8 workloads: weights transposed once to [.., N, K] and run on the e4m3 "
                         "tensor-core kind (nk, default), or as drawn and expanded to fp16 on chip (kn); "
                         "nk_a8: nk weights with W8A8 activations (opt-in, changes the result)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="plain stream order instead of programmatic dependent launch (MOE_OPT_PDL 0)")
    ap.add_argument("--b-prefetch", type=int, default=None,
                    help="weight boxes prefetched into L2 this many k-blocks ahead (MOE_OPT_B_PREFETCH)")
    ap.add_argument("--shared-ctas", type=int, default=None,
                    help="CTAs of the shared expert's side-stream GEMMs (MOE_OPT_SHARED_CTAS; 0 = all)")
    ap.add_argument("--dynamic-tiles", type=int, default=None, choices=[0, 1, 2],
                    help="grouped GEMM tiles handed out by an atomic counter (MOE_OPT_DYNAMIC_TILES)")
    ap.add_argument("--split-routing", action="store_true",
                    help="router projection and top-k, histogram and scatter as separate launches "
                         "(MOE_OPT_FUSED_ROUTING 0)")
    ap.add_argument("--cluster-sort", action="store_true",
                    help="init_routing without the fused router's histograms: the 8-CTA cluster "
                         "sort (two kernels above 65536 rows); MOE_OPT_FUSED_ROUTING 3")
    ap.add_argument("--fused-combine", action="store_true",
                    help="routed down pass adds weighted rows into [T, D] fp32 sums "
                         "(MOE_OPT_FUSED_COMBINE 1; the combine's summation order then varies)")
    ap.add_argument("--shared-in-gemm", action="store_true",
                    help="shared expert as the last group of the routed GEMMs (MOE_OPT_SHARED_IN_GEMM 1; "
                         "layers whose I_shared equals I)")
    ap.add_argument("--lpt", action="store_true",
                    help="grouped GEMMs run the experts heaviest first (MOE_OPT_TILE_ORDER 1)")
    ap.add_argument("--serial-shared", action="store_true",
                    help="shared expert on the caller's stream (MOE_OPT_SHARED_STREAM 0)")
    ap.add_argument("--shared-fork", type=int, default=None, choices=[1, 2],
                    help="where the shared expert's side stream forks (MOE_OPT_SHARED_STREAM: "
                         "1 = once x is ready, 2 = after init_routing)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T of the workload (smaller cases for profiling)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E of the workload (smaller cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
