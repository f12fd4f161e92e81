"""Benchmark of the Beam routed-MoE forward pass (libbeam_moe.so) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|skewed|tiny|T<n>]
                    [--impl reference] [--no-secondary] [--weights bf16|fp8] [--no-sweep]

A step is one beam_moe_forward call over one batch of T tokens: router, dispatch,
gate/up GEMM with SwiGLU, down GEMM, combine. Inputs and weights are synthetic, seeded,
of Beam's layer shape, resident in HBM before timing starts. L2 is flushed (a 512 MB
write) before every timed step; each step is bracketed by CUDA events on the launching
stream and the reported time is the sum over K steps. Under torchrun each rank runs an
independent replica on its own GPU (the path does not shard across GPUs here), and the
time is the max over ranks.

The default workload is Beam decode (T=16); one JSON line is printed by rank 0, carrying
the dominant kernel's roofline, the CPU oracle's throughput on a bounded sample, the
end-to-end number through host buffers (beam_moe_forward_host), and every other Beam
workload, each with its own rooflines and clocks: prefill (T=4096), the skewed load
(T=32768, 16 hot experts), the token-count sweep (T = 1 ... 16384) and the same block on
FP8 E4M3 expert weights (decode and prefill). --weights fp8 makes the FP8 block the
headline (used to profile it on smaller shapes).
--impl reference times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparse_moe_transformer_bias_b300 import abi, moe, workloads as W  # noqa: E402

METRIC = "Beam MoE-layer tokens/s (T=16 decode, T=4096 prefill); % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the expert
# kernel over its algorithmic bytes, from one-launch ncu captures of the same kernels on the
# same workloads with one group of 32 experts (the size a capture may hold): decode T=16 and
# the prefill-shaped T=512 (128 rows per expert, as at T=4096 with 256 experts). The bench
# scales its own algorithmic bytes by these ratios (the traffic is the touched experts'
# weights plus the activations, both in proportion). Keys: (workload, weights); remove an
# entry when its kernel changes after the capture.
TRAFFIC_RATIO = {("decode", "bf16"): 2521638912 / 2520514560, ("prefill", "bf16"): 2606890752 / 2642411520,
                 ("decode", "fp8"): 1266699776 / 1263534080, ("prefill", "fp8"): 1472596224 / 1385431040,
                 ("decode", "nvfp4"): 716357632 / 712049024, ("prefill", "nvfp4"): 836847616 / 844104064}

# Dense tensor rate of a contraction's own operand type over BF16's, from the nominal B300
# figures (BF16 2.25, FP8 4.5, NVFP4 13.5 PFLOP/s dense): the tensor peak of the FP8 and
# NVFP4 expert kernels is the measured BF16 burst rate times this ratio.
PEAK_RATIO = {"bf16": 1.0, "fp8": 2.0, "nvfp4": 6.0}


def peaks():
    try:
        p = json.load(open(PEAKS_FILE))
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload(name, n_group=8):
    if name in W.WORKLOADS:
        shape, T, hot = W.WORKLOADS[name]
    elif name.startswith("T") and name[1:].isdigit():
        shape, T, hot = W.BEAM, int(name[1:]), 0
    else:
        raise SystemExit(f"unknown workload {name}")
    if n_group != shape.n_group:
        # Fewer expert groups (32 experts each): a smaller device footprint of the same
        # kernels, used for profiler captures.
        shape = W.MoEShape(d=shape.d, I=shape.I, E=32 * n_group, n_group=n_group,
                           topk_group=min(shape.topk_group, n_group), top_k=shape.top_k, scale=shape.scale)
        name = f"{name}_E{shape.E}"
    return name, shape, T, hot


# ---------------------------------------------------------------- clocks sampler
class Clocks:
    FIELDS = ("clocks.sm", "clocks.max.sm", "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the measured arm
def make_layer(shape, T, hot, device, experts=None, seed=0):
    x = W.make_tokens(shape, T, seed, device)
    wr, b = W.make_router(shape, seed, device, hot_experts=hot)
    if experts is None:
        experts = W.make_experts(shape, seed, device)
    return x, wr, b, experts


def algorithmic(shape, T, n_touched, rows, fp8=False, fp4=False):
    """Algorithmic FLOPs and bytes of the whole layer and of the expert kernel (one launch:
    gate/up + SwiGLU and down over the touched experts' weights). FP8 experts: one byte
    per weight plus one FP32 scale per weight row. NVFP4 experts: half a byte per weight,
    one byte of block scale per 16 weights and one FP32 tensor scale per matrix; their
    activations (x, h) move as four NVFP4 pieces (codes 2 bytes and scales 1/4 byte per
    element) instead of BF16 rows."""
    d, I, E, K = shape.d, shape.I, shape.E, shape.top_k
    if fp4:
        w_bytes = n_touched * (3 * d * I // 2 + 3 * d * I // 16 + 3 * 4)
    elif fp8:
        w_bytes = n_touched * (3 * d * I + (2 * I + d) * 4)
    else:
        w_bytes = n_touched * 3 * d * I * 2
    layer_flops = T * (K * 3 * 2 * d * I + 2 * d * E)
    layer_bytes = w_bytes + E * d * 4 + E * 4 + 2 * T * d * 2 + T * K * 8
    # weights once; x_perm read, h written and read back, y (BF16) written
    act = 2 + 0.25 if fp4 else 2  # bytes per activation element moved
    mlp = {"flops": 2 * rows * d * I * 3,
           "bytes": int(w_bytes + rows * d * act + 2 * rows * I * act + rows * d * 2)}
    return layer_flops, layer_bytes, {"expert_mlp": mlp}


def measure(name, shape, T, hot, steps, warmup, experts, device, flush, pk, e2e=True, experts_fp8=None,
            experts_fp4=None):
    """Times beam_moe_forward (or, given experts_fp8 / experts_fp4, beam_moe_forward_fp8 /
    beam_moe_forward_nvfp4) on the workload."""
    x, wr, b, (wg, wu, wd) = make_layer(shape, T, hot, device, experts)
    out = torch.empty((T, shape.d), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()
    idx, _ = moe.route(x, wr, b, shape)
    n_touched = int(torch.unique(idx).numel())
    rows = T * shape.top_k
    fp8 = experts_fp8 is not None
    fp4 = experts_fp4 is not None

    def step():
        if fp4:
            moe.forward_nvfp4(x, wr, b, experts_fp4, shape, out=out, stream=stream)
        elif fp8:
            moe.forward_fp8(x, wr, b, experts_fp8, shape, out=out, stream=stream)
        else:
            moe.forward(x, wr, b, wg, wu, wd, shape, out=out, stream=stream)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    launches = abi.beam_moe_last_launch_count()

    # Pass 1: the headline, no stage events inside the step.
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    clocks = Clocks(torch.cuda.current_device())
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(steps):
        flush.zero_()
        e0[i].record(stream)
        step()
        e1[i].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    step_ms = [a.elapsed_time(c) for a, c in zip(e0, e1)]
    total_ms = max_over_ranks(sum(step_ms))

    # Pass 2: per-stage durations from the library's own events on the same stream.
    abi.beam_moe_timing_enable(True)
    stage_sum = {s: 0.0 for s in abi.STAGES}
    n2 = max(3, min(steps, 50))
    for _ in range(n2):
        flush.zero_()
        step()
        for k, v in abi.beam_moe_timing_read().items():
            stage_sum[k] += v
    abi.beam_moe_timing_enable(False)
    stage_ms = {k: v / n2 for k, v in stage_sum.items()}

    layer_flops, layer_bytes, kern = algorithmic(shape, T, n_touched, rows, fp8, fp4)
    t_roof_s = max(layer_flops / (pk["bf16_tflops"] * 1e12), layer_bytes / (pk["hbm_gbs"] * 1e9))
    ms_per_step = total_ms / steps
    dom = "expert_mlp"
    kf, kb = kern[dom]["flops"], kern[dom]["bytes"]
    t_dom = stage_ms[dom] * 1e-3
    wdt = "nvfp4" if fp4 else "fp8" if fp8 else "bf16"
    t_peak = pk["bf16_tflops"] * PEAK_RATIO[wdt]
    hbm_bound = kb / (pk["hbm_gbs"] * 1e9) >= kf / (t_peak * 1e12)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": kb / t_dom / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs, copy)"}
    else:
        roof = {"bound": "tensor", "achieved": kf / t_dom / 1e12, "peak": t_peak, "unit": "TFLOP/s",
                "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, burst)" + (
                    "" if wdt == "bf16" else f" x {PEAK_RATIO[wdt]:g}, the nominal {wdt.upper()}/BF16 dense ratio")}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["algorithmic_bytes" if hbm_bound else "algorithmic_flops"] = kb if hbm_bound else kf
    roof["kernel_ms"] = stage_ms[dom]
    ratio = TRAFFIC_RATIO.get((name, wdt))
    roof["traffic"] = int(ratio * kb) if ratio is not None and shape.n_group == 8 else None
    roof["frac_of_sustained"] = (kf / t_dom / 1e12 / (pk["bf16_tflops_sustained"] * PEAK_RATIO[wdt])
                                 if not hbm_bound else None)

    res = {
        "value": T * steps / (total_ms * 1e-3),
        "ms_per_step": ms_per_step,
        "roofline": roof,
        "ms_per_step_median": statistics.median(step_ms),
        "ms_per_step_p10": float(np.percentile(step_ms, 10)),
        "ms_per_step_p90": float(np.percentile(step_ms, 90)),
        "near_tie_tokens": near_tie_count(shape, moe.router_logits(x, wr, shape).cpu().numpy(), b.cpu().numpy()),
        "layer_roofline": {"t_roof_ms": t_roof_s * 1e3, "frac": t_roof_s * 1e3 / ms_per_step,
                           "flops": layer_flops, "bytes": layer_bytes,
                           "tensor_frac_of_burst": layer_flops / (pk["bf16_tflops"] * 1e12) / (ms_per_step * 1e-3),
                           "tensor_frac_of_sustained":
                               layer_flops / (pk["bf16_tflops_sustained"] * 1e12) / (ms_per_step * 1e-3)},
        "stage_ms": stage_ms,
        "n_touched_experts": n_touched,
        "gpu_launches": launches * steps,
        "clocks": clk,
    }
    if e2e:
        res["e2e"] = measure_e2e(shape, T, x, wr, b, wg, wu, wd, steps, warmup, flush)
    return res


def near_tie_count(shape, logits, bias, tie=1e-6):
    """Tokens whose selection sits on a near-tie, from the library's own FP32 logits: a gap
    below `tie` between neighbouring ranked group scores (the kept groups and the next one)
    or between neighbouring ranked biased scores of the kept groups' experts (the picks and
    the next one). On those tokens an ulp of the sigmoid can legitimately change a pick; the
    parity tests accept any tie-consistent choice there. A diagnostic of the inputs only."""
    T = logits.shape[0]
    G, S, TG, K = shape.n_group, shape.E // shape.n_group, shape.topk_group, shape.top_k
    s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    c = (s + bias[None, :].astype(np.float32)).astype(np.float32)
    top2 = -np.sort(-c.reshape(T, G, S), axis=2)[:, :, :2]
    gs = (top2[:, :, 0] + top2[:, :, 1]).astype(np.float32)
    order = np.argsort(-gs, axis=1, kind="stable")
    gsr = np.take_along_axis(gs, order, axis=1).astype(np.float64)
    ng = min(TG + 1, G)
    g_gap = (gsr[:, :ng - 1] - gsr[:, 1:ng]).min(axis=1) if ng > 1 else np.full(T, np.inf)
    kept = np.zeros((T, G), bool)
    np.put_along_axis(kept, order[:, :TG], True, axis=1)
    cc = np.where(np.repeat(kept, S, axis=1), c.astype(np.float64), -np.inf)
    cs = -np.sort(-cc, axis=1)[:, :min(K + 1, TG * S)]
    e_gap = np.where(np.isfinite(cs[:, 1:]), cs[:, :-1] - cs[:, 1:], np.inf).min(axis=1)
    return int(((g_gap < tie) | (e_gap < tie)).sum())


def measure_e2e(shape, T, x, wr, b, wg, wu, wd, steps, warmup, flush):
    """Host tokens in, host output out, through the library's host-buffer call
    (beam_moe_forward_host via moe.forward_host): the H2D copy of the step's tokens, the
    forward pass and the D2H copy of its output are all inside the timed region."""
    x_host = x.cpu().pin_memory()
    out_host = torch.empty((T, shape.d), dtype=torch.bfloat16, pin_memory=True)
    x_dev = torch.empty_like(x)
    out_dev = torch.empty((T, shape.d), dtype=torch.bfloat16, device=x.device)
    stream = torch.cuda.current_stream()
    # more untimed steps than the device-timed pass: the host path (pinned copies, pool
    # allocations, the first synchronisations after the stage-timing pass) settles slower
    for _ in range(max(warmup, 20)):
        flush.zero_()
        moe.forward_host(x_host, wr, b, wg, wu, wd, shape, out_host=out_host, stream=stream)
    total = 0.0
    per_step = []
    for _ in range(steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        moe.forward_host(x_host, wr, b, wg, wu, wd, shape, out_host=out_host, stream=stream)
        per_step.append(time.perf_counter() - t0)
        total += per_step[-1]
    total = max_over_ranks(total * 1e3) * 1e-3
    res = {"value": T * steps / total, "unit": "tokens/s", "h2d_bytes_per_step": T * shape.d * 2,
           "d2h_bytes_per_step": T * shape.d * 2, "call": "beam_moe_forward_host",
           "timer": "host wall clock around each synchronous step",
           "ms_per_step_p10_p50_p90": [float(np.percentile(per_step, q)) * 1e3 for q in (10, 50, 90)]}
    # The same through moe.ForwardGraph: the call captured once, replayed per step.
    g = moe.ForwardGraph(x_dev, wr, b, wg, wu, wd, shape, out=out_dev)
    stream = torch.cuda.current_stream()

    def graph_step():
        x_dev.copy_(x_host, non_blocking=True)
        g.replay()
        out_host.copy_(out_dev, non_blocking=True)
        stream.synchronize()

    for _ in range(warmup):
        graph_step()
    total = 0.0
    for _ in range(steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        graph_step()
        total += time.perf_counter() - t0
    total = max_over_ranks(total * 1e3) * 1e-3
    res["graph"] = {"value": T * steps / total, "unit": "tokens/s", "call": "moe.ForwardGraph.replay"}
    return res


# ---------------------------------------------------------------- CPU oracle arm
def oracle_tokens_per_s(shape, x, wr, b, wg, wu, wd, n_tokens, seed=0):
    """The CPU oracle (as it stands) on a seeded sample of tokens of the workload: router
    logits, routing, experts, combine. Returns (tokens/s, seconds, sample, threads)."""
    from oracle import oracle as O
    T = x.shape[0]
    tokens = W.sample_tokens(T, n_tokens, seed=seed).numpy()
    xb = O.bf16_bits(x)
    wr_h = wr.cpu().numpy()
    b_h = b.cpu().numpy()
    logits = O.router_logits(shape, xb[tokens], wr_h)
    idx, _ = O.route(shape, logits, b_h)
    needed = set(np.unique(idx).tolist())
    experts = O.experts_from(wg, wu, wd, only=needed)
    host = {e: experts(e) for e in needed}
    t0 = time.perf_counter()
    O.forward(shape, xb, b_h, lambda e: host.get(e), tokens=tokens, router_w=wr_h)
    dt = time.perf_counter() - t0
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return len(tokens) / dt, dt, f"{len(tokens)} of {T} tokens (seeded), full layer incl. router", threads


# ---------------------------------------------------------------- distributed plumbing
def rank_world():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(v):
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(v)], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return float(v)


def summary(workload_name, r, steps):
    """The per-workload object of the JSON line."""
    keys = ("value", "ms_per_step", "ms_per_step_median", "ms_per_step_p10", "ms_per_step_p90", "roofline",
            "layer_roofline", "stage_ms", "n_touched_experts", "near_tie_tokens", "gpu_launches", "clocks")
    out = {"workload": workload_name, "unit": "tokens/s", "steps": steps}
    out.update({k: r[k] for k in keys})
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-tokens", type=int, default=None)
    ap.add_argument("--n-group", type=int, default=8, help="expert groups of 32 (8 = Beam); fewer for profiling")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8", "nvfp4"], help="expert weights of the headline")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the token-count sweep T in {1, 8, 64, 256, 1024, 4096, 16384} (BF16)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, world, local = rank_world()
    name, shape, T, hot = workload(args.workload, args.n_group)
    pk, pk_src = peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        torch.cuda.set_device(local)
        x, wr, b, (wg, wu, wd) = make_layer(shape, T, hot, "cuda")
        n_tok = args.oracle_tokens or (4 if shape.d >= 1024 else 64)
        vals, secs = [], 0.0
        for i in range(args.warmup + args.steps):
            v, dt, sample, thr = oracle_tokens_per_s(shape, x, wr, b, wg, wu, wd, min(n_tok, T), seed=100 + i)
            if i >= args.warmup:
                vals.append(dt)
                secs += dt
        tokens = min(n_tok, T) * args.steps
        value = tokens / secs
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{name} T={T}", "d": shape.d, "I": shape.I, "E": shape.E},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                             "sample": f"{min(n_tok, T)} seeded tokens of {T} per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = "cuda"
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    experts = W.make_experts(shape, 0, device)
    torch.cuda.synchronize()

    head_fp8 = W.make_experts_fp8(shape, 0, device) if args.weights == "fp8" else None
    head_fp4 = W.make_experts_nvfp4(shape, 0, device) if args.weights == "nvfp4" else None
    res = measure(name, shape, T, hot, args.steps, args.warmup, experts, device, flush, pk,
                  e2e=head_fp8 is None and head_fp4 is None, experts_fp8=head_fp8, experts_fp4=head_fp4)
    del head_fp8, head_fp4
    secondary = None
    if not args.no_secondary and name == "decode" and args.n_group == 8 and args.weights == "bf16":
        s_name, s_shape, s_T, s_hot = workload("prefill")
        s_steps = max(10, min(args.steps, 50))
        sec = measure(s_name, s_shape, s_T, s_hot, s_steps, args.warmup, experts, device, flush, pk, e2e=False)
        secondary = summary(f"Beam prefill T={s_T}", sec, s_steps)

    skewed = None
    if not args.no_secondary and name == "decode" and args.n_group == 8 and args.weights == "bf16":
        k_name, k_shape, k_T, k_hot = workload("skewed")
        k_steps = max(10, min(args.steps, 20))
        r = measure(k_name, k_shape, k_T, k_hot, k_steps, args.warmup, experts, device, flush, pk, e2e=False)
        skewed = summary(f"Beam skewed load T={k_T}, {k_hot} hot experts (+0.5 bias)", r, k_steps)

    fp8 = None
    if not args.no_secondary and name == "decode" and args.n_group == 8 and args.weights == "bf16":
        # The block on FP8 E4M3 expert weights (same draws, quantised per row): decode and prefill.
        experts_fp8 = W.make_experts_fp8(shape, 0, device)
        fp8 = {}
        for f_name in ("decode", "prefill"):
            f_name, f_shape, f_T, f_hot = workload(f_name)
            f_steps = args.steps if f_name == "decode" else max(10, min(args.steps, 50))
            r = measure(f_name, f_shape, f_T, f_hot, f_steps, args.warmup, experts, device, flush, pk, e2e=False,
                        experts_fp8=experts_fp8)
            fp8[f_name] = summary(f"Beam {f_name} T={f_T}, FP8 E4M3 experts (per-row FP32 scales)", r, f_steps)
        del experts_fp8

    fp4 = None
    if not args.no_secondary and name == "decode" and args.n_group == 8 and args.weights == "bf16":
        # The block on NVFP4 expert weights (same draws, quantised): decode and prefill.
        experts_fp4 = W.make_experts_nvfp4(shape, 0, device)
        fp4 = {}
        for f_name in ("decode", "prefill"):
            f_name, f_shape, f_T, f_hot = workload(f_name)
            f_steps = args.steps if f_name == "decode" else max(10, min(args.steps, 50))
            r = measure(f_name, f_shape, f_T, f_hot, f_steps, args.warmup, experts, device, flush, pk, e2e=False,
                        experts_fp4=experts_fp4)
            fp4[f_name] = summary(f"Beam {f_name} T={f_T}, NVFP4 experts (E2M1, E4M3 block scales per 16, FP32 "
                                  f"tensor scale)", r, f_steps)
        del experts_fp4

    sweep = None
    if not args.no_sweep and not args.no_secondary and args.n_group == 8 and args.weights == "bf16":
        sweep = []
        for sT in W.SWEEP_T:
            s_name, s_shape, _, _ = workload(f"T{sT}")
            s_steps = max(10, min(args.steps, 30))
            r = measure(s_name, s_shape, sT, 0, s_steps, args.warmup, experts, device, flush, pk, e2e=False)
            lr = r["layer_roofline"]
            entry = summary(f"Beam T={sT}", r, s_steps)
            entry["T"] = sT
            entry["layer_bound"] = ("hbm" if lr["bytes"] / (pk["hbm_gbs"] * 1e9) >=
                                    lr["flops"] / (pk["bf16_tflops"] * 1e12) else "tensor")
            sweep.append(entry)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x, wr, b, (wg, wu, wd) = make_layer(shape, T, hot, device, experts)
        n_tok = args.oracle_tokens or min(T, 16)
        v, dt, sample, thr = oracle_tokens_per_s(shape, x, wr, b, wg, wu, wd, n_tok)
        cpu = {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle", "sample": sample, "seconds": dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"] * world, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "ms_per_step_median": res["ms_per_step_median"],
            "ms_per_step_p10": res["ms_per_step_p10"], "ms_per_step_p90": res["ms_per_step_p90"],
            "near_tie_tokens": res["near_tie_tokens"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) tokens, N(0,0.02^2) FP32 router, U(-0.1,0.1) bias, "
                    "BF16 experts std 1/sqrt(fan_in))",
            "config": {"workload": f"Beam MoE layer {name} T={T}" + (f", {hot} hot experts" if hot else ""),
                       "T": T, "d": shape.d, "I": shape.I, "E": shape.E, "n_group": shape.n_group,
                       "topk_group": shape.topk_group, "top_k": shape.top_k, "scale": shape.scale,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed (512 MB write) before every timed step",
                       "expert_weights": {"bf16": "BF16", "fp8": "FP8 E4M3, per-row FP32 scales",
                                          "nvfp4": "NVFP4 (E2M1, E4M3 block scales, FP32 tensor scale)"}[args.weights]},
            "roofline": {**res["roofline"],
                         "peak_source": res["roofline"]["peak_source"] if pk_src == "measured" else "fallback"},
            "layer_roofline": res["layer_roofline"],
            "stage_ms": res["stage_ms"],
            "n_touched_experts": res["n_touched_experts"],
            "cpu_baseline": cpu,
            "e2e": res.get("e2e"),
            "gpu_launches": res["gpu_launches"],
            "clocks": res["clocks"],
        }
        if secondary:
            line["secondary"] = secondary
        if skewed:
            line["skewed"] = skewed
        if fp8:
            line["fp8_experts"] = fp8
        if fp4:
            line["nvfp4_experts"] = fp4
        if sweep:
            line["sweep"] = sweep
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
