#!/usr/bin/env python3
"""Benchmark of the MoE layer forward on B300: tokens/s of one full forward (router,
dispatch, grouped SwiGLU experts, combine, balance statistics) through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One JSON line on stdout (rank 0).  With --gpus N > 1 (launched by torch.distributed.run)
every rank runs an independent replica of the workload on its own GPU (weak scaling; the
forward has no cross-GPU exchange) and the time is the maximum over ranks.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload
(rank 0 only), the slow program the kernels are checked against.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_top_routing_router_b300 import configs as K  # noqa: E402
from sparse_top_routing_router_b300.inputs import make_inputs, token_subset  # noqa: E402

METRIC = "MoE-layer fwd tokens/s on 1 B300; % of bf16 tensor peak / % of HBM roofline"
DEFAULT_CONFIG = K.DSV3_PREFILL.name
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "expert_gate_up_traffic.txt")
L2_BYTES = 126e6          # B300 L2
KERNEL_SRC = os.path.join(ROOT, "sparse_top_routing_router_b300", "csrc", "expert_tc.cu")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_seed(base: int, rank: int) -> int:
    """Each replica draws its own batch (and weights) from seed base + rank."""
    return base + rank


def reduce_max_ms(ms: float, dist, device) -> float:
    """The timed region ends when the slowest rank ends: max over ranks."""
    if dist is None:
        return ms
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(cfg: K.MoEConfig, cf) -> dict:
    d = {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I, "k": cfg.k,
         "score": cfg.score, "renorm": cfg.renorm, "shared_expert": cfg.shared,
         "capacity_factor": cf, "router": "fp32", "experts": cfg.dtype}
    if cfg.n_groups > 1:
        d["router_groups"] = {"n_groups": cfg.n_groups, "topk_groups": cfg.topk_groups}
    if cfg.fp8_experts:
        d["experts"] = "fp8 e4m3, per-output-channel fp32 scales; bf16 activations"
    if cfg.expert_choice:
        d["routing"] = f"expert choice: each expert takes its C = T*k/E = {cfg.T * cfg.k // cfg.E} best tokens"
    return d


def l2_note(cfg: K.MoEConfig) -> str:
    elt = 1 if cfg.fp8_experts else (2 if cfg.dtype == "bf16" else 4)
    w_all = 3 * (cfg.E + (1 if cfg.shared else 0)) * cfg.H * cfg.I * elt
    if w_all > L2_BYTES:
        return (f"inputs larger than L2: the expert weights ({w_all / 1e9:.2f} GB) stream "
                "from HBM every step (no flush needed)")
    return (f"inputs fit in L2 ({w_all / 1e6:.1f} MB of weights), no flush: a latency "
            "figure, not a bandwidth one")


def run_config(cfg: K.MoEConfig, cf, world: int) -> dict:
    """The `config` object of both arms' JSON lines: the workload, the L2 statement and
    the parallelism."""
    return dict(workload_config(cfg, cf), l2=l2_note(cfg), parallelism=f"replicas x{world}")


def step_quantiles(xs) -> dict:
    """Median, 10th and 90th percentile (linear interpolation) and mean of per-step times."""
    v = sorted(xs)

    def q(f):
        if len(v) == 1:
            return v[0]
        pos = f * (len(v) - 1)
        lo = int(pos)
        hi = min(lo + 1, len(v) - 1)
        return v[lo] + (v[hi] - v[lo]) * (pos - lo)
    return {"median": q(0.5), "p10": q(0.1), "p90": q(0.9), "mean": sum(v) / len(v)}


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampled every 100 ms; only samples stamped inside the timed region's
    wall-clock window are kept."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        import datetime
        sm, mx, pw, reasons, n_all = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            n_all += 1
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm_v, mx_v = float(f[2]), float(f[3])
            except ValueError:
                continue
            if self.t0 is not None and not (self.t0 - 0.05 <= ts <= self.t1 + 0.05):
                continue
            sm.append(sm_v)
            mx.append(mx_v)
            try:
                pw.append(float(f[4]))
            except ValueError:
                pass
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "samples": len(sm), "samples_total": n_all,
                "window_s": (self.t1 - self.t0) if self.t0 else None,
                "reasons": sorted(reasons)}


def traffic_from_profile(workload: str):
    """DRAM bytes per launch of expert_gate_up on `workload` from the committed ncu
    summary (a JSON list, one entry per workload), if the kernel source has not changed
    since the counters were taken; else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as fh:
        j = json.load(fh)
    with open(KERNEL_SRC, "rb") as fh:
        h = hashlib.sha256(fh.read()).hexdigest()[:16]
    for entry in (j if isinstance(j, list) else [j]):
        if entry.get("workload_name") == workload and entry.get("kernel_sha") == h:
            return dict(entry, source=f"ncu capture, {os.path.relpath(PROFILE_TRAFFIC, ROOT)}")
    return None


def traffic_for_run(cfg: K.MoEConfig, cf, bias_update):
    """The committed traffic figure for this run, if it runs what was profiled: the
    workload's own routing.  A routing variant (group limit, expert choice, bias updates,
    FP8 weights), other sizes or a capacity other than the workload's first one see other
    expert sizes, so such a run carries no traffic figure."""
    plain = (cfg == K.BY_NAME.get(cfg.name) and bias_update is None
             and cf == (cfg.capacity_factors[0] if cfg.capacity_factors else None))
    return traffic_from_profile(cfg.name) if plain else None


# --------------------------------------------------------------------------- CPU oracle

def blas_threads() -> int:
    """Threads numpy's BLAS runs the oracle's matmuls with."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


_HOST_CACHE = {}
_HOST_CACHE_BYTES = [0]
_HOST_CACHE_LIMIT = 16 << 30


def host_cores() -> int:
    """Host cores this process may run on (nproc)."""
    return len(os.sched_getaffinity(0))


def _host(t):
    """t as a float64 host array (exact for bf16 and fp32 values), kept for later calls
    while the cache holds less than 16 GB."""
    key = (t.data_ptr(), tuple(t.shape), str(t.device))
    a = _HOST_CACHE.get(key)
    if a is None:
        a = t.detach().to("cpu").double().numpy()
        if _HOST_CACHE_BYTES[0] + a.nbytes <= _HOST_CACHE_LIMIT:
            _HOST_CACHE[key] = a
            _HOST_CACHE_BYTES[0] += a.nbytes
    return a


def oracle_sample(cfg, d, cf, n_tokens: int, seed: int):
    """Time the fp64 oracle: routing of all T tokens (capacity is a batch property), then
    experts + combine for a seeded sample of n_tokens.  The inputs are staged in host
    memory as float64 (exact for bf16 and fp32 values) before the clock starts; the expert
    weights are widened one expert at a time as the oracle asks for them, and the time
    spent widening is taken off the clock, so the figure is the oracle's arithmetic, not
    its staging.  Widened weights are kept for later samples up to 16 GB.
    Returns (t_route, t_ffn, tokens, staging seconds)."""
    from oracle import moe_oracle as O

    X = _host(d["X"])
    Wg = _host(d["Wg"])
    bias = _host(d["bias"]) if "bias" in d else None
    lb = _host(d["logit_bias"]) if "logit_bias" in d else None
    C = None if cf is None else O.capacity(cf, cfg.T, cfg.k, cfg.E)
    t0 = time.perf_counter()
    if cfg.expert_choice:
        r = O.route_expert_choice(X, Wg, cfg.k, cfg.score, lb)
    else:
        r = O.route(X, Wg, cfg.k, cfg.score, cfg.renorm, bias, lb, C, n_groups=cfg.n_groups,
                    topk_groups=cfg.topk_groups)
    t_route = time.perf_counter() - t0
    tokens = token_subset(cfg.T, n_tokens, seed).numpy()
    staging = [0.0]

    def fetch(e):
        t1 = time.perf_counter()
        w = (_host(d["W_gate"][e]), _host(d["W_up"][e]), _host(d["W_down"][e]))
        staging[0] += time.perf_counter() - t1
        return w

    shared = (_host(d["Ws_gate"]), _host(d["Ws_up"]), _host(d["Ws_down"])) if cfg.shared \
        else None
    t0 = time.perf_counter()
    O.combine_subset(X, r, fetch, tokens, shared)
    t_ffn = time.perf_counter() - t0 - staging[0]
    return t_route, t_ffn, int(tokens.size), staging[0]


def cpu_baseline_sample(cfg, d, cf, first_tokens: int, min_seconds: float):
    """The oracle's bounded sample for the cpu_baseline figure: routing of all T tokens,
    then experts + combine of a seeded token sample that starts at first_tokens and
    doubles until the expert stage alone takes min_seconds or the sample is the whole
    batch.  A few tokens would time the oracle reading each touched expert's weights
    rather than computing with them: per token it touches k whole experts."""
    n = max(1, min(first_tokens, cfg.T))
    res = oracle_sample(cfg, d, cf, n, seed=1)
    while res[1] < min_seconds and res[2] < cfg.T:
        n = min(2 * n, cfg.T)
        res = oracle_sample(cfg, d, cf, n, seed=1)
    return res


def reference_sample_tokens(cfg, d, cf, step_budget_s: float) -> int:
    """Tokens per step of the reference arm: the sample doubles from 2 while one step, by
    the wall clock and with its weight staging, stays within step_budget_s.  Each size
    runs twice on seeds of its own and the second run is timed: the first stages the
    experts a small layer then keeps cached (as the timed steps find them), while a large
    layer stages fresh experts on both, as its timed steps do."""
    n, seed = min(2, cfg.T), 10_000
    oracle_sample(cfg, d, cf, n, seed)      # stages the inputs
    while n < cfg.T:
        n2 = min(2 * n, cfg.T)
        oracle_sample(cfg, d, cf, n2, seed + 1)
        t0 = time.perf_counter()
        oracle_sample(cfg, d, cf, n2, seed + 2)
        seed += 2
        if time.perf_counter() - t0 > step_budget_s:
            break
        n = n2
    return n


def run_reference(args, cfg, cf):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    d = make_inputs(cfg, device="cpu")
    step_budget = args.ref_budget / (args.warmup + args.steps)
    n_tok = args.ref_tokens or reference_sample_tokens(cfg, d, cf, step_budget)
    times = []
    for i in range(args.warmup + args.steps):
        tr, tf, n, _ = oracle_sample(cfg, d, cf, n_tok, seed=1 + i)
        if i >= args.warmup:
            times.append(tr + tf * cfg.T / n)      # seconds per step, extrapolated to T
        log(f"reference step {i}: route {tr:.2f}s ffn({n} tok) {tf:.2f}s")
    q = step_quantiles(times)
    v = cfg.T / q["median"]
    sample = (f"routing of all {cfg.T} tokens + experts/combine of {n_tok} seeded tokens "
              f"per step (expert weights widened to float64 outside the clock), throughput "
              f"extrapolated to {cfg.T} tokens; median of {args.steps} steps"
              + ("" if args.ref_tokens else
                 f"; {n_tok} = the largest doubling of 2 tokens whose step fits "
                 f"{step_budget:.2f} s, so the {args.warmup + args.steps} steps take about "
                 f"{args.ref_budget:g} s"))
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * q["median"],
            "step_ms": {k: 1e3 * x for k, x in q.items()},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": run_config(cfg, cf, world),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": blas_threads(),
                             "nproc": host_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm

def run_gpu(args, cfg, cf):
    from sparse_top_routing_router_b300.layer import MoELayer

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    d = make_inputs(cfg, device=dev, seed=replica_seed(cfg.seed, rank))
    layer = MoELayer(cfg, d, device=local, capacity_factor=cf, bias_gamma=args.bias_update)
    X = d["X"]
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        layer.forward(X)
    torch.cuda.synchronize()
    st = layer.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    R = int(layer.offsets[-1].item())

    # ---- timed region: K forwards, inputs resident in HBM
    layer.ctx.set_tracing(True)
    layer.ctx.trace_read()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    barrier()
    torch.cuda.synchronize()
    # one event between consecutive forwards: per-step times, median reported
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clocks.mark(True)
    evs[0].record(stream)
    for i in range(args.steps):
        layer.forward(X)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    barrier()
    clk = clocks.stop()
    ms = evs[0].elapsed_time(evs[-1])
    q = step_quantiles([evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)])
    kern = layer.ctx.trace_read()
    layer.ctx.set_tracing(False)
    ms = reduce_max_ms(ms, dist, dev)
    q = {key: reduce_max_ms(v, dist, dev) for key, v in q.items()}
    ms_step = q["median"]
    value = world * cfg.T / (ms_step / 1e3)

    # ---- end to end: pinned host X -> device, forward, bf16 Y -> pinned host, the copies
    # of neighbouring steps overlapped with compute (MoELayer.host_pipeline)
    Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    Xh.copy_(X)
    Yh = [torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    layer.host_pipeline(Xh, Yh, 4, stream)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.host_pipeline(Xh, Yh, args.steps, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1)
    ms_e2e = reduce_max_ms(ms_e2e, dist, dev)
    st = layer.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    pk = peaks()
    n_gu, ms_gu = kern["expert_gate_up"]
    n_dn, ms_dn = kern["expert_down"]
    gu_ms = ms_gu / max(n_gu, 1)
    dn_ms = ms_dn / max(n_dn, 1)
    rows = R + (cfg.T if cfg.shared else 0)
    gu_flops = 2.0 * rows * cfg.H * 2 * cfg.I
    dn_flops = 2.0 * rows * cfg.I * cfg.H
    elt = 2 if cfg.dtype == "bf16" else 4
    welt = 1 if cfg.fp8_experts else elt     # bytes per expert weight
    # experts with at least one kept row (expert-choice routing fills every expert)
    n_touched = int((torch.diff(layer.offsets) > 0).sum().item()) + (1 if cfg.shared else 0)
    # FP8 weights carry one fp32 scale per output channel: 2I + H per expert
    w_scales = 4 * (2 * cfg.I + cfg.H) if cfg.fp8_experts else 0
    w_touched = n_touched * (3 * cfg.H * cfg.I * welt + w_scales)
    # algorithmic bytes of the gate/up launch: its touched weights once, A rows in, h out
    gu_bytes = (n_touched * (2 * cfg.H * cfg.I * welt + (8 * cfg.I if cfg.fp8_experts else 0))
                + rows * cfg.H * elt + rows * cfg.I * 2)
    prof = traffic_for_run(cfg, cf, args.bias_update)
    # The headline fraction is against the burst bf16 peak (a cuBLAS GEMM timed alone);
    # the fraction of the power-capped sustained peak is given beside it.
    tpeak = pk["bf16_tflops"]
    spk = pk.get("bf16_tflops_sustained")
    src = "%s (MEASURED_PEAKS.json, burst)" % pk["source"]
    tensor_bound = R >= 128 * cfg.E     # rows per expert fill the 128/256-row tiles
    if tensor_bound:
        achieved = gu_flops / (gu_ms / 1e3) / 1e12
        roofline = {"kernel": "expert_gate_up", "bound": "tensor", "achieved": achieved,
                    "peak": tpeak, "unit": "TFLOP/s", "frac": achieved / tpeak,
                    "frac_of_sustained_peak": achieved / spk if spk else None,
                    "peak_source": src, "timed_region_ms": ms,
                    "traffic": prof["dram_bytes_per_launch"] if prof else None,
                    "traffic_source": prof["source"] if prof else None,
                    "algorithmic_flops_per_launch": gu_flops,
                    "algorithmic_bytes_per_launch": gu_bytes, "avg_launch_ms": gu_ms}
    else:
        achieved = gu_bytes / (gu_ms / 1e3) / 1e9
        roofline = {"kernel": "expert_gate_up", "bound": "hbm", "achieved": achieved,
                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / pk["hbm_gbs"],
                    "peak_source": "%s (MEASURED_PEAKS.json, copy)" % pk["source"],
                    "traffic": prof["dram_bytes_per_launch"] if prof else None,
                    "traffic_source": prof["source"] if prof else None,
                    "algorithmic_bytes_per_launch": gu_bytes, "avg_launch_ms": gu_ms}
    gemm_tflops = (gu_flops + dn_flops) / ((gu_ms + dn_ms) / 1e3) / 1e12
    extra = {
        "expert_gemms": {"tflops": gemm_tflops, "frac_of_burst_peak": gemm_tflops / tpeak,
                         "frac_of_sustained_peak": gemm_tflops / spk if spk else None,
                         "ms": gu_ms + dn_ms},
        "touched_experts": n_touched,
        "hbm_on_touched_weights": {
            "bytes_per_step": w_touched,
            "gbs_whole_step": w_touched / (ms_step / 1e3) / 1e9,
            "frac_whole_step": w_touched / (ms_step / 1e3) / 1e9 / pk["hbm_gbs"],
            "gbs_expert_gemms": w_touched / ((gu_ms + dn_ms) / 1e3) / 1e9,
            "frac_expert_gemms": w_touched / ((gu_ms + dn_ms) / 1e3) / 1e9 / pk["hbm_gbs"]},
    }
    launches = sum(n for n, _ in kern.values())
    layer_flops = cfg.flops(R)
    kernels = {k: {"launches": n, "ms_per_step": t / args.steps,
                   "share": t / max(sum(x for _, x in kern.values()), 1e-9)}
               for k, (n, t) in kern.items() if n}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "step_ms": dict(q, timed_region=ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) random-init weights)",
        "config": dict(run_config(cfg, cf, world),
                       **({"bias_update_gamma": args.bias_update}
                          if args.bias_update is not None else {})),
        "kept_rows": R,
        "tflops": world * layer_flops / (ms_step / 1e3) / 1e12,
        "roofline": roofline,
        "e2e": {"value": world * cfg.T * args.steps / (ms_e2e / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": X.numel() * X.element_size(),
                "d2h_bytes_per_step": Yh[0].numel() * Yh[0].element_size(),
                "how": "pinned host X -> device, forward, bf16 Y -> pinned host every step; "
                       "copies on two copy streams overlap the neighbouring steps' compute"},
        "gpu_launches": launches,
        **extra,
        "kernels": kernels,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        try:
            tr, tf, n, stage_s = cpu_baseline_sample(cfg, d, cf, args.cpu_tokens,
                                                     args.cpu_seconds)
        except Exception as exc:          # the GPU figures above still get printed
            line["cpu_baseline"] = {"value": None, "unit": "tokens/s", "kind": "oracle",
                                    "error": f"{type(exc).__name__}: {exc}"}
            print(json.dumps(line), flush=True)
            if dist is not None:
                dist.destroy_process_group()
            return
        v = cfg.T / (tr + tf * cfg.T / n)
        line["cpu_baseline"] = {
            "value": v, "unit": "tokens/s", "cores": blas_threads(), "nproc": host_cores(),
            "kind": "oracle",
            "sample": f"fp64 oracle: routing of all {cfg.T} tokens ({tr:.2f} s) + experts and "
                      + (f"combine of all {cfg.T} tokens ({tf:.2f} s)" if n >= cfg.T else
                         f"combine of {n} seeded tokens ({tf:.2f} s), extrapolated to "
                         f"{cfg.T} tokens")
                      + f"; expert weights widened to float64 one expert at a time outside "
                        f"the clock ({stage_s:.1f} s); the token sample starts at "
                        f"{min(args.cpu_tokens, cfg.T)} and doubles until the expert stage "
                        f"takes {args.cpu_seconds:g} s or covers the batch"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(K.BY_NAME))
    ap.add_argument("--capacity-factor", type=float, default=None)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=512,
                    help="first token sample of the cpu_baseline oracle (it doubles)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="grow the cpu_baseline sample until its expert stage takes this long")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="tokens per reference step (0: the largest that fits --ref-budget)")
    ap.add_argument("--ref-budget", type=float, default=150.0,
                    help="seconds the reference arm's warm-up and timed steps may take")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bias-update", type=float, default=None, metavar="GAMMA",
                    help="end every forward with the bias update step (selection bias "
                         "-/+ GAMMA for over/underloaded experts)")
    ap.add_argument("--fp8-experts", action="store_true",
                    help="expert weights as FP8 E4M3 codes with per-channel scales")
    ap.add_argument("--expert-choice", action="store_true",
                    help="expert-choice routing: every expert takes its C = T*k/E best tokens")
    ap.add_argument("--router-groups", default=None, metavar="G:M",
                    help="group-limited routing: G expert groups, M of them per token")
    ap.add_argument("--shape", default=None, metavar="T=..,E=..",
                    help="the workload's recipe at other sizes (T, H, E, I, k), for small "
                         "profiling cases; such a line is not a bench figure of the workload")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)     # fewer warm-up steps give no valid number
    cfg = K.BY_NAME[args.config]
    if args.shape:
        kw = {}
        for item in args.shape.split(","):
            key, _, val = item.partition("=")
            if key not in ("T", "H", "E", "I", "k") or not val.isdigit():
                ap.error(f"--shape takes T, H, E, I, k as KEY=integer, not {item!r}")
            kw[key] = int(val)
        cfg = K.scaled(cfg, name=f"{cfg.name}@{args.shape}", **kw)
    if args.bias_update is not None and cfg.selection_bias_std <= 0:
        ap.error("--bias-update needs a workload with a selection bias (sigmoid scoring)")
    if args.router_groups:
        G, M = (int(v) for v in args.router_groups.split(":"))
        cfg = dataclasses.replace(cfg, n_groups=G, topk_groups=M)
    if args.fp8_experts:
        if cfg.dtype != "bf16":
            ap.error("--fp8-experts needs a bf16 workload")
        cfg = dataclasses.replace(cfg, fp8_experts=True)
    if args.expert_choice:
        if args.router_groups or args.capacity_factor is not None or args.bias_update is not None:
            ap.error("--expert-choice takes no groups, capacity factor or bias update")
        cfg = dataclasses.replace(cfg, expert_choice=True, capacity_factors=())
    cf = args.capacity_factor
    if cf is None and cfg.capacity_factors:
        cf = cfg.capacity_factors[0]
    if args.impl == "reference":
        run_reference(args, cfg, cf)
    else:
        run_gpu(args, cfg, cf)


if __name__ == "__main__":
    main()
