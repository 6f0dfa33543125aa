"""Benchmark: forward pass of the Mixtral-shaped MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
    python bench.py --stage route|permute [--T T --H H --E E --k K]   (one stage alone)

A step is one whole layer forward (route -> permute -> GEMM0+SwiGLU ->
GEMM1+scatter -> combine) over one batch of T tokens, through the C ABI
(moe_layer_forward). Inputs are seeded synthetic bf16 tensors of the
configuration's shape, resident in HBM before timing. L2 is flushed (a
256 MiB write) between timed steps; each step is timed with one pair of CUDA
events on the launching stream and nothing recorded between its stages.
A second pass of the same steps, with the library recording an event before
every stage, gives the per-stage times and the GEMM0 roofline. Prints one JSON
line (rank 0).

Multi-GPU: the layer's tokens are independent, so N GPUs run N independent
replicas of the workload (weak scaling, no collective on the data path);
the barrier/max-over-ranks timing follows the launcher's contract.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the only place besides the cpu_baseline field where the benchmark
runs the oracle).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from token_dispatch_grouped_moe_gb300.configs import CONFIGS  # noqa: E402

METRIC = "MoE layer fwd bf16 TFLOP/s & tokens/s on 1 GB300; % of tensor peak / HBM BW"
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one GEMM0 launch, from a
# one-pass ncu capture of this benchmark at the configuration's full size of the kernel
# as it is now, keyed by (configuration, CTAs per MMA, who fills x_perm); kernels
# without such a capture report null. (The captures of earlier forms of the kernel are
# in the profile summaries.)
GEMM0_TRAFFIC = {
    # grouped_gemm_kernel<2, 1> (GEMM0 + SwiGLU, CTA pairs, dense x_perm tiles): 3049.9 MB read +
    # 462.7 MB written, profiles/launches_mixtral_layer.md
    ("mixtral", 2, "kernel"): 3_512_600_000,
}
L2_FLUSH_BYTES = 256 << 20


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest value over the ranks of the process group (the value itself
    on one rank): each rank times its own replica, the job takes the slowest."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_workload(cfg, device):
    import torch
    from token_dispatch_grouped_moe_gb300.inputs import make_inputs
    inp = make_inputs(cfg.T, cfg.H, cfg.F, cfg.E, Fs=cfg.Fs, seed=cfg.seed)
    return inp, {n: v.to(device) for n, v in inp.items()}


def roofline_stage_bytes(cfg):
    """Algorithmic bytes of the HBM-bound stages (per launch)."""
    T, H, E, k, R = cfg.T, cfg.H, cfg.E, cfg.k, cfg.R
    n_slots = k + (1 if cfg.Fs else 0)
    return {
        "route": T * H * 2 + H * E * 2 + T * k * 8,
        "combine": n_slots * T * H * 4 + T * H * 2,
        "permute_index": R * 4 * 4 + E * 8,
        # the dispatch with x_perm materialised, as the scope table defines it:
        # every routed row read from x and written to x_perm
        "permute": 2 * R * H * 2,
        # the least a dispatch can move: each token's row of x read once, each
        # routed row of x_perm written once, the index arrays (the token-side
        # copy moves about this; it reads x once where the rows are read k times
        # in the definition above, so that figure can exceed the copy bandwidth)
        "permute_min": T * H * 2 + R * H * 2 + R * 4 * 4,
    }


def cpu_baseline(cfg, inp, budget_s=15.0, max_tokens=None):
    """The oracle, as it stands, on a bounded sample of this workload's tokens."""
    from oracle.oracle import Oracle
    from token_dispatch_grouped_moe_gb300.inputs import bf16_bits
    O = Oracle()
    b = {n: bf16_bits(v) for n, v in inp.items()}
    flops_per_token = cfg.flops() / cfg.T

    def run(n):
        xs = b["x"][:n]
        t0 = time.perf_counter()
        _, idx, w = O.route(xs, b["Wg"], cfg.k)
        O.layer_rows(np.arange(n, dtype=np.int64), idx, w, xs, b["W1"], b["W3"], b["W2"],
                     b.get("W1s"), b.get("W3s"), b.get("W2s"))
        return time.perf_counter() - t0

    n = max(1, min(O.num_threads(), cfg.T))
    dt = run(n)
    # grow the sample to about budget_s of CPU work
    target = int(n * budget_s / max(dt, 1e-3))
    if max_tokens:
        target = min(target, max_tokens)
    target = max(n, min(cfg.T, target))
    if target > n:
        n = target
        dt = run(n)
    return {"value": n * flops_per_token / dt / 1e12, "unit": "TFLOP/s", "cores": O.num_threads(),
            "kind": "oracle", "tokens_per_s": n / dt,
            "sample": f"first {n} of {cfg.T} tokens of the {cfg.name} workload (route + FFN + combine)"}


def bench_ours(args, cfg):
    import torch
    from token_dispatch_grouped_moe_gb300 import build as cuda_build
    from token_dispatch_grouped_moe_gb300 import lib

    rank, world, local = dist_env()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if not os.path.exists(lib.LIB_PATH):
        cuda_build.build()
    lib.load()
    lib.set_combine({"auto": lib.COMBINE_AUTO, "fused": lib.COMBINE_FUSED,
                     "separate": lib.COMBINE_SEPARATE}[args.combine])
    lib.set_gemm_fusion({"auto": lib.GEMM_FUSION_AUTO, "on": lib.GEMM_FUSION_ON,
                         "off": lib.GEMM_FUSION_OFF}[args.gemm_fusion])
    lib.set_cta_group({"auto": lib.CTA_GROUP_AUTO, "one": lib.CTA_GROUP_ONE,
                       "pair": lib.CTA_GROUP_PAIR}[args.cta_group])
    lib.set_x_perm_copy({"auto": lib.X_PERM_COPY_AUTO, "inline": lib.X_PERM_COPY_INLINE,
                         "kernel": lib.X_PERM_COPY_KERNEL}[args.x_perm_copy])
    lib.set_router({"auto": lib.ROUTER_OPT_AUTO, "fma": lib.ROUTER_OPT_FMA,
                    "tensor": lib.ROUTER_OPT_TENSOR}[args.router])

    inp, g = make_workload(cfg, device)
    dims = lib.make_dims(cfg.T, cfg.H, cfg.F, cfg.E, cfg.k, cfg.Fs)
    plan = lib.layer_plan(dims)
    ws = lib.workspace(dims, device=device)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    names = ["before_route", "before_permute", "before_gemm0", "before_gemm1", "before_shared",
             "before_combine", "after_combine"]

    def new_events():
        # torch creates the CUDA event on its first record; record once so the
        # raw handle exists before the library records it between stages
        evs = [torch.cuda.Event(enable_timing=True) for _ in names]
        for e in evs:
            e.record(stream)
        se = lib.StageEvents(*[lib.ctypes.c_void_p(e.cuda_event) for e in evs])
        return evs, se

    def step(se=None):
        lib.layer_forward(dims, g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], ws, W1s=g.get("W1s"),
                          W3s=g.get("W3s"), W2s=g.get("W2s"), out=out, events=se)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if lib.check(ws) != lib.MOE_OK:
        raise RuntimeError("device error during warm-up")

    # the timed region: K layer calls, each bracketed by one pair of events on
    # the launching stream and nothing between its stages (an event recorded
    # between two kernels costs the second one its launch overlap, about 5 us)
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    launches0 = lib.launch_count()
    for i in range(args.steps):
        flush.fill_(1)
        step_evs[i][0].record(stream)
        step()
        step_evs[i][1].record(stream)
    launches = lib.launch_count() - launches0   # the library's own count of its kernels
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if lib.check(ws) != lib.MOE_OK:
        raise RuntimeError("device error during timing")
    step_ms = [e0.elapsed_time(e1) for e0, e1 in step_evs]
    ms = max_over_ranks(float(np.sum(step_ms)) / args.steps, device)

    # stage pass: the same K calls again, the library recording an event before
    # every stage: the per-stage times and the GEMM0 roofline come from here
    recs = [new_events() for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(1)
        step(recs[i][1])
    torch.cuda.synchronize()
    if lib.check(ws) != lib.MOE_OK:
        raise RuntimeError("device error during the stage pass")
    stage_ms = {n: [] for n in ("route", "permute", "gemm0", "gemm1", "shared", "combine")}
    for evs, _ in recs:
        t = [evs[0].elapsed_time(e) for e in evs]
        for j, n in enumerate(stage_ms):
            stage_ms[n].append(t[j + 1] - t[j])
    stage_step_ms = float(np.mean([evs[0].elapsed_time(evs[-1]) for evs, _ in recs]))

    # end to end through the C ABI with host buffers (moe_layer_forward_host):
    # x from pinned host memory, the layer, out back to pinned host memory,
    # the token chunks' copies overlapping the kernels
    x_host = inp["x"].pin_memory()
    out_host = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(g["x"])
    out_dev = torch.empty_like(g["x"])
    host_chunks = args.host_chunks if args.host_chunks > 0 else lib.host_chunks(dims)
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        lib.layer_forward_host(dims, x_host, g["Wg"], g["W1"], g["W3"], g["W2"], ws, x_dev, out_dev, out_host,
                               W1s=g.get("W1s"), W3s=g.get("W3s"), W2s=g.get("W2s"), n_chunks=host_chunks)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    if not torch.equal(out_dev, out):
        raise RuntimeError("the host-buffer call's output differs from the device call's")
    e2e = max_over_ranks(float(np.mean(e2e_ms)), device)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None

    peaks = measured_peaks()
    flops = cfg.flops()
    # the library runs both routed GEMMs as one launch below 512 rows per expert
    # (or when forced): then the gemm0 stage holds both and gemm1 is empty
    fused_gemms = plan.gemm_fusion == lib.GEMM_FUSION_ON
    gemm0_ms = float(np.mean(stage_ms["gemm0"]))
    gemm0_flops = 4 * cfg.R * cfg.H * cfg.F + (2 * cfg.R * cfg.F * cfg.H if fused_gemms else 0)
    achieved = gemm0_flops / (gemm0_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    stage_summary = {n: round(float(np.mean(v)), 4) for n, v in stage_ms.items()}
    by = roofline_stage_bytes(cfg)
    stage_roofline = {
        "gemm0": {"tflops": round(achieved, 1), "frac": round(achieved / peak, 4)},
        "route": {"gbs": round(by["route"] / (np.mean(stage_ms["route"]) * 1e-3) / 1e9, 1)},
    }
    if fused_gemms:
        stage_roofline["gemm0"]["includes"] = "GEMM0 + GEMM1 (one launch)"
        stage_roofline["gemm1"] = {"fused": "in the gemm0 launch", "tflops": None}
    else:
        stage_roofline["gemm1"] = {"tflops": round(2 * cfg.R * cfg.F * cfg.H /
                                                   (np.mean(stage_ms["gemm1"]) * 1e-3) / 1e12, 1)}
    if np.mean(stage_ms["combine"]) > 0.01:   # a separate combine kernel ran
        gbs = by["combine"] / (np.mean(stage_ms["combine"]) * 1e-3) / 1e9
        stage_roofline["combine"] = {"gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}
    else:
        stage_roofline["combine"] = {"fused": "done by the GEMM1 epilogue (last contribution)"}
    if not fused_gemms:
        stage_roofline["gemm1"]["frac"] = round(stage_roofline["gemm1"]["tflops"] / peak, 4)
    stage_roofline["route"]["frac"] = round(stage_roofline["route"]["gbs"] / peaks["hbm_gbs"], 4)
    if plan.x_perm_copy == lib.X_PERM_COPY_KERNEL:
        # index phases + the x_perm copy, against the copy's algorithmic bytes
        t_perm = np.mean(stage_ms["permute"]) * 1e-3
        gbs = by["permute"] / t_perm / 1e9
        gbs_min = by["permute_min"] / t_perm / 1e9
        stage_roofline["permute"] = {"gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                                     "bytes": "2*R*H*2 (routed rows read and written)",
                                     "min_bytes_gbs": round(gbs_min, 1),
                                     "min_bytes_frac": round(gbs_min / peaks["hbm_gbs"], 4)}

    value = world * flops / (ms * 1e-3) / 1e12
    fused = plan.combine == lib.COMBINE_FUSED
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "tokens_per_s": round(world * cfg.T / (ms * 1e-3), 1),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "step_ms_stats": {"median": round(float(np.median(step_ms)), 4), "min": round(float(np.min(step_ms)), 4),
                          "max": round(float(np.max(step_ms)), 4)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded randn: x sigma 1, weights sigma 0.02, bf16)",
        "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} F={cfg.F} E={cfg.E} top-{cfg.k}"
                               + (f" shared F={cfg.Fs}" if cfg.Fs else "") + " SwiGLU",
                   "T": cfg.T, "H": cfg.H, "F": cfg.F, "E": cfg.E, "k": cfg.k, "F_shared": cfg.Fs,
                   "l2": "flushed (256 MiB write) between timed steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor",
                     "kernel": "grouped GEMM0 + SwiGLU and GEMM1, one launch (tcgen05)" if fused_gemms
                     else "grouped GEMM0 + SwiGLU (tcgen05" + (", CTA pairs)" if plan.cta_group == 2
                                                              else ")"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": None if fused_gemms else GEMM0_TRAFFIC.get(
                         (cfg.name, plan.cta_group, {1: "inline", 2: "kernel"}.get(plan.x_perm_copy))),
                     "traffic_unit": "bytes per launch",
                     "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"},
        "timing": {"value": "K layer calls, one event pair each, no events between stages",
                   "stage_ms": "a second pass of K calls with an event before every stage",
                   "stage_pass_ms_per_step": round(stage_step_ms, 4)},
        "router": {0: "stream", 1: "sliced", 2: "cluster", 3: "block", 4: "tensor"}.get(plan.router),
        "gemm_plan": {"cta_group": plan.cta_group, "cta_group_gemm1": plan.cta_group_gemm1,
                      "tile": [plan.tile_m, plan.tile_n, plan.tile_k],
                      "stages": plan.stages, "one_launch": fused_gemms, "combine_fused": fused,
                      "x_perm_copy": {1: "inline", 2: "kernel"}.get(plan.x_perm_copy)},
        "stage_ms": stage_summary,
        "stage_roofline": stage_roofline,
        "e2e": {"value": round(world * flops / (e2e * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e, 4), "h2d_bytes_per_step": cfg.T * cfg.H * 2,
                "d2h_bytes_per_step": cfg.T * cfg.H * 2, "call": "moe_layer_forward_host",
                "chunks": host_chunks},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, budget_s=args.cpu_budget)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


def bench_reference(args, cfg):
    """The oracle (CPU) as the reference arm: each step is a bounded sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    from oracle.oracle import Oracle
    from token_dispatch_grouped_moe_gb300.inputs import bf16_bits, make_inputs
    O = Oracle()
    inp = make_inputs(cfg.T, cfg.H, cfg.F, cfg.E, Fs=cfg.Fs, seed=cfg.seed)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    n_tok = max(1, min(cfg.T, args.ref_tokens))
    flops_per_token = cfg.flops() / cfg.T

    def step(i):
        lo = (i * n_tok) % cfg.T
        xs = b["x"][lo:lo + n_tok]
        _, idx, w = O.route(xs, b["Wg"], cfg.k)
        O.layer_rows(np.arange(xs.shape[0], dtype=np.int64), idx, w, xs, b["W1"], b["W3"], b["W2"],
                     b.get("W1s"), b.get("W3s"), b.get("W2s"))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = (time.perf_counter() - t0) / args.steps
    value = n_tok * flops_per_token / dt / 1e12
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "tokens_per_s": round(n_tok / dt, 3),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 FFN / f32 routing (CPU oracle)",
        "data": "synthetic (seeded randn: x sigma 1, weights sigma 0.02, bf16)",
        "config": {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} F={cfg.F} E={cfg.E} top-{cfg.k}",
                   "T": cfg.T, "H": cfg.H, "F": cfg.F, "E": cfg.E, "k": cfg.k, "F_shared": cfg.Fs},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": O.num_threads(),
                         "kind": "oracle",
                         "sample": f"{n_tok} of {cfg.T} tokens per step of the {cfg.name} workload"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }



def bench_stage(args):
    """One stage through the C ABI at any shape (--T --H --E --k), outside the
    layer call: `route` (moe_route; T*H*2 + H*E*2 + T*k*8 bytes) or `permute`
    (moe_permute with x_perm; 2*T*k*H*2 bytes: the routed rows read and written,
    and, as min_bytes, T*H*2 + T*k*H*2 + T*k*16: x read once, x_perm written, the
    index arrays). Before every timed call L2 is
    emptied of the inputs by writing and then reading a 256 MiB buffer (the
    read leaves L2 holding clean lines, so the timed call pays no write-back
    of the flush); each call is timed with CUDA events on the current stream.
    Prints one JSON line with the median."""
    import torch
    from token_dispatch_grouped_moe_gb300 import build as cuda_build
    from token_dispatch_grouped_moe_gb300 import lib
    from token_dispatch_grouped_moe_gb300.inputs import make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("--stage needs a GPU")
    if not os.path.exists(lib.LIB_PATH):
        cuda_build.build()
    lib.load()
    dev = torch.device("cuda")
    T, H, E, k = args.T, args.H, args.E, args.k
    inp = make_inputs(T, H, 64, E, seed=0, only=("x", "Wg"))
    x, Wg = inp["x"].to(dev), inp["Wg"].to(dev)
    dims = lib.make_dims(T, H, 64, E, k)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ws = None
    if args.stage == "permute":
        ws = lib.workspace(dims, device=dev)
        lib.route(dims, x, Wg, topk_idx=idx, topk_w=w)

    def call():
        if args.stage == "route":
            lib.route(dims, x, Wg, topk_idx=idx, topk_w=w)
        else:
            lib.permute(dims, idx, ws, x=x, want_x_perm=True)

    times = []
    for i in range(args.warmup + args.steps):
        flush.fill_(1)
        flush.view(torch.float32).sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) * 1e-3)
    if ws is not None and lib.check(ws) != lib.MOE_OK:
        raise RuntimeError("device error in the stage calls")
    t = float(np.median(times))
    work = T * H * 2 + H * E * 2 + T * k * 8 if args.stage == "route" else 2 * T * k * H * 2
    work_min = None if args.stage == "route" else T * H * 2 + T * k * H * 2 + T * k * 4 * 4
    peaks = measured_peaks()
    gbs = work / t / 1e9
    line = {"stage": args.stage, "config": {"T": T, "H": H, "E": E, "k": k},
            "us_median": round(t * 1e6, 2), "us_min": round(min(times) * 1e6, 2),
            "algorithmic_bytes": work, "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
            "peak_source": f"{peaks['source']} HBM copy bandwidth (MEASURED_PEAKS.json)",
            "steps": args.steps, "warmup": args.warmup}
    if work_min is not None:
        line.update(min_bytes=work_min, min_bytes_gbs=round(work_min / t / 1e9, 1),
                    min_bytes_frac=round(work_min / t / 1e9 / peaks["hbm_gbs"], 4))
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="mixtral", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--combine", default="auto", choices=["auto", "fused", "separate"],
                    help="where the layer sums the expert rows (GEMM1 epilogue or a separate kernel)")
    ap.add_argument("--gemm-fusion", default="auto", choices=["auto", "on", "off"],
                    help="both routed GEMMs in one persistent launch, or two launches")
    ap.add_argument("--cta-group", default="auto", choices=["auto", "one", "pair"],
                    help="CTAs per tensor-core MMA in the dense-A expert GEMMs")
    ap.add_argument("--x-perm-copy", default="auto", choices=["auto", "inline", "kernel"],
                    help="x_perm filled inside GEMM0 while it runs, or by a kernel before it")
    ap.add_argument("--router", default="auto", choices=["auto", "fma", "tensor"],
                    help="the router kernels: the table's choice, the FMA routers, or the tensor-core router")
    ap.add_argument("--host-chunks", type=int, default=0,
                    help="token chunks of the end-to-end host-buffer call (0: the library's choice)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--ref-tokens", type=int, default=64, help="oracle tokens per reference step")
    ap.add_argument("--stage", choices=["route", "permute"], default=None,
                    help="time one stage alone at the shape --T --H --E --k instead of the layer")
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--E", type=int, default=8)
    ap.add_argument("--k", type=int, default=2)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    if args.stage:
        print(json.dumps(bench_stage(args)), flush=True)
        return
    cfg = CONFIGS[args.config]
    line = bench_reference(args, cfg) if args.impl == "reference" else bench_ours(args, cfg)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
