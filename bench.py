"""Benchmark of the routed MoE layer forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload nano_decode|nano_prefill|latent|nvfp4_prefill|
                                nano_decode_fp8|nano_prefill_fp8|tiny]

One step = one whole layer forward (route, permute, grouped expert FFN, combine; the
LatentMoE workload adds its two projections) over one batch of seeded synthetic tokens,
through the library's C ABI. Prints one JSON line.

The default workload is the Nano-shaped prefill layer: 16384 tokens (two 8192-token
sequences), H=2688, 128 experts, top-6, F=1856, with a Zipf-skewed selection bias; it is
the largest single-GPU configuration of the 128-expert, top-6, bf16 layer. nano_decode is
the 64-token decode layer. The NVFP4 prefill workload quantises the expert weights once, untimed, and
runs moe_forward_nvfp4 (activation quantisation included in every step); the *_fp8
workloads do the same with per-tensor E4M3 experts (moe_forward_fp8). Inputs and
weights are resident in HBM before the timed region starts. L2 is
flushed before every timed step: a 512 MiB write, then a 256 MiB read, so that the write's
dirty lines are written back before the step starts rather than inside it. Each step is timed with CUDA events on
the launching stream; the grouped expert FFN, the dominant kernel, is timed the same way.

"e2e" is the same layer through the C ABI with the input coming from pinned host memory
and the output going back to it every step. The steps are pipelined as a serving loop runs
them: step i+1's input copy and step i-1's output copy overlap step i's compute, on their
own streams with two device buffers each. This loop does not flush L2 (the flush would be
inside the timed stream); every workload streams more than L2 per step.

The CPU-baseline leg times the fp64 oracle on all host cores (one thread per core) on a
bounded random sample of the same workload's tokens. The same leg reports the run's parity
("parity"): the oracle's routing of every token with the near-ties (gap < 1e-5) counted, and
the sampled tokens' output errors against this run's GPU output.

--impl reference times the fp64 CPU oracle on the host's cores, on a bounded sample of the
same workload, and prints the same line with "impl": "reference".

Under torchrun (N > 1) each rank runs an independent replica of the layer on its own GPU.
The layer shards by tokens with no exchange. There is no data-path collective: ranks only
meet at the timing barriers and the max-over-ranks of the elapsed time.
"""
from __future__ import annotations

import argparse
import ctypes
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

import moe_synth  # noqa: E402

METRIC = "MoE-layer tokens/s and % of roofline (128 experts top-6, bf16) on 1 B300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# Dense FP4 tensor rate relative to BF16 on B300 (nominal 13.5 vs 2.25 PFLOP/s): the FP4
# peak is the measured BF16 peak times this ratio.
FP4_OVER_BF16 = 13.5 / 2.25
FP8_OVER_BF16 = 4.5 / 2.25
L2_FLUSH_BYTES = 512 << 20
L2_EVICT_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(values, device, world: int):
    """Element-wise maximum of per-rank timings (ms) over all ranks; unchanged on one rank.
    Replicas run the same workload, so the slowest rank sets the job's time."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput of `world` replicas that each process tokens_per_rank tokens per
    step, timed by the slowest rank."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# ------------------------------------------------------------------- algorithmic counts ----

def counts_from_routing(idx: np.ndarray, E: int) -> np.ndarray:
    return np.bincount(idx.reshape(-1), minlength=E)


def layer_algorithmic(w: moe_synth.Workload, counts: np.ndarray) -> dict:
    """FLOPs and bytes the method must do/move (weights touched + layer input/output)."""
    D, rows = w.D, w.rows
    touched = int((counts > 0).sum())
    f_router = 2.0 * w.T * (w.latent if (w.latent and w.router_on_latent) else w.H) * w.E
    f_experts = 4.0 * rows * D * w.F
    f_proj = 4.0 * w.T * w.H * w.latent if w.latent else 0.0
    # bf16 weights: 2 bytes per element; NVFP4: half a byte of code plus one E4M3 scale per
    # 16 elements
    w_bytes = (0.5 + 1.0 / 16) if w.nvfp4 else (1.0 if w.fp8 else 2.0)
    b_weights = touched * 2.0 * D * w.F * w_bytes
    b_router = w.E * (D if (w.latent and w.router_on_latent) else w.H) * 2.0
    b_proj = 2.0 * w.H * w.latent * 2 if w.latent else 0.0
    b_io = 2.0 * w.T * w.H * 2
    # per expert-GEMM launch (up and down alike): one expert matrix per touched expert, plus
    # the routed activations read (bf16, E4M3, or NVFP4 codes and scales) and written (bf16)
    a_in = (0.5 + 1.0 / 16) if w.nvfp4 else (1.0 if w.fp8 else 2.0)
    ffn_bytes_per_launch = touched * D * w.F * w_bytes + rows * (D + w.F) * (a_in + 2.0) / 2
    return {"flops": f_router + f_experts + f_proj, "bytes": b_weights + b_router + b_proj + b_io,
            "flops_router": f_router, "flops_experts": f_experts, "flops_proj": f_proj,
            "touched": touched, "ffn_flops_per_launch": 2.0 * rows * D * w.F,
            "ffn_bytes_per_launch": ffn_bytes_per_launch}


def kernels_per_step(w: moe_synth.Workload, gathered: bool = False,
                     fused_combine: bool = False) -> int:
    """Library kernels one timed step launches (memsets excluded), mirroring the C library's
    choices: the fused small-batch routing kernel (T <= 256, E <= 256, routing width <= 6144)
    or router logits + top-k + permutation (one small-batch block, or mark/count/scan, then
    the map writer / row copy). With gathered (moe_forward_gathered) the up-projection
    gathers its token rows itself, so the fused routing needs no separate row copy."""
    T, E, k = w.T, w.E, w.k
    d_route = (w.latent * (3 if w.router_on_latent else 0) or w.H) if w.latent else w.H
    fused = T <= 256 and E <= 256 and d_route <= 6144 and k <= 32
    words = (T + 31) // 32
    perm = 1 if (words <= 64 and words * E <= 8192) else 3
    # routing: one fused kernel, or logits, top-k, the permutation and its map writer
    route_q = 1 if fused else 2 + perm + 1
    if w.nvfp4:   # routing, amax x, pad, quantise x, zero the padding rows, up,
        return route_q + 8   # quantise h, down, combine
    if w.fp8:     # routing, amax x, quantise x, up, quantise h, down, combine
        return route_q + 6
    gather_in_gemm = gathered
    if fused:
        route = 1 if gather_in_gemm else 2     # + the row copy
    else:
        route = 2 + perm + 1                   # + the map writer (and row copy)
    if w.latent:  # projection in, routing in the latent space, FFN, combine, projection out
        return 1 + route + 2 + 1 + 1
    if fused_combine:  # zero the fixed-point sums, FFN (combine in the epilogue), convert
        return route + 1 + 2 + 1
    return route + 2 + 1


# ------------------------------------------------------------------------ clock sampler ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.t0 = self.t1 = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "25"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        for ts, line in self.lines:
            if self.t0 is not None and not (self.t0 - 0.05 <= ts <= (self.t1 or ts) + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------ ours (GPU) ----

def run_ours(args, w: moe_synth.Workload):
    import torch
    import torch.distributed as dist

    import sparse_mixture_experts_57_b300 as moe

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = moe.lib()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    inp = moe_synth.layer_inputs(w)
    d = {k: moe_synth.to_torch(v, dev) for k, v in inp.items()}
    T, H, E, k, F, D = w.T, w.H, w.E, w.k, w.F, w.D
    rows = T * k
    P = lambda t: t.data_ptr()  # noqa: E731

    # device buffers
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, k), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    evict = torch.ones(L2_EVICT_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # the write leaves up to L2's size of dirty lines; the read replaces them with clean
        # lines of another buffer, so their write-back to HBM happens here, untimed
        flush.zero_()
        evict.sum()

    def chk(code, what):
        if code != 0:
            raise moe.MoeError(code, what)

    # Every workload runs as its whole-layer C call, the call a user makes. The expert GEMMs,
    # the dominant kernels, are timed inside it with the library's profiling hook, which
    # records caller-owned events around the up- and down-projection GEMMs on the stream.
    if w.latent:
        ws = torch.empty(L.latent_moe_workspace_size(T, H, w.latent, E, k, F,
                                                     int(w.router_on_latent)),
                         dtype=torch.uint8, device=dev)

        def layer_call(xp, yp, ip, gp):
            chk(L.latent_moe(xp, P(d["w_in"]), P(d["w_out"]), P(d["w_router"]), P(d["bias"]),
                             int(w.router_on_latent), P(d["w_up"]), P(d["w_down"]), T, H,
                             w.latent, E, k, F, yp, ip, gp, P(ws), ws.numel(), sp), "latent_moe")
    elif w.fp8:
        # weight quantisation is a set-up step, outside the timed region
        f8_up = moe.moe_quantize_fp8_weights(d["w_up"])
        f8_down = moe.moe_quantize_fp8_weights(d["w_down"])
        del d["w_up"], d["w_down"]
        ws = torch.empty(L.moe_forward_fp8_workspace_size(T, H, E, k, F), dtype=torch.uint8,
                         device=dev)

        def layer_call(xp, yp, ip, gp):
            chk(L.moe_forward_fp8(xp, P(d["w_router"]), P(d["bias"]), *f8_up.ptrs(),
                                  *f8_down.ptrs(), T, H, E, k, F, yp, ip, gp, P(ws), ws.numel(),
                                  sp), "moe_forward_fp8")
    elif w.nvfp4:
        # weight quantisation is a set-up step, outside the timed region
        nv_up = moe.moe_quantize_nvfp4_weights(d["w_up"])
        nv_down = moe.moe_quantize_nvfp4_weights(d["w_down"])
        del d["w_up"], d["w_down"]
        ws = torch.empty(L.moe_forward_nvfp4_workspace_size(T, H, E, k, F), dtype=torch.uint8,
                         device=dev)

        def layer_call(xp, yp, ip, gp):
            chk(L.moe_forward_nvfp4(xp, P(d["w_router"]), P(d["bias"]), *nv_up.ptrs(),
                                    *nv_down.ptrs(), T, H, E, k, F, yp, ip, gp, P(ws),
                                    ws.numel(), sp), "moe_forward_nvfp4")
    else:
        # the standard bf16 layer: moe_forward, or one of its opt-in forms
        fwd_name = ("moe_forward_gathered" if args.gathered else
                    "moe_forward_fused_combine" if args.fused_combine else "moe_forward")
        size_fn = (L.moe_forward_fused_combine_workspace_size if args.fused_combine
                   else L.moe_forward_workspace_size)
        ws = torch.empty(size_fn(T, H, E, k, F), dtype=torch.uint8, device=dev)
        fwd_fn = getattr(L, fwd_name)

        def layer_call(xp, yp, ip, gp):
            chk(fwd_fn(xp, P(d["w_router"]), P(d["bias"]), P(d["w_up"]), P(d["w_down"]), T, H,
                       E, k, F, yp, ip, gp, P(ws), ws.numel(), sp), fwd_name)

    call_name = ("latent_moe" if w.latent else "moe_forward_fp8" if w.fp8 else
                 "moe_forward_nvfp4" if w.nvfp4 else fwd_name)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def hook_events(n):
        """n groups of the 4 profiling events, created (recorded once) so that their CUDA
        handles exist."""
        groups = [[ev() for _ in range(4)] for _ in range(n)]
        for g in groups:
            for e in g:
                e.record(stream)
        return groups

    def step(evs=None):
        if evs is not None:
            handles = (ctypes.c_void_p * 4)(*[e.cuda_event for e in evs])
            chk(L.moe_set_profile_events(handles, 4), "moe_set_profile_events")
        layer_call(P(d["x"]), P(y), P(idx), P(gates))
        if evs is not None:
            chk(L.moe_set_profile_events(None, 0), "moe_set_profile_events")

    # kernels per step: route 2, permutation 2-4, FFN 2, combine 1 (bf16); the latent layer
    # adds its two projections; the NVFP4 layer replaces the gather by amax, padding,
    # two quantisations and the two block-scaled GEMMs
    launches_per_step = kernels_per_step(w, args.gathered, args.fused_combine)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)

    K = args.steps
    s_ev = [ev() for _ in range(K)]
    e_ev = [ev() for _ in range(K)]
    g_ev = hook_events(K)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("t0")
    wall0 = time.perf_counter()
    for i in range(K):
        flush_l2()
        s_ev[i].record(stream)
        step(g_ev[i])
        e_ev[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks.mark("t1")
    time.sleep(0.25)
    clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(s_ev, e_ev)]
    # the dominant kernels: the up- and down-projection GEMMs, each bracketed by the hook
    up_ms = [g[0].elapsed_time(g[1]) for g in g_ev]
    down_ms = [g[2].elapsed_time(g[3]) for g in g_ev]
    ffn_ms = [a + b for a, b in zip(up_ms, down_ms)]
    # phases of a step: before the up-projection GEMM, from its start to the end of the
    # down-projection GEMM, after it
    phase_ms = {"before_up_gemm": statistics.mean(s.elapsed_time(g[0]) for s, g in zip(s_ev, g_ev)),
                "up_gemm": statistics.mean(up_ms),
                "between_gemms": statistics.mean(g[1].elapsed_time(g[2]) for g in g_ev),
                "down_gemm": statistics.mean(down_ms),
                "after_down_gemm": statistics.mean(g[3].elapsed_time(e) for g, e in zip(g_ev, e_ev))}
    ms = statistics.mean(step_ms)
    ffn = statistics.mean(ffn_ms)
    ms, ffn = max_over_ranks([ms, ffn], dev, world)
    assert moe.get_device_status() == 0

    # ---- end to end through the C ABI: pinned host x in, host y out, every step. Steps are
    # pipelined as a serving loop would run them: step i+1's input copy (host -> device) and
    # step i-1's output copy (device -> host) run on their own streams while step i computes,
    # with two device buffers for each; every step still moves its own input and output.
    # No L2 flush here: a flush would sit inside the timed stream. Every workload moves
    # 0.9 GB or more through HBM per step (expert weights, routed activations), several times
    # L2, so a step finds at most the last ~100 MB its predecessor touched.
    x_host = d["x"].cpu().pin_memory()
    y_host = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(d["x"]) for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [ev(), ev()]
    ev_comp = [ev(), ev()]
    ev_out = [ev(), ev()]
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            if started[b]:
                h2d.wait_event(ev_comp[b])       # step i-2 has finished reading x_dev[b]
            x_dev[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(h2d)
        stream.wait_event(ev_in[b])
        if started[b]:
            stream.wait_event(ev_out[b])         # step i-2's output has left y_dev[b]
        layer_call(P(x_dev[b]), P(y_dev[b]), None, None)
        ev_comp[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_comp[b])
            y_host[b].copy_(y_dev[b], non_blocking=True)
            ev_out[b].record(d2h)
        started[b] = True

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    t_a, t_b = ev(), ev()
    t_a.record(h2d)
    for i in range(args.warmup, args.warmup + K):
        e2e_step(i)
    d2h.wait_event(ev_comp[(args.warmup + K - 1) % 2])
    t_b.record(d2h)
    torch.cuda.synchronize()
    e2e = t_a.elapsed_time(t_b) / K
    e2e = max_over_ranks([e2e], dev, world)[0]
    assert moe.get_device_status() == 0

    routing = idx.cpu().numpy()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    clk = clocks.summary()
    # The dense tensor peak: the burst figure for kernels timed in a run that kept its
    # clocks, the sustained one (a seconds-long GEMM loop under the power cap) for kernels
    # timed inside a long run whose clocks the power cap brought down.
    capped = ("sw_power_cap" in clk["reasons"] and clk["sm_mhz"] is not None and
              clk["sm_mhz"] < 0.95 * clk["sm_max_mhz"])
    p_bf16 = peaks["bf16_tflops_sustained"] if capped else peaks["bf16_tflops"]
    bf16_src = (f"{peak_src} bf16 sustained (the run was power-capped)" if capped
                else f"{peak_src} bf16 burst")
    alg = layer_algorithmic(w, counts_from_routing(routing, E))
    launches = 2  # the up- and down-projection GEMMs, each bracketed by the hook
    p_fp4 = p_bf16 * FP4_OVER_BF16
    p_fp8 = p_bf16 * FP8_OVER_BF16
    p_tensor = p_fp4 if w.nvfp4 else (p_fp8 if w.fp8 else p_bf16)
    gemm_flops = alg["ffn_flops_per_launch"] * launches
    gemm_bytes = alg["ffn_bytes_per_launch"] * launches
    if gemm_flops / p_tensor / 1e12 >= gemm_bytes / peaks["hbm_gbs"] / 1e9:
        bound = "tensor"
        achieved = gemm_flops / (ffn / 1e3) / 1e12
        peak = p_tensor
        unit = "TFLOP/s"
    else:
        bound = "hbm"
        achieved = gemm_bytes / (ffn / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    if w.nvfp4 or w.fp8:
        t_flops = (alg["flops_experts"] / (p_fp4 if w.nvfp4 else p_fp8) +
                   (alg["flops_router"] + alg["flops_proj"]) / p_bf16) / 1e12
    else:
        t_flops = alg["flops"] / (p_bf16 * 1e12)
    roof_ms = max(t_flops, alg["bytes"] / (peaks["hbm_gbs"] * 1e9)) * 1e3
    traffic = None if (args.gathered or args.fused_combine) else \
        read_traffic(w.name, alg["touched"])
    out = {
        "metric": METRIC,
        "value": job_tokens_per_s(world, T, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("nvfp4 experts, bf16 router" if w.nvfp4 else
                  "e4m3 experts (per-tensor scales), bf16 router" if w.fp8 else "bf16"),
        "data": "synthetic (seeded, random-init weights of the named shape)",
        "config": {"workload": w.name, "T": T, "H": H, "E": E, "k": k, "F": F,
                   "latent": w.latent or None, "bias": w.bias,
                   "l2": "flushed before every step (512 MiB write, then 256 MiB read)",
                   "layer_call": call_name,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic,
                     "traffic_source": ("dram__bytes_read.sum + dram__bytes_write.sum per launch "
                                        "from the committed ncu summary of this kernel source "
                                        "(profiles/), not measured in this run")
                     if traffic is not None else None,
                     "kernel": ("expert up- and down-projection GEMMs ("
                                + ("block-scaled NVFP4 tcgen05" if w.nvfp4 else
                                   "E4M3 tcgen05" if w.fp8 else "bf16 tcgen05")
                                + (", the down-projection adding into the fixed-point sums"
                                   if args.fused_combine else "")
                                + (", the up-projection gathering token rows"
                                   if args.gathered else "")
                                + f"), timed inside {call_name} by moe_set_profile_events"),
                     "peak_source": (f"{bf16_src} x {FP4_OVER_BF16:g} (nominal FP4/BF16)"
                                     if (w.nvfp4 and bound == "tensor") else
                                     f"{bf16_src} x {FP8_OVER_BF16:g} (nominal FP8/BF16)"
                                     if (w.fp8 and bound == "tensor") else
                                     bf16_src if bound == "tensor" else f"{peak_src} copy"),
                     "frac_of_burst": (achieved / (peaks["bf16_tflops"] * p_tensor / p_bf16)
                                       if bound == "tensor" else achieved / peak),
                     "ffn_ms": ffn, "launches_timed": launches},
        "layer_roofline": {"time_ms": roof_ms, "frac": roof_ms / ms,
                           "tflops": alg["flops"] / (ms / 1e3) / 1e12,
                           "hbm_gbs": alg["bytes"] / (ms / 1e3) / 1e9,
                           "touched_experts": alg["touched"],
                           "peak_source": f"{bf16_src}; {peak_src} copy"},
        "e2e": {"value": job_tokens_per_s(world, T, e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "ms_per_step": e2e, "pipelined": "input copy of step i+1 and output copy "
                "of step i-1 overlap step i", "l2": "not flushed; each step streams more "
                "than L2"},
        "gpu_launches": launches_per_step * K,
        "phase_ms": phase_ms,
        "clocks": clk,
        "wall_s": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        # the CPU-baseline leg: the oracle timed on the host cores; its sample, and the
        # oracle's routing of every token, also give this run's parity numbers (untimed)
        out["cpu_baseline"], sample = cpu_baseline(w, inp, budget_s=args.cpu_budget)
        out["parity"] = parity_report(w, inp, moe_synth.from_torch_bf16(y), routing, sample)
    if world > 1:
        dist.destroy_process_group()
    return out


def read_traffic(workload: str, units: int):
    """DRAM bytes per grouped-GEMM launch from the committed ncu summary, if it still
    describes the current kernel source (else null). The summary gives either bytes per
    launch measured on this workload's full-size launches, or bytes per unit (touched
    expert matrix), in which case a launch moves `units` of them."""
    if "[" in workload:          # scaled cases have no committed counters
        return None
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_{workload}.md")
    try:
        with open(path) as f:
            txt = f.read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        if line.startswith("traffic_bytes_per_unit:"):
            vals["t"] = float(line.split(":", 1)[1])
        if line.startswith("traffic_bytes_per_launch:"):
            vals["l"] = float(line.split(":", 1)[1])
        if line.startswith("kernel_source_sha256:"):
            vals["h"] = line.split(":", 1)[1].strip()
    if vals.get("h") != kernel_source_hash():
        return None
    if "l" in vals:                # measured on this workload's full-size launches
        return vals["l"]
    return vals["t"] * units if "t" in vals else None


def kernel_source_hash() -> str:
    import hashlib
    p = os.path.join(ROOT, "sparse_mixture_experts_57_b300", "csrc")
    h = hashlib.sha256()
    for name in ("grouped_gemm.cu", "grouped_gemm_2sm.cu", "tc.cuh", "tc2.cuh"):
        with open(os.path.join(p, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ------------------------------------------------------------------- oracle (CPU) legs ----

def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_sample(w, inp, toks):
    """The oracle's layer on a subset of tokens: route them, run their experts, combine.
    Returns (output rows, the oracle's routing of those tokens)."""
    from oracle import moe_oracle as O
    x = inp["x"][toks]
    if w.latent:
        x_lat = O.latent_project_in(x, inp["w_in"])
        r = O.route(x_lat if w.router_on_latent else x, inp["w_router"], inp["bias"], w.k)
        y_lat = O.moe_tokens(x_lat, r["idx"], r["gates"], inp["w_up"], inp["w_down"])
        return y_lat @ O.widen_bf16(inp["w_out"]).T, r
    r = O.route(x, inp["w_router"], inp["bias"], w.k)
    if w.nvfp4:
        # the sample's own hidden amax stands in for the tensor-wide one: same per-token work
        return O.moe_tokens_nvfp4(inp["x"], x, r["idx"], r["gates"], inp["w_up"],
                                  inp["w_down"]), r
    if w.fp8:
        h_amax = O.fp8_hidden_amax(x, r["idx"], inp["w_up"])     # over the sample
        return O.moe_tokens_fp8(inp["x"], x, r["idx"], r["gates"], inp["w_up"], inp["w_down"],
                                h_amax), r
    return O.moe_tokens(x, r["idx"], r["gates"], inp["w_up"], inp["w_down"]), r


class _BlasThreads:
    """Context manager that sets the BLAS thread count of numpy's OpenBLAS for its duration
    (threadpoolctl when installed, else OpenBLAS's own setter found among the loaded
    libraries; without either it does nothing)."""

    def __init__(self, n: int):
        self.n, self.ctx, self.setter, self.prev = n, None, None, None

    @staticmethod
    def _openblas():
        import ctypes
        try:
            with open("/proc/self/maps") as f:
                paths = {ln.split()[-1] for ln in f if "openblas" in ln.lower() and "/" in ln}
        except OSError:
            return None, None
        for path in sorted(paths):
            try:
                lib = ctypes.CDLL(path)
            except OSError:
                continue
            for pre in ("scipy_", ""):
                for suf in ("64_", ""):
                    set_fn = getattr(lib, f"{pre}openblas_set_num_threads{suf}", None)
                    get_fn = getattr(lib, f"{pre}openblas_get_num_threads{suf}", None)
                    if set_fn is not None and get_fn is not None:
                        return set_fn, get_fn
        return None, None

    def __enter__(self):
        try:
            from threadpoolctl import threadpool_limits
            self.ctx = threadpool_limits(self.n)
            self.ctx.__enter__()
            return self
        except ImportError:
            pass
        set_fn, get_fn = self._openblas()
        if set_fn is not None:
            self.prev = int(get_fn())
            set_fn(self.n)
            self.setter = set_fn
        return self

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)
        elif self.setter is not None:
            self.setter(self.prev)
        return False


class OraclePool:
    """The oracle run on all host cores: one thread per core, each evaluating its own chunk
    of tokens with single-threaded BLAS (numpy releases the GIL in its array kernels)."""

    def __init__(self, w, inp, threads=None):
        import concurrent.futures as cf
        self.w, self.inp = w, inp
        self.threads = threads or _host_cores()
        self.ex = cf.ThreadPoolExecutor(self.threads)

    def run(self, chunks):
        """Evaluate the token chunks concurrently; returns ([(toks, y, routing)], wall s)."""
        with _BlasThreads(1):
            t0 = time.perf_counter()
            res = list(self.ex.map(lambda t: (t, *_oracle_sample(self.w, self.inp, t)), chunks))
            return res, time.perf_counter() - t0

    def close(self):
        self.ex.shutdown()


def _chunks(rng, T, n_chunks, per_chunk):
    toks = np.sort(rng.choice(T, min(T, n_chunks * per_chunk), replace=False))
    return [toks[i::n_chunks] for i in range(n_chunks) if toks[i::n_chunks].size]


def cpu_baseline(w, inp, budget_s=20.0):
    """Time the oracle as it stands on a bounded sample of the workload, on all host cores.
    Returns (the cpu_baseline object, the sampled tokens' oracle outputs and routing)."""
    rng = np.random.default_rng(123)
    pool = OraclePool(w, inp)
    per = 2
    done, t_total, sample = 0, 0.0, []
    try:
        while True:
            res, dt = pool.run(_chunks(rng, w.T, pool.threads, per))
            t_total += dt
            sample += res
            done += sum(len(t) for t, _, _ in res)
            if t_total >= budget_s or done >= w.T:
                break
    finally:
        pool.close()
    base = {"value": done / t_total, "unit": "tokens/s", "cores": pool.threads, "kind": "oracle",
            "sample": f"{done} of {w.T} tokens (random, {per} per thread per round, "
                      f"{pool.threads} threads with single-threaded BLAS), fp64 numpy oracle: "
                      f"route, expert FFNs of the chosen experts, combine; {t_total:.1f} s wall",
            "cpu_model": _cpu_model()}
    return base, sample


def parity_report(w, inp, y_gpu, idx_gpu, sample) -> dict:
    """Agreement of this run's GPU outputs with the oracle (not timed): the oracle's routing
    of every token (near-ties counted), and the relative Frobenius / max-abs errors of the
    sampled tokens' outputs (the CPU baseline's own sample)."""
    from oracle import moe_oracle as O
    tie_gap = 1e-5
    if w.latent:
        x_lat = O.latent_project_in(inp["x"], inp["w_in"])
        r = O.route(x_lat if w.router_on_latent else inp["x"], inp["w_router"], inp["bias"], w.k)
    else:
        r = O.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    same = (np.sort(idx_gpu, axis=1) == np.sort(r["idx"], axis=1)).all(axis=1)
    near = r["gap"] < tie_gap
    out = {"oracle": "fp64 numpy", "tokens": int(w.T), "near_tie_gap": tie_gap,
           "near_tie_count": int(near.sum()),
           "selection_differs_near_tie": int((~same & near).sum()),
           "selection_differs_non_tie": int((~same & ~near).sum())}
    if w.nvfp4 or w.fp8:
        out["outputs"] = ("not compared here: the oracle needs the tensor-wide amax of h, "
                          "i.e. the whole layer; the tests compare sampled tokens with it")
        return out
    toks = np.concatenate([t for t, _, _ in sample])
    ref = np.concatenate([y for _, y, _ in sample])
    keep = same[toks]
    got = O.widen_bf16(y_gpu[toks[keep]])
    ref = ref[keep]
    err = got - ref
    rms = float(np.sqrt(np.mean(ref * ref)))
    out.update({"sampled_tokens": int(keep.sum()),
                "rel_frob": float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)),
                "maxabs_over_rms": float(np.abs(err).max() / max(rms, 1e-30)),
                "tolerance": {"rel_frob": 1e-2, "maxabs_over_rms": 3e-2}})
    return out


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    inp = moe_synth.layer_inputs(w)
    rng = np.random.default_rng(7)
    pool = OraclePool(w, inp)
    per = 1
    try:
        for _ in range(args.warmup):
            pool.run(_chunks(rng, w.T, pool.threads, per))
        times, n = [], 0
        for _ in range(args.steps):
            res, dt = pool.run(_chunks(rng, w.T, pool.threads, per))
            n = sum(len(t) for t, _, _ in res)
            times.append(dt)
    finally:
        pool.close()
    ms = statistics.mean(times) * 1e3
    value = n / (ms / 1e3)
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "F": w.F,
                       "latent": w.latent or None, "bias": w.bias},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": pool.threads,
                             "kind": "oracle",
                             "sample": f"{n} random tokens of {w.T} per step ({per} per thread, "
                                       f"{pool.threads} threads) through the fp64 oracle",
                             "cpu_model": _cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="nano_prefill",
                    choices=list(moe_synth.WORKLOADS))
    ap.add_argument("--T", type=int, default=None,
                    help="override the token count (a scaled case, e.g. for profiling)")
    ap.add_argument("--E", type=int, default=None,
                    help="override the expert count (E, or E' of the latent layer; scaled case)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--gathered", action="store_true",
                    help="standard layer: time moe_forward_gathered (whole-layer bracket)")
    ap.add_argument("--fused-combine", action="store_true",
                    help="standard layer: time moe_forward_fused_combine (whole-layer bracket)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = moe_synth.WORKLOADS[args.workload]
    if (args.gathered or args.fused_combine) and (w.latent or w.nvfp4 or w.fp8):
        ap.error("--gathered and --fused-combine apply to the bf16 standard layer")
    if args.gathered and args.fused_combine:
        ap.error("--gathered and --fused-combine select different entry points")
    if args.T is not None or args.E is not None:
        import dataclasses
        T = args.T if args.T is not None else w.T
        E = args.E if args.E is not None else w.E
        w = dataclasses.replace(w, T=T, E=E, name=f"{w.name}[T={T},E={E}]")
    if args.steps is None:
        # enough steps for about two seconds of timed work (clock samples land inside it)
        args.steps = {"nano_decode": 2000, "nano_decode_fp8": 2000, "tiny": 2000}.get(w.name, 500) \
            if args.impl == "ours" else 5
    args.warmup = max(3, args.warmup) if args.impl == "ours" else args.warmup
    out = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
