"""Benchmark of the NVFP4 W4A4 MoE expert forward on GB300.

One step = one pass of the whole expert path (scale check, token reorder,
a1 quantisation, w13 GEMM + SiLU*up + a2 quantisation, w2 GEMM + weighted
combine) over one batch: the prefill-shaped layer of 8192 tokens, 128
experts, hidden 2816, intermediate 704, top-8 with Zipf(1.1) routing.  Inputs
are synthetic and seeded; weights are N(0, 0.02) BF16 draws quantised to NVFP4
on the device.  Prints one JSON line (rank 0).

The throughput comes from K timed steps of the plain forward; the per-kernel
split (and the roofline's kernel time) from a second timed region of K steps
that records an event around every kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle on a bounded sample of the same
workload (the reference arm).  Under torchrun (N > 1) each rank runs an
independent replica of the layer on its own GPU (the path has no exchange
step); value = tokens of all ranks / max rank time.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import inputs as S  # noqa: E402

METRIC = "NVFP4 MoE layer tokens/s; quant GB/s and expert-GEMM FP4 TFLOPS vs GB300 peak"
WORKLOAD = ("prefill MoE layer: 8192 tokens, 128 experts, hidden 2816, intermediate 704, top-8, "
            "Zipf(1.1) routing with 8 idle experts")
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio on GB300
# kernels one layer step launches: scale check, token reorder, a1 quantiser, w13 GEMM, w2 GEMM
LAUNCHES_PER_STEP = 5

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the two GEMM kernels
# on the 8192-token prefill layer, from one ncu capture of the two GEMM kernels with those two
# counters.  It holds for the kernel source it was taken on: any change to these files makes it null.
NCU_TRAFFIC = {
    "tokens": 8192,
    "source_sha1": {"nvfp4_w4a4_moe_gb300/csrc/kernels_gemm.cu": "ee89b1bd0b301a010b6a6b5ed745514ab4f0a956",
                    "nvfp4_w4a4_moe_gb300/csrc/tc_common.cuh": "a2ee1d30e584fa75518c2785c3cd69d7ddb8da35",
                    "nvfp4_w4a4_moe_gb300/csrc/common.cuh": "0428d7d24646c64d83c1960a2dc5b0380bbe36ed"},
    "bytes": {"gemm_w13": 394253312 + 103216640, "gemm_w2": 278187264 + 64749312},
}


def measured_traffic(kernel: str, tokens: int):
    """The ncu DRAM bytes per launch of `kernel`, or None when there is no
    capture for it, for this token count, or for the current kernel source."""
    import hashlib
    if tokens != NCU_TRAFFIC["tokens"] or kernel not in NCU_TRAFFIC["bytes"]:
        return None
    root = os.path.dirname(os.path.abspath(__file__))
    for rel, digest in NCU_TRAFFIC["source_sha1"].items():
        try:
            with open(os.path.join(root, rel), "rb") as f:
                if hashlib.sha1(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return NCU_TRAFFIC["bytes"][kernel]


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        p.update({k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in d})
        p["source"] = "measured"
    return p


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 20 ms) around the timed region; each sample is
    stamped on arrival, and the summary keeps those between mark_start() and
    mark_end() (all of them if none fell inside)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []  # (arrival time, line)
        self.t_start = self.t_end = None

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        inside = [ln for t, ln in self.lines
                  if self.t_start is not None and self.t_end is not None and self.t_start <= t <= self.t_end]
        for ln in inside or [ln for _, ln in self.lines]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": len(inside)}


class NvmlClockSampler:
    """In-process, read-only NVML queries (SM clock, its maximum, and the
    clock-event reasons) every `period_s` from a thread, stamped on arrival,
    so that a timed region of a few milliseconds holds several samples.  No
    setting of the GPU is changed.  `ok` is False when libnvidia-ml cannot be
    loaded or the device is not found; the caller then falls back to
    nvidia-smi."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid: str | None, period_s: float = 0.001):
        import ctypes
        self.period = period_s
        self.samples = []  # (time, sm_mhz, max_mhz, reason bits)
        self.t_start = self.t_end = None
        self.ok = False
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = (lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) if uuid
                  else lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)))
            if rc != 0:
                return
            self.lib, self.h, self.ct = lib, h, ctypes
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = reasons or lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _query(self):
        c = self.ct
        sm, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, c.byref(mx))
        self.reasons_fn(self.h, c.byref(rs))
        return (time.monotonic(), sm.value, mx.value, rs.value)

    def _run(self):
        while not self._stop.is_set():
            q = self._query()
            if q:
                self.samples.append(q)
            time.sleep(self.period)

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def __enter__(self):
        if self.ok:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
            time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        if self.ok:
            time.sleep(0.02)
            self._stop.set()
            self.thread.join(timeout=5)
        return False

    def summary(self):
        inside = [q for q in self.samples
                  if self.t_start is not None and self.t_end is not None and self.t_start <= q[0] <= self.t_end]
        use = inside or self.samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({name for q in use for bit, name in self.REASONS.items() if q[3] & bit})
        return {"sm_mhz": statistics.median(q[1] for q in use), "sm_max_mhz": max(q[2] for q in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "source": f"NVML, in process, every {self.period * 1e3:g} ms"}


def clock_sampler(uuid: str | None):
    """NVML in process when available, else nvidia-smi."""
    s = NvmlClockSampler(uuid)
    return s if s.ok else ClockSampler(uuid)


# --------------------------------------------------------------------------- workload
def make_layer_device(layer, m, torch, seed: int, ue8m0: bool = False):
    """Device weights: N(0, 0.02) BF16 draws quantised on the device (UE8M0
    block scales with ue8m0)."""
    E, H, I = layer.E, layer.H, layer.I
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    w13 = (torch.randn((E, 2 * I, H), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    w2 = (torch.randn((E, H, I), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    q13, sf13, s13 = m.quantize_weights(w13, ue8m0=ue8m0)
    q2, sf2, s2 = m.quantize_weights(w2, ue8m0=ue8m0)
    in13 = torch.from_numpy(layer.w13_input_scale).cuda()
    w = m.MoEWeights(E, H, I, q13, sf13, s13, in13, q2, sf2, s2, torch.ones(E, device="cuda"),
                     sf_format=m.SF_UE8M0 if ue8m0 else m.SF_E4M3)
    return w, (w13, w2)


def calibrate_w2_on_device(m, torch, w, x, ids, tw, layer):
    """w2 input scale = amax of SiLU(gate)*up per expert / 2688, from one
    forward that keeps h (calibration stand-in; outside the timed region)."""
    T, k, E, I = layer.T, layer.k, layer.E, layer.I
    _, ws = m.moe_forward(w, x, ids, tw, flags=m.DEBUG_KEEP_H | m.SYNC_CHECK)
    it = m.intermediates_of(ws, T, layer.H, I, E, k)
    pad = it["pad_offsets"].cpu().numpy()
    counts = np.diff(np.concatenate([[0], np.bincount(layer.topk_ids.ravel(), minlength=E).cumsum()]))
    h = it["h"]
    amax = np.zeros(E, np.float32)
    for e in range(E):
        if counts[e]:
            amax[e] = float(h[pad[e]:pad[e] + counts[e]].abs().max())
    amax[amax == 0] = amax.max()
    w.w2_input_scale = torch.from_numpy(S.input_scale_from_amax(amax)).cuda()
    del ws


def algorithmic(layer, n_active):
    """Algorithmic bytes / FLOPs per launch of each stage (minimum traffic)."""
    T, H, I, k, E = layer.T, layer.H, layer.I, layer.k, layer.E
    R = T * k
    fp4 = 0.5 + 1.0 / 16.0  # bytes per element: packed code + its share of a scale byte
    return {
        "validate": {"bytes": 4 * 4 * E},
        "route": {"bytes": R * 4 * 3 + R * 4},
        "quant_a1": {"bytes": T * H * 2 + R * H * fp4 + R * 4 * 2},
        "gemm_w13": {"bytes": R * H * fp4 + n_active * 2 * I * H * fp4 + R * I * fp4,
                     "flops": 2.0 * R * 2 * I * H},
        "gemm_w2": {"bytes": R * I * fp4 + n_active * H * I * fp4 + T * H * 4, "flops": 2.0 * R * H * I},
    }


def combine_ranks(total_ms: float, tokens_per_rank: int, steps: int, dist=None):
    """Replicas: every rank times its own K steps between barriers; the job's
    time is the slowest rank's, and its throughput counts every rank's tokens.
    Returns (ms per step, tokens/s).  Works on NCCL (GPU tensors) and gloo."""
    world = 1
    if dist is not None:
        import torch
        world = dist.get_world_size()
        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_step = total_ms / steps
    return ms_step, tokens_per_rank * world / (ms_step * 1e-3)


def run_ours(args, rank, world):
    import torch

    import nvfp4_w4a4_moe_gb300 as m

    m.load()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    layer = S.prefill(args.tokens)
    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.k
    w, _bf16 = make_layer_device(layer, m, torch, seed=1003 + 17 * rank)
    x = torch.from_numpy(layer.x.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(layer.topk_ids).cuda()
    tw = torch.from_numpy(layer.topk_w).cuda()
    calibrate_w2_on_device(m, torch, w, x, ids, tw, layer)
    del _bf16
    m.prepare_weights(w)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    flags = m.SCALES_PREVALIDATED
    stream = torch.cuda.current_stream()

    # one checked call first: scale check with the host sync, device status clean
    m.moe_forward(w, x, ids, tw, out=out, ws=ws, flags=m.SYNC_CHECK)

    K, W = args.steps, args.warmup
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for _ in range(W):
        m.moe_forward(w, x, ids, tw, out=out, ws=ws, flags=flags)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(0).uuid)
    except Exception:
        uuid = None
    # Two timed regions of K steps each.  The first runs the layer as a user
    # does and gives the throughput; the second records six events per step
    # (before and after every kernel) for the per-kernel times, which the
    # records themselves lengthen by about 2 us each, so it does not set value.
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pstart, pstop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clock_sampler(uuid if rank == 0 else None) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clocks.mark_start()
        start.record(stream)
        for i in range(K):
            m.moe_forward(w, x, ids, tw, out=out, ws=ws, flags=flags)
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        pstart.record(stream)
        for i in range(K):
            m.moe_forward_profiled(w, x, ids, tw, evs[i], out=out, ws=ws, flags=flags)
        pstop.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        if dist:
            dist.barrier()
    total_ms = start.elapsed_time(stop)
    status, _ = m.moe_status(ws)
    if status != m.OK:
        raise RuntimeError(f"device status {status} after the timed steps")
    ms_step, value = combine_ranks(total_ms, T, K, dist)
    ms_step_profiled = pstart.elapsed_time(pstop) / K
    stage_ms = {name: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) / K
                for j, name in enumerate(m.STAGES)}

    if args.only_w4a16:
        res = w4a16_leg(m, torch, w, layer, x, ids, tw, args)
        return {"metric": METRIC, "value": res["prefill"]["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
                "config": {"T": T, "path": "w4a16"}, "w4a16": res, "note": "W4A16 only (profiling run)"}

    if args.only_layer:
        return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": K, "warmup": W, "ms_per_step": ms_step, "config": {"T": T},
                "kernels": {n: {"ms": v} for n, v in stage_ms.items()}, "note": "layer only (profiling run)"}

    # host-checked step (scale check synchronised on the host), for reference
    t0 = time.perf_counter()
    for _ in range(5):
        m.moe_forward(w, x, ids, tw, out=out, ws=ws, flags=0)
    torch.cuda.synchronize()
    ms_checked = (time.perf_counter() - t0) * 1e3 / 5

    # quantiser workload: 4096 tokens x 2816, uniform top-8, 1% outliers x50
    qres = quant_workload(m, torch, w, args)

    # e2e: host buffers in, host buffers out, through the host entry point
    e2e = e2e_host(m, torch, w, layer, args)
    decode = decode_leg(m, torch, w, args)
    router = router_leg(m, torch, args)
    ue8m0 = ue8m0_leg(m, torch, args)
    w4a16 = w4a16_leg(m, torch, w, layer, x, ids, tw, args)
    stack = stack_leg(m, torch, args) if not args.no_stack else None

    pk = peaks()
    n_active = int((np.bincount(layer.topk_ids.ravel(), minlength=E) > 0).sum())
    alg = algorithmic(layer, n_active)
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    dom = max(stage_ms, key=stage_ms.get)
    a = alg[dom]
    t_s = stage_ms[dom] * 1e-3
    if "flops" in a and a["flops"] / (fp4_peak * 1e12) > a["bytes"] / (pk["hbm_gbs"] * 1e9):
        roof = {"bound": "tensor", "achieved": a["flops"] / t_s / 1e12, "peak": fp4_peak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": a["bytes"] / t_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(dom, T)
    roof["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    roof["kernel"] = dom
    roof["peak_source"] = (f"{pk['source']} HBM copy" if roof["bound"] == "hbm" else
                           f"{pk['source']} bf16 burst x {FP4_OVER_BF16:g} (nominal FP4:BF16)")

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 e2m1 x e2m1 (e4m3 block scales), fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T, "E": E, "H": H, "I": I, "k": k,
                   "routed_rows": T * k, "active_experts": n_active,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (0.43 GB of weights + 0.2 GB activations per step)",
                   "scale_check": "device-side each step; host sync skipped in the timed steps",
                   "ms_per_step_with_host_scale_check": ms_checked},
        "roofline": roof,
        "kernels": {n: {"ms": v, "share": v / sum(stage_ms.values()),
                        "algorithmic_bytes": alg[n]["bytes"],
                        "gbs": alg[n]["bytes"] / (v * 1e-3) / 1e9,
                        "frac_hbm": alg[n]["bytes"] / (v * 1e-3) / 1e9 / pk["hbm_gbs"]}
                    for n, v in stage_ms.items()},
        "kernels_note": (f"per-kernel CUDA-event times from a second timed region of {K} steps with six "
                         f"events per step ({ms_step_profiled:.4f} ms per step there, against "
                         f"{ms_step:.4f} ms without the events)"),
        "gemm": {
            "w13_tflops": alg["gemm_w13"]["flops"] / (stage_ms["gemm_w13"] * 1e-3) / 1e12,
            "w2_tflops": alg["gemm_w2"]["flops"] / (stage_ms["gemm_w2"] * 1e-3) / 1e12,
            "fp4_peak_tflops": fp4_peak,
            "w13_frac_fp4_peak": alg["gemm_w13"]["flops"] / (stage_ms["gemm_w13"] * 1e-3) / 1e12 / fp4_peak,
            "w2_frac_fp4_peak": alg["gemm_w2"]["flops"] / (stage_ms["gemm_w2"] * 1e-3) / 1e12 / fp4_peak,
        },
        "quant": qres,
        "decode": decode,
        "router": router,
        "ue8m0": ue8m0,
        "w4a16": w4a16,
        "stack": stack,
        "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
        line["cpu_baseline"]["oracle_timings"] = oracle_timings(args)
    if dist:
        dist.destroy_process_group()
    return line


def quant_workload(m, torch, w, args):
    """The activation quantiser on the quantiser workload (4096 x 2816, 128
    experts, uniform top-8, input_scale = U(0.5,2) amax/2688), timed as the
    a1-quantiser stage of the expert path."""
    L = S.quantiser()
    T, H, E, k = L.T, L.H, L.E, L.k
    x = torch.from_numpy(L.x.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(L.topk_ids).cuda()
    tw = torch.from_numpy(L.topk_w).cuda()
    wq = m.MoEWeights(E, H, w.I, w.w13_q, w.w13_sf, w.w13_scale2, torch.from_numpy(L.w13_input_scale).cuda(),
                      w.w2_q, w.w2_sf, w.w2_scale2, w.w2_input_scale)
    wq.prepared = w.prepared
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.moe_workspace_size(T, H, w.I, E, k), dtype=torch.uint8, device="cuda")
    m.moe_forward(wq, x, ids, tw, out=out, ws=ws, flags=m.SYNC_CHECK)
    n = max(20, args.steps // 2)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
    for i in range(n):
        m.moe_forward_profiled(wq, x, ids, tw, evs[i], out=out, ws=ws, flags=m.SCALES_PREVALIDATED)
    torch.cuda.synchronize()
    ms = sum(evs[i][2].elapsed_time(evs[i][3]) for i in range(n)) / n  # the a1-quantiser stage
    R = T * k
    nbytes = T * H * 2 + R * H * (0.5 + 1 / 16) + R * 8
    pk = peaks()
    return {"workload": "4096 tokens x 2816, 128 experts, uniform top-8, 1% outliers x50",
            "ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "note": "bytes = x read once + codes and scales written + routing reads"}


# about 25 ms at the SM clock: longer than the host takes to issue 500 graph replays
REPLAY_QUEUE_SPIN_CYCLES = 50_000_000


def decode_leg(m, torch, w, args):
    """The decode-shaped layers (same experts, 1-64 tokens): latency per call
    of the plain forward, of a CUDA-graph replay of one call (replays queued
    on the GPU; also as paced by the host's launches), and per call
    inside a graph of ten back-to-back calls (as in a captured multi-layer
    decode step, where one call's first kernel overlaps the previous call's
    tail), tokens/s, and the bandwidth over the weight bytes of the experts
    the batch touches (codes + block scales of w13 and w2).  A replayed call
    finds the weights it touched in L2 (26.8 MB at one token), so one more
    figure takes the calls of a graph over eight copies of the weights at
    other addresses (3.4 GB), as in a decode step through eight layers: each
    call's weights come from HBM."""
    H, I, E = w.H, w.I, w.E
    per_expert = 2 * I * H // 2 + 2 * I * H // 16 + H * I // 2 + H * I // 16
    copies = [(w.w13_q.clone(), w.w2_q.clone(), w.prepared.clone()) for _ in range(8)]
    res = {}
    for T in (1, 8, 32, 64):
        L = S.decode(T)
        k = L.k
        x = torch.from_numpy(L.x.view(np.int16)).cuda().view(torch.bfloat16)
        ids = torch.from_numpy(L.topk_ids).cuda()
        tw = torch.from_numpy(L.topk_w).cuda()
        wd = m.MoEWeights(E, H, I, w.w13_q, w.w13_sf, w.w13_scale2, torch.from_numpy(L.w13_input_scale).cuda(),
                          w.w2_q, w.w2_sf, w.w2_scale2, w.w2_input_scale)
        wd.prepared = w.prepared
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        ws = torch.empty(m.moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
        m.moe_forward(wd, x, ids, tw, out=out, ws=ws, flags=m.SYNC_CHECK)
        n = 500
        flags = m.SCALES_PREVALIDATED
        for _ in range(20):
            m.moe_forward(wd, x, ids, tw, out=out, ws=ws, flags=flags)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(n):
            m.moe_forward(wd, x, ids, tw, out=out, ws=ws, flags=flags)
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / n * 1e3
        graph_us, graph_err, graph10_us, copies_us, graph_host_paced_us = None, None, None, None, None
        try:
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                m.moe_forward(wd, x, ids, tw, out=out, ws=ws, flags=flags)
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s):
                    m.moe_forward(wd, x, ids, tw, out=out, ws=ws, flags=flags, stream=s)
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(20):
                g.replay()
            torch.cuda.synchronize()
            # replays issued back to back from the host: at one token the host's
            # graph launches (about 20 us each on this machine) pace the GPU
            a.record()
            for _ in range(n):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            graph_host_paced_us = a.elapsed_time(b) / n * 1e3
            # the same replays queued behind a spin kernel, so that the GPU runs
            # them back to back: the device time of one replay
            torch.cuda._sleep(REPLAY_QUEUE_SPIN_CYCLES)
            a.record()
            for _ in range(n):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            graph_us = a.elapsed_time(b) / n * 1e3
            st, _ = m.moe_status(ws)
            if st != m.OK:
                graph_us, graph_err = None, f"device status {st} after graph replays"
            # ten calls captured in one graph: the steady per-call time
            g10 = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g10, stream=s):
                    for _ in range(10):
                        m.moe_forward(wd, x, ids, tw, out=out, ws=ws, flags=flags, stream=s)
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(3):
                g10.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(n // 10):
                g10.replay()
            b.record()
            torch.cuda.synchronize()
            graph10_us = a.elapsed_time(b) / (n // 10 * 10) * 1e3
            # one call per weight copy in one graph
            wcs = []
            for w13q, w2q, prep in copies:
                wc = m.MoEWeights(E, H, I, w13q, w.w13_sf, w.w13_scale2, wd.w13_input_scale, w2q, w.w2_sf,
                                  w.w2_scale2, w.w2_input_scale)
                wc.prepared = prep
                wcs.append(wc)
            g8 = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g8, stream=s):
                    for wc in wcs:
                        m.moe_forward(wc, x, ids, tw, out=out, ws=ws, flags=flags, stream=s)
            torch.cuda.current_stream().wait_stream(s)
            for _ in range(3):
                g8.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(n // 8):
                g8.replay()
            b.record()
            torch.cuda.synchronize()
            copies_us = a.elapsed_time(b) / (n // 8 * 8) * 1e3
            st, _ = m.moe_status(ws)
            if st != m.OK:
                copies_us, graph_err = None, f"device status {st} after the weight-copy graph"
        except Exception as ex:  # capture support depends on the driver; report, do not fail the run
            graph_err = f"{type(ex).__name__}: {ex}"[:200]
        touched = len(np.unique(L.topk_ids))
        best = graph_us if graph_us is not None else us
        res[str(T)] = {"us_per_call": us, "us_per_graph_replay": graph_us,
                       "us_per_graph_replay_host_paced": graph_host_paced_us,
                       "us_per_call_in_graph_of_10": graph10_us,
                       "us_per_call_over_8_weight_copies": copies_us, "graph_error": graph_err,
                       "tokens_per_s": T / (best * 1e-6), "experts_touched": touched,
                       "weight_gbs": touched * per_expert / (best * 1e-6) / 1e9}
    return res


def w4a16_leg(m, torch, w, layer, x, ids, tw, args):
    """The W4A16 path (NVFP4 weights, BF16 activations, kind::f16 tensor
    cores) on the same prefill layer and on the decode shapes: time per call
    (CUDA events around back-to-back calls; decode also from a CUDA graph),
    tokens/s, the GEMMs' BF16 TFLOP/s against the measured BF16 peak, and the
    decode weight bandwidth over the touched experts' codes and scales."""
    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.k
    m.prepare_weights_w4a16(w)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.moe_w4a16_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    m.moe_forward_w4a16(w, x, ids, tw, out=out, ws=ws, flags=m.SYNC_CHECK)
    flags = m.SCALES_PREVALIDATED
    for _ in range(3):
        m.moe_forward_w4a16(w, x, ids, tw, out=out, ws=ws, flags=flags)
    n = 20
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(n):
        m.moe_forward_w4a16(w, x, ids, tw, out=out, ws=ws, flags=flags)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    status, _ = m.moe_status(ws)
    if status != m.OK:
        raise RuntimeError(f"W4A16 device status {status}")
    flops = 6.0 * T * k * H * I  # gate/up (2 x 2I x H) + down (2 x H x I) per routed row
    pk = peaks()
    res = {"prefill": {"T": T, "ms_per_call": ms, "tokens_per_s": T / (ms * 1e-3),
                       "layer_tflops": flops / (ms * 1e-3) / 1e12,
                       "frac_bf16_peak": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                       "note": "whole call (scale check, reorder, row gather, both GEMMs) against the BF16 burst peak"}}
    per_expert = 2 * I * H // 2 + 2 * I * H // 16 + H * I // 2 + H * I // 16
    dec = {}
    for Td in (1, 64):
        L = S.decode(Td)
        xd = torch.from_numpy(L.x.view(np.int16)).cuda().view(torch.bfloat16)
        idd, twd = torch.from_numpy(L.topk_ids).cuda(), torch.from_numpy(L.topk_w).cuda()
        od = torch.empty((Td, H), dtype=torch.float32, device="cuda")
        wsd = torch.empty(m.moe_w4a16_workspace_size(Td, H, I, E, L.k), dtype=torch.uint8, device="cuda")
        m.moe_forward_w4a16(w, xd, idd, twd, out=od, ws=wsd, flags=m.SYNC_CHECK)
        for _ in range(20):
            m.moe_forward_w4a16(w, xd, idd, twd, out=od, ws=wsd, flags=flags)
        nd = 300
        torch.cuda.synchronize()
        a.record()
        for _ in range(nd):
            m.moe_forward_w4a16(w, xd, idd, twd, out=od, ws=wsd, flags=flags)
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / nd * 1e3
        graph_us, graph_err = None, None
        try:
            g = torch.cuda.CUDAGraph()
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                with torch.cuda.graph(g, stream=st):
                    m.moe_forward_w4a16(w, xd, idd, twd, out=od, ws=wsd, flags=flags, stream=st)
            torch.cuda.current_stream().wait_stream(st)
            for _ in range(20):
                g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(nd):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            graph_us = a.elapsed_time(b) / nd * 1e3
        except Exception as ex:  # capture support depends on the driver; report, do not fail the run
            graph_err = f"{type(ex).__name__}: {ex}"[:200]
        touched = len(np.unique(L.topk_ids))
        best = graph_us if graph_us is not None else us
        dec[str(Td)] = {"us_per_call": us, "us_per_graph_replay": graph_us, "graph_error": graph_err,
                        "experts_touched": touched, "weight_gbs": touched * per_expert / (best * 1e-6) / 1e9}
    res["decode"] = dec
    return res


def ue8m0_leg(m, torch, args):
    """The activation quantiser with E4M3 and with UE8M0 block scales on the
    quantiser workload (4096 x 2816, 128 experts, uniform top-8), through the
    stand-alone entry point: each call runs the scale check (with its host
    synchronisation), the token reorder and the quantiser, so the difference
    between the two is the quantiser's."""
    L = S.quantiser()
    x = torch.from_numpy(L.x.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(L.topk_ids).cuda()
    scale = torch.from_numpy(L.w13_input_scale).cuda()
    ws = torch.empty(m.quantize_workspace_size(L.T, L.k, L.E), dtype=torch.uint8, device="cuda")
    res = {}
    for name, fmt in (("e4m3", 0), ("ue8m0", m.SF_UE8M0)):
        layout = m.SF_SWIZZLED | fmt
        for _ in range(5):
            m.quantize_experts(x, ids, scale, L.E, sf_layout=layout, ws=ws)
        n = 50
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            m.quantize_experts(x, ids, scale, L.E, sf_layout=layout, ws=ws)
        torch.cuda.synchronize()
        res[name] = {"us_per_call": (time.perf_counter() - t0) / n * 1e6}
    out = {"workload": "4096 tokens x 2816, 128 experts, uniform top-8", "calls": res,
           "note": "synchronous calls: scale check + token reorder + quantiser each"}

    # the prefill layer with UE8M0 block scales on the weights, a1 and a2
    layer = S.prefill(args.tokens)
    wu, bf = make_layer_device(layer, m, torch, seed=1003, ue8m0=True)
    del bf
    xl = torch.from_numpy(layer.x.view(np.int16)).cuda().view(torch.bfloat16)
    idl = torch.from_numpy(layer.topk_ids).cuda()
    twl = torch.from_numpy(layer.topk_w).cuda()
    calibrate_w2_on_device(m, torch, wu, xl, idl, twl, layer)
    outl = torch.empty((layer.T, layer.H), device="cuda")
    wsl = torch.empty(m.moe_workspace_size(layer.T, layer.H, layer.I, layer.E, layer.k), dtype=torch.uint8,
                      device="cuda")
    m.moe_forward(wu, xl, idl, twl, out=outl, ws=wsl, flags=m.SYNC_CHECK)
    for _ in range(5):
        m.moe_forward(wu, xl, idl, twl, out=outl, ws=wsl, flags=m.SCALES_PREVALIDATED)
    n = 50
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(n):
        m.moe_forward(wu, xl, idl, twl, out=outl, ws=wsl, flags=m.SCALES_PREVALIDATED)
    e.record()
    torch.cuda.synchronize()
    st, _ = m.moe_status(wsl)
    ms = s.elapsed_time(e) / n
    out["prefill_layer"] = {"T": layer.T, "ms_per_call": ms, "tokens_per_s": layer.T / (ms * 1e-3), "status": st,
                            "note": "UE8M0 block scales throughout (weights, a1, a2), carried to the tensor "
                                    "cores as E4M3 powers of two relative to each operand row's largest"}
    del wu, outl, wsl
    return out


def router_leg(m, torch, args):
    """The router (softmax / top-k / renormalise) on N(0,1) FP32 logits of the
    layer's shape (128 experts, top-8), at the prefill and the decode token
    counts.  Two times per launch: back-to-back calls through the binding
    (host-bound at small sizes), and launches replayed from a CUDA graph of
    50 launches (the device's own time per launch).  Bandwidth is over the
    router's bytes (logits read, ids and weights written); the logits (4 MB
    at 8192 tokens) stay in L2 between launches, so it is a latency figure."""
    E, k = 128, 8
    per_graph, reps = 50, 10
    res = {}
    for T in (args.tokens, 64, 1):
        lg = torch.from_numpy(np.random.default_rng([7100, T]).standard_normal((T, E)).astype(np.float32)).cuda()
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        for _ in range(20):
            m.router_topk(lg, k, ids, tw)
        n = 500
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(n):
            m.router_topk(lg, k, ids, tw)
        b.record()
        torch.cuda.synchronize()
        us_call = a.elapsed_time(b) / n * 1e3
        us_graph, graph_err = None, None
        try:
            g = torch.cuda.CUDAGraph()
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                with torch.cuda.graph(g, stream=st):
                    for _ in range(per_graph):
                        m.router_topk(lg, k, ids, tw, stream=st)
            torch.cuda.current_stream().wait_stream(st)
            g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            us_graph = a.elapsed_time(b) / (reps * per_graph) * 1e3
        except Exception as ex:  # capture support depends on the driver; report, do not fail the run
            graph_err = f"{type(ex).__name__}: {ex}"[:200]
        nbytes = T * E * 4 + T * k * 8
        best = us_graph if us_graph is not None else us_call
        res[str(T)] = {"us_per_call": us_call, "us_per_launch_in_graph": us_graph, "graph_error": graph_err,
                       "bytes": nbytes, "gbs": nbytes / (best * 1e-6) / 1e9}
    return {"E": E, "k": k, "logits": "fp32 ~N(0,1)", "tokens": res,
            "note": "not part of the timed step: the step's routing is an input of the expert path"}


def e2e_host(m, torch, w, layer, args):
    T, H, k = layer.T, layer.H, layer.k
    xh = torch.from_numpy(layer.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ih = torch.from_numpy(layer.topk_ids).pin_memory()
    wh = torch.from_numpy(layer.topk_w).pin_memory()
    oh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    ws = torch.empty(m.moe_host_workspace_size(T, H, w.I, w.E, k), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        m.moe_forward_host(w, xh, ih, wh, out_host=oh, ws=ws, flags=m.SCALES_PREVALIDATED)
    n = max(10, args.steps // 10)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(n):
        m.moe_forward_host(w, xh, ih, wh, out_host=oh, ws=ws, flags=m.SCALES_PREVALIDATED)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    return {"value": T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": T * H * 2 + T * k * 8, "d2h_bytes_per_step": T * H * 4,
            "entry_point": "nvfp4_moe_forward_host (pinned host buffers)"}


# --------------------------------------------------------------------------- oracle arm
def oracle_sample_setup(n_tokens: int):
    """The oracle's inputs for a bounded sample of the prefill workload: the
    first n_tokens tokens, oracle-quantised weights of the experts they use
    (same N(0, 0.02) distribution, the generator's own draws), and a fixed
    w2 input scale (the oracle's time does not depend on the scale values)."""
    import oracle
    layer = S.prefill()
    toks = np.arange(n_tokens)
    W = oracle.Weights(layer.E, layer.H, layer.I)
    used = np.unique(layer.topk_ids[toks])
    for e in used:
        W.w13_q[e], W.w13_sf[e], W.w13_scale2[e] = oracle.quantize_weight(layer.weight_bf16(int(e), "w13"))
        W.w2_q[e], W.w2_sf[e], W.w2_scale2[e] = oracle.quantize_weight(layer.weight_bf16(int(e), "w2"))
    for e in range(layer.E):
        if e not in used:
            W.w13_scale2[e] = W.w2_scale2[e] = np.float32(1.0)
    W.w13_input_scale = layer.w13_input_scale.copy()
    W.w2_input_scale = np.full(layer.E, np.float32(16.0 / 2688.0))
    return oracle, layer, W, toks


def cpu_baseline(args):
    """The oracle on the first tokens of the prefill workload, as many as take
    about args.cpu_seconds of CPU work.  The sample is sized from a run on
    args.cpu_tokens tokens: each expert a sample touches costs a fixed weight
    decoding, so a much smaller calibration would understate the rate."""
    orc, layer, W, toks = oracle_sample_setup(8192)  # every token of the prefill layer
    n0 = min(len(toks), args.cpu_tokens)
    t0 = time.perf_counter()
    orc.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=toks[:n0])
    rate = n0 / (time.perf_counter() - t0)
    toks = toks[:int(min(len(toks), max(n0, rate * args.cpu_seconds)))]
    t0 = time.perf_counter()
    orc.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=toks)
    dt = time.perf_counter() - t0
    return {"value": len(toks) / dt, "unit": "tokens/s", "cores": orc.threads(), "kind": "oracle",
            "sample": f"{len(toks)} of 8192 prefill tokens ({len(toks) * layer.k} routed rows), whole expert "
                      f"path, {dt:.1f} s"}


def stack_leg(m, torch, args):
    """The 30-layer stack: 30 decode-shaped layers (128 experts, 2816 x 704,
    top-8) at 2048 tokens, each with its own device-drawn weights and its own
    seeded routing (drawn independently of its input: the expert path only),
    residual add + RMSNorm (eps 1e-6) between layers.  One step = all 30
    layers (forward + normalisation each), timed with CUDA events; tokens/s =
    2048 / step time."""
    LAYERS, T = 30, 2048
    layers = []
    out = ws = None
    for li in range(LAYERS):
        L = S.stack_layer(li, T)
        w, bf = make_layer_device(L, m, torch, seed=5004 + 100 * li)
        del bf
        x = torch.from_numpy(L.x.view(np.int16)).cuda().view(torch.bfloat16)
        ids = torch.from_numpy(L.topk_ids).cuda()
        tw = torch.from_numpy(L.topk_w).cuda()
        calibrate_w2_on_device(m, torch, w, x, ids, tw, L)
        m.prepare_weights(w)
        if li == 0:
            x0 = x
            out = torch.empty((T, L.H), dtype=torch.float32, device="cuda")
            ws = torch.empty(m.moe_workspace_size(T, L.H, L.I, L.E, L.k), dtype=torch.uint8, device="cuda")
        layers.append((w, ids, tw))
    xa, xb = x0.clone(), torch.empty_like(x0)
    for (w, ids, tw) in layers:  # the checked pass: every layer's scale check with the host sync
        m.moe_forward(w, xa, ids, tw, out=out, ws=ws, flags=m.SYNC_CHECK)
        m.residual_rmsnorm(xa, out, 1e-6, x_next=xb)
        xa, xb = xb, xa

    def step():
        nonlocal xa, xb
        xa.copy_(x0)
        for (w, ids, tw) in layers:
            m.moe_forward(w, xa, ids, tw, out=out, ws=ws, flags=m.SCALES_PREVALIDATED)
            m.residual_rmsnorm(xa, out, 1e-6, x_next=xb)
            xa, xb = xb, xa

    for _ in range(3):
        step()
    n = max(5, args.steps // 20)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(n):
        step()
    b.record()
    torch.cuda.synchronize()
    st, _ = m.moe_status(ws)
    ms = a.elapsed_time(b) / n
    res = {"layers": LAYERS, "T": T, "ms_per_stack": ms, "tokens_per_s": T / (ms * 1e-3),
           "ms_per_layer": ms / LAYERS, "status": st, "steps": n,
           "note": "each step: a 5.8 MB copy of the first input, then 30 x (expert forward + residual RMSNorm)"}
    del layers, out, ws
    torch.cuda.empty_cache()
    return res


def oracle_timings(args):
    """The oracle on one core and on all cores: the tiny layer (whole path)
    and the quantiser workload (routed-row quantisation of a bounded token
    sample; GB/s over the same algorithmic bytes the GPU's figure uses)."""
    import oracle as orc
    orc.build()
    tiny = S.tiny()
    res = {}
    W = orc.quantize_layer_weights(tiny)
    q = S.quantiser()
    ntok = min(q.T, args.oracle_quant_tokens)
    xq, idq = q.x[:ntok], q.topk_ids[:ntok]
    nbytes = ntok * q.H * 2 + ntok * q.k * q.H * (0.5 + 1 / 16) + ntok * q.k * 8
    saved = os.environ.get("ORACLE_THREADS")
    try:
        for label, threads in (("1_core", 1), ("all_cores", 0)):
            if threads:
                os.environ["ORACLE_THREADS"] = str(threads)
            elif saved is None:
                os.environ.pop("ORACLE_THREADS", None)
            else:
                os.environ["ORACLE_THREADS"] = saved
            t0 = time.perf_counter()
            reps = 0
            while reps < 3 or time.perf_counter() - t0 < 1.0:
                orc.moe_forward(tiny.x, tiny.topk_ids, tiny.topk_w, W)
                reps += 1
            t_tiny = (time.perf_counter() - t0) / reps
            t0 = time.perf_counter()
            orc.quantize_experts(xq, idq, q.w13_input_scale, q.E)
            t_q = time.perf_counter() - t0
            res[label] = {"threads": orc.threads(),
                          "tiny_layer": {"ms": t_tiny * 1e3, "tokens_per_s": tiny.T / t_tiny},
                          "quantiser": {"tokens": ntok, "s": t_q, "gbs": nbytes / t_q / 1e9,
                                        "tokens_per_s": ntok / t_q}}
    finally:
        if saved is None:
            os.environ.pop("ORACLE_THREADS", None)
        else:
            os.environ["ORACLE_THREADS"] = saved
    return res


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on the host cores; each
    step is the whole expert path for a bounded token sample of the workload,
    sized from a calibration run so that all steps take about two minutes."""
    if rank != 0:
        return None
    orc, layer, W, toks = oracle_sample_setup(args.cpu_tokens)
    t0 = time.perf_counter()
    orc.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=toks[:64])
    rate = 64 / (time.perf_counter() - t0)
    n = int(min(len(toks), max(8, rate * 120.0 / max(1, args.steps + args.warmup))))
    toks = toks[:n]
    for _ in range(args.warmup):
        orc.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=toks)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=toks)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = len(toks) / (ms * 1e-3)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int64 exact products, fp64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "T": layer.T, "E": layer.E, "H": layer.H, "I": layer.I,
                       "k": layer.k, "sample_tokens_per_step": len(toks)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": orc.threads(), "kind": "oracle",
                             "sample": f"{len(toks)} of 8192 prefill tokens per step, whole expert path"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=1024)  # reference arm: largest token sample per step
    ap.add_argument("--cpu-seconds", type=float, default=15.0)  # cpu_baseline: CPU work to time
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack", action="store_true")  # skip the 30-layer stack leg
    ap.add_argument("--oracle-quant-tokens", type=int, default=512)  # oracle quantiser timing sample
    ap.add_argument("--tokens", type=int, default=8192,
                    help="prefill tokens (8192 is the benchmark workload; smaller values for ncu captures)")
    ap.add_argument("--only-w4a16", action="store_true",
                    help="time only the W4A16 path on the prefill layer (for profiling runs)")
    ap.add_argument("--only-layer", action="store_true",
                    help="time only the layer steps (no quantiser workload, e2e or CPU baseline)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    line = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
