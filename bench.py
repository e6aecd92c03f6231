"""Benchmark of the chunk denoising step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--config default|sr|base|sr1|long|ibase|block|small|tiny] [--impl ours|reference]

One step is one pass of the whole hot path through the library's public API
(chunk_stream_step): 3D RoPE of the chunk's q and k, attention of the chunk's
queries over [reference | boundary | chunk], and the W_o GEMM with the Euler
update fused into its epilogue; the last step of every chunk also rolls the
boundary.  Inputs are seeded synthetic tensors shaped like the workload, two
input sets alternate between steps (each larger than the 129 MB L2), resident
in HBM before timing.  Each rank runs an independent replica (sessions are
independent; no collective on the data path), so scaling is weak.

The default run measures the SR-shaped chunk (the largest configuration that
fits one GPU) as the headline line, and the base-DiT chunk, the 1-step SR
chunk, the long session (4 sessions x 64 chunks), the interpolation-chunk step
and the DiT attention-block step under the keys "base", "sr1", "long",
"ibase" and "block".
Printed: one JSON line on rank 0.  value = dense attention TFLOP per step /
device time per step (whole job); e2e = the same through the C-ABI call that
takes host buffers: every step, the host -> device copy of the step's q, k, v
from pinned memory and the device -> host read of the updated state x inside
the timed region.  The reference arm
(--impl reference) times the fp64 CPU oracle on bounded samples of the same
workload and extrapolates each to a full step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from streaming_avatar_video_gb300 import inputs as I  # noqa: E402

METRIC = "chunk-attention TFLOP/s (% of bf16 tensor peak); latent frames/s per denoise step"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one attention
# launch, from one ncu capture per workload, keyed by the sha256 of the kernel
# sources the capture was taken on (attention.cu, ptx.cuh, common.h); any later
# change of them reports null.
ATTN_TRAFFIC = {
    # profiles/chunk_attention_base.md and profiles/chunk_attention_sr.md: the fused-RoPE kernel the stream
    # runs; base 291.848 MB read + 61.056 MB written, SR 1720.399 MB read + 295.447 MB written
    "e8953a85b0dbd3b45a18a45a833dfcf75489c2be595551076a0736069d9ff2e2": {"base": 352904192, "sr": 2015845632},
}


def attn_traffic(workload: str):
    import hashlib
    h = hashlib.sha256()
    for f in ("attention.cu", "ptx.cuh", "common.h"):
        with open(os.path.join(ROOT, "streaming_avatar_video_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    # the 1-step SR chunk launches the same attention as the SR chunk
    return ATTN_TRAFFIC.get(h.hexdigest(), {}).get("sr" if workload == "sr1" else workload)


NOMINAL_BF16_TFLOPS = 2250.0
# a timed region shorter than this compares with the burst GEMM figure
BURST_REGION_S = 3.0


def describe(w: I.Workload) -> str:
    return (f"{w.name}: B{w.B} H{w.H} D{w.D} chunk {w.F}x{w.grid_h}x{w.grid_w}={w.n_q} q tokens, "
            f"{w.n_ref} ref + {w.n_b} boundary + {w.n_q} chunk kv tokens, "
            f"{w.steps} Euler steps/chunk (shift {w.shift:g})")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """SM clock, power draw and clock-event (throttle) reasons sampled during
    a timed region.  Read-only NVML queries through ctypes every 5 ms on a
    thread of this process, so that even a region of a few tens of
    milliseconds gets samples under load; nvidia-smi -lms 25 when the NVML
    library cannot be loaded.  Nothing here changes a setting of the GPU."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int, period_s: float = 0.005):
        self.device = device
        self.period = period_s
        self.samples = []  # (sm MHz, power W, reasons bitmask)
        self.sm_max = None
        self.source = None
        self._nvml = None
        self._h = None
        self._proc = None

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            ok = False
            props = torch.cuda.get_device_properties(self.device)
            if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
                bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0
            if not ok:
                ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.device), ctypes.byref(h)) == 0
            if not ok:
                return False
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.sm_max = float(mx.value)
            self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self._nvml, self._h = lib, h
            return True
        except Exception:
            return False

    def _poll(self):
        import ctypes
        lib, h = self._nvml, self._h
        mhz, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
                self._reasons(h, ctypes.byref(rs))
                self.samples.append((float(mhz.value), mw.value / 1000.0, int(rs.value)))
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        if self._open_nvml():
            self.source = "nvml"
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return self
        self.source = "nvidia-smi"
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.source == "nvml":
            self._stop.set()
            self._thread.join(timeout=1.0)
            try:
                self._nvml.nvmlShutdown()
            except Exception:
                pass
            return
        if self._proc is None:
            return
        time.sleep(0.15)
        self._proc.terminate()
        try:
            out, _ = self._proc.communicate(timeout=5)
        except Exception:
            self._proc.kill()
            out = ""
        names = {5: 0x8, 6: 0x40, 7: 0x20, 8: 0x4}
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx, pw = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            bits = 0
            for i, b in names.items():
                if f[i].lower() == "active":
                    bits |= b
            self.samples.append((sm, pw, bits))
            self.sm_max = mx

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": [], "samples": 0, "source": self.source}
        bits = 0
        for _, _, b in self.samples:
            bits |= b
        return {"sm_mhz": statistics.median(s[0] for s in self.samples), "sm_max_mhz": self.sm_max,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b),
                "power_w_median": round(statistics.median(s[1] for s in self.samples), 1),
                "samples": len(self.samples), "source": self.source}


def dist_setup(backend: str = "nccl"):
    """Reads RANK / LOCAL_RANK / WORLD_SIZE (torchrun) and joins the process
    group when there is more than one rank.  Returns (world, rank, local)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    """The largest of every rank's value (the slowest rank's time)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, ms_max: float) -> float:
    """Units per second of the whole job: every rank processes the same
    number of units (weak scaling), the job ends with the slowest rank."""
    return world * units_per_rank / (ms_max * 1e-3)


# ------------------------------------------------------------------ our arm

def run_ours(args, w: I.Workload, world: int, rank: int, local: int):
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    seed = 1 + rank
    dts = S.flow_time_grid(w.steps, w.shift)

    # two input sets (each > L2) alternate between steps; generated on the host, resident in HBM
    sets = []
    for c in range(2):
        st = I.step_inputs(w, seed, c, 0)
        sets.append((st.q, st.k, st.v))
    dsets = [tuple(t.to(dev) for t in s) for s in sets]
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).to(dev)
    x = I.state_x(w, seed).to(dev)

    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base, host_io=0 if args.no_e2e else 8)
    cs.set_reference(rk.to(dev), rv.to(dev))
    # prime: one chunk end so that every timed step attends over the boundary too
    q, k, v = dsets[0]
    cs.step(q, k, v, wo, x, dts[0], True)
    cs.end_chunk()

    state = {"i": 0}

    def one_step(events=None):
        # 3 launches (RoPE of k, attention, W_o + Euler), and the boundary's RoPE after a chunk's last step
        i = state["i"]
        s = i % w.steps
        q, k, v = dsets[i & 1]
        last = s == w.steps - 1
        if events is not None:
            cs.set_step_events(events)
        cs.step(q, k, v, wo, x, dts[s], last)
        if last:
            cs.end_chunk()
        state["i"] = i + 1

    for _ in range(args.warmup):
        one_step()
    cs.sync()

    # timed region: K steps with nothing else on the stream (events between the
    # kernels of a step cost a few % of it: they break the programmatic overlap)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        l0 = S.savgb_kernel_launches()
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for k_ in range(args.steps):
            one_step()
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    launches = S.savgb_kernel_launches() - l0  # the library's own count of the kernels it enqueued
    clocks = clk.summary()

    # end-to-end through the public API with host buffers, right after the
    # headline region so that both run in the same thermal and power state
    e2e = None
    if not args.no_e2e:
        e2e, state["i"] = run_e2e(args, w, cs, sets, wo, x, dts, dev, stream, world, state["i"])

    # a second K-step timed region, with CUDA events around each stage of
    # every step, for the per-kernel times and the roofline
    start_i, end_i = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk_i:
        barrier(world)
        torch.cuda.synchronize()
        start_i.record(stream)
        for k_ in range(args.steps):
            one_step(ev[k_])
        end_i.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    cs.sync()
    ms_local = start.elapsed_time(end)
    ms_total = max_over_ranks(world, ms_local)
    ms_step = ms_total / args.steps
    ms_step_instr = max_over_ranks(world, start_i.elapsed_time(end_i)) / args.steps
    rope_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    wo_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    clocks_i = clk_i.summary()

    attn_flops = w.attn_flops(True)
    value = whole_job_rate(world, attn_flops, ms_step) / 1e12
    frames_per_s = whole_job_rate(world, w.B * w.F, ms_step)
    attn_tflops = attn_flops / (attn_ms * 1e-3) / 1e12
    pk, pk_kind = peaks()
    # the kernels' timed region lasts K steps; a region of a few seconds or
    # less compares with cuBLAS's burst figure, a longer one with the
    # sustained (power-capped) one
    region_s = ms_step_instr * args.steps * 1e-3
    use_burst = region_s < BURST_REGION_S
    peak = pk["bf16_tflops"] if use_burst else pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    peak_kind = (f"{pk_kind} bf16 burst (cuBLAS 8192^3, best of 10): the kernels' timed region lasts "
                 f"{region_s:.2f} s (< {BURST_REGION_S:g} s)" if use_burst else
                 f"{pk_kind} bf16 sustained (cuBLAS back to back for 4 s): the kernels' timed region lasts "
                 f"{region_s:.2f} s")
    # the stream rotates q inside the attention kernel when its RoPE table fits;
    # the RoPE pass then moves k alone
    fused = cs.fused_q_rope
    rope_bytes = 2 * 2 * (1 if fused else 2) * w.B * w.n_q * w.hid  # read + write, 2 bytes each
    wo_flops = w.wo_flops()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    exp_forms = None
    if fused and not args.no_exp_forms:
        exp_forms = time_exp_forms(S, w, dsets, dev, stream, max(3, min(args.steps, 20)))
    rope_loop_ms = time_rope_loop(S, w, dsets, stream, max(20, args.steps))

    cs.close()

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v/ref, W_o ~ N(0,1/hid), x ~ N(0,1))",
        "config": config_of(w, world),
        "latent_frames_per_s": round(frames_per_s, 1),
        "pct_of_bf16_peak": {"nominal_2250": round(100 * attn_tflops / NOMINAL_BF16_TFLOPS, 1),
                             f"{pk_kind}_sustained": round(100 * attn_tflops / pk.get("bf16_tflops_sustained",
                                                                                       pk["bf16_tflops"]), 1),
                             f"{pk_kind}_burst": round(100 * attn_tflops / pk["bf16_tflops"], 1)},
        # one exp per score: B*H*Nq*Nkv per attention launch
        "softmax_exps": {"per_step": w.B * w.H * w.n_q * w.n_kv,
                         "per_s": round(w.B * w.H * w.n_q * w.n_kv / (attn_ms * 1e-3), 1)},
        "kernels_timed_region": {"steps": args.steps, "ms_per_step": round(ms_step_instr, 4), "clocks": clocks_i,
                                 "what": "a second K-step region with CUDA events around each stage of every step"},
        "kernels_ms": {("rope3d_k" if fused else "rope3d_qk"): round(rope_ms, 4),
                       ("chunk_attention_qrope" if fused else "chunk_attention"): round(attn_ms, 4),
                       "out_proj_euler": round(wo_ms, 4)},
        "kernel_rates": {
            "chunk_attention_tflops": round(attn_tflops, 1),
            "out_proj_euler_tflops": round(wo_flops / (wo_ms * 1e-3) / 1e12, 1),
            "rope3d_gbs": round(rope_bytes / (rope_ms * 1e-3) / 1e9, 1),
            # the k-only pass timed back to back (programmatic launch overlapping each launch's table build with
            # the previous one's tail, as between the kernels of a step), not between events
            "rope3d_k_loop": {"ms": round(rope_loop_ms, 4),
                              "gbs": round(4 * w.B * w.n_q * w.hid / (rope_loop_ms * 1e-3) / 1e9, 1),
                              f"pct_of_{pk_kind}_copy": round(100 * 4 * w.B * w.n_q * w.hid / (rope_loop_ms * 1e-3)
                                                              / 1e9 / pk["hbm_gbs"], 1)},
            "rope3d_pct_of_hbm": {"nominal_8000": round(100 * rope_bytes / (rope_ms * 1e-3) / 8e12, 1),
                                  f"{pk_kind}_copy": round(100 * rope_bytes / (rope_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 1)},
        },
        "clock_normalised": clock_normalised(attn_flops, attn_ms, wo_flops, wo_ms, clocks_i.get("sm_mhz"), sms),
        "roofline": {
            "kernel": ("chunk_attention_qrope (attn_fwd_kernel<128, 2, 2, true, false>: RoPE of q fused)" if fused
                       else "chunk_attention (attn_fwd_kernel<128, 3, 2, false, false>)"),
            "bound": "tensor",
            "achieved": round(attn_tflops, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "TFLOP/s",
            "frac": round(attn_tflops / peak, 4),
            "frac_of": "measured" if pk_kind == "measured" else "fallback",
            "traffic": attn_traffic(w.name),
            "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
            "algorithmic": f"4*B*H*Nq*Nkv*D = {attn_flops / 1e12:.4f} TFLOP per launch",
            "min_bytes": 2 * w.B * w.hid * (2 * w.n_q + 2 * w.n_kv),
        },
        "softmax_exp_forms": exp_forms,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": None,
    }
    return result


def config_of(w: I.Workload, world: int) -> dict:
    """The workload description shared by both arms' JSON lines."""
    return {
        "workload": describe(w),
        "parallelism": f"replicas x{world} (independent sessions)",
        "global_batch": world * w.B,
        "l2": "inputs larger than L2: two alternating input sets of "
              f"{3 * w.B * w.n_q * w.hid * 2 / 1e6:.0f} MB",
    }


def clock_normalised(attn_flops, attn_ms, wo_flops, wo_ms, sm_mhz, sms):
    """Kernel work per SM clock at the median SM clock sampled during the
    timed regions: clocks per 128x128x16 bf16 MMA (2*128*128*16 flops) and
    flops per clock per SM.  Boxes settle at different clocks under the power
    cap; these figures compare kernels across them."""
    if not sm_mhz:
        return None
    per_mma = 2.0 * 128 * 128 * 16

    def one(flops, ms):
        clk = ms * 1e-3 * sm_mhz * 1e6
        return {"clocks_per_mma_128x128x16": round(clk / (flops / per_mma / sms), 2),
                "flop_per_clk_per_sm": round(flops / (clk * sms), 1)}

    return {"sm_mhz_median": sm_mhz, "sms": sms, "chunk_attention": one(attn_flops, attn_ms),
            "out_proj_euler": one(wo_flops, wo_ms)}


def time_rope_loop(S, w, dsets, stream, k):
    """The RoPE pass of a stream step (k alone, chunk-local positions) as k
    back-to-back launches between two events, alternating the two input sets
    (each larger than L2) into one output; ms per launch."""
    out = torch.empty_like(dsets[0][1])
    grid = (w.F, w.grid_h, w.grid_w)
    for i in range(max(10, k)):  # warm-up: the memory clock ramps with sustained traffic
        S.rope3d_apply(dsets[i & 1][1], out, *grid, 0, w.rope_base)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(k):
        S.rope3d_apply(dsets[i & 1][1], out, *grid, 0, w.rope_base)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / k


def time_exp_forms(S, w, dsets, dev, stream, k):
    """The attention kernel with RoPE of q inside, as the stream runs it
    (packed bf16x2 exponentials), against its instantiation with fp32
    exponentials and exact row sums (the one the log-sum-exp output selects),
    on this workload's shapes: k stand-alone launches of each, alternated in
    rounds, CUDA events on the launching stream.  Both read one prebuilt
    cos/sin table."""
    q, kk, v = dsets[0]
    segs = [(kk[:, :w.n_ref].contiguous(), v[:, :w.n_ref].contiguous())]
    if w.n_b:
        segs.append((kk[:, :w.n_b].contiguous(), v[:, :w.n_b].contiguous()))
    segs.append((kk, v))
    grid = (w.F, w.grid_h, w.grid_w)
    tab = S.chunk_attention_qrope_table(w.D, grid, 0, w.rope_base)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.n_q), dtype=torch.float32, device=dev)
    times = {"packed": [], "fp32": []}
    for _ in range(2):  # warm both
        S.chunk_attention_qrope_with_table(q, grid, tab, segs, 0, out)
        S.chunk_attention_qrope_with_table(q, grid, tab, segs, 0, out, lse=lse)
    torch.cuda.synchronize()
    for r in range(4):
        for form in ("packed", "fp32") if r % 2 == 0 else ("fp32", "packed"):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(k):
                S.chunk_attention_qrope_with_table(q, grid, tab, segs, 0, out, lse=lse if form == "fp32" else None)
            b.record(stream)
            torch.cuda.synchronize()
            times[form].append(a.elapsed_time(b) / k)
    S.savgb_device_check()
    pk = statistics.median(times["packed"])
    fp = statistics.median(times["fp32"])
    flops = w.attn_flops(True)
    return {"packed_bf16x2_exp_ms": round(pk, 4), "fp32_exp_ms": round(fp, 4),
            "packed_tflops": round(flops / (pk * 1e-3) / 1e12, 1), "fp32_tflops": round(flops / (fp * 1e-3) / 1e12, 1),
            "fp32_over_packed": round(fp / pk, 4),
            "what": f"stand-alone chunk_attention_qrope_with_table launches, {k} per round, 4 rounds alternating "
                    "the forms, median of the rounds; the fp32 form is the one the log-sum-exp output selects"}


def run_e2e(args, w, cs, sets, wo, x, dts, dev, stream, world, i0=0):
    """Same metric through the C-ABI call with HOST buffers:
    chunk_stream_step_host takes the step's q, k, v from pinned host memory
    and reads the updated state x back into pinned host memory every step.
    The library uploads each step's inputs into one of eight device slots on
    a copy stream, up to seven steps ahead of the compute, and reads x back
    from a staging copy (written by the W_o update beside x, two alternating)
    on a second copy stream while the next steps compute.  The timed region ends
    once the last read-back has landed (join_copies, then an event)."""
    hsets = [tuple(t.pin_memory() for t in s) for s in sets]
    hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    n = max(3, min(args.steps, 60))

    def step(i, read_back=True, ev=None):
        s_idx = (i0 + i) % w.steps
        last = s_idx == w.steps - 1
        hq, hk, hv = hsets[i & 1]
        cs.step_host(hq, hk, hv, wo, x, dts[s_idx], last, x_host=hx if read_back else None)
        if ev is not None:
            ev.record(stream)
        if last:
            cs.end_chunk()

    for i in range(3):
        step(i)
    cs.sync()
    copies = time_copies_alone(hsets[0], hx, dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        a.record(stream)
        for i in range(3, 3 + n):
            step(i)
        cs.join_copies()
        b.record(stream)
        torch.cuda.synchronize()
    cs.sync()
    ms = max_over_ranks(world, a.elapsed_time(b)) / n
    # diagnostics, after the timed region: the same loop with the uploads only,
    # and the period of every step of one more pass (events on the compute stream)
    i_next = 3 + n
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record(stream)
    for i in range(i_next, i_next + n):
        step(i, read_back=False)
    b2.record(stream)
    torch.cuda.synchronize()
    cs.sync()
    i_next += n
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    stage = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    evs[0].record(stream)
    for j, i in enumerate(range(i_next, i_next + n)):
        cs.set_step_events(stage[j])
        step(i, ev=evs[j + 1])
    cs.join_copies()
    torch.cuda.synchronize()
    cs.sync()
    i_next += n
    periods = [round(evs[j].elapsed_time(evs[j + 1]), 3) for j in range(n)]
    # a step starts once its upload has landed: the gap after the previous step is the upload's wait; W_o's span
    # includes its wait for the read-back that last used its staging copy
    upload_wait = [round((evs[j] if j == 0 else stage[j - 1][3]).elapsed_time(stage[j][0]), 3) for j in range(n)]
    wo_span = [round(stage[j][2].elapsed_time(stage[j][3]), 3) for j in range(n)]
    h2d = sum(t.numel() * t.element_size() for t in sets[0])
    d2h = x.numel() * x.element_size()
    return {"value": round(whole_job_rate(world, w.attn_flops(True), ms) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "clocks": clk.summary(), "copies_alone": copies,
            "diagnostics": {"uploads_only_ms_per_step": round(a2.elapsed_time(b2) / n, 4),
                            "step_periods_ms": periods,
                            "upload_wait_ms": upload_wait,
                            "wo_incl_readback_wait_ms": wo_span,
                            "what": "after the timed region: the same loop without read-backs, and for each step "
                                    "of one more pass its period, the compute stream's wait for its upload and "
                                    "the span of its W_o update with any wait for an earlier read-back (events "
                                    "on the compute stream)"},
            "api": "C ABI chunk_stream_step_host: pinned host q/k/v in, x read back to pinned host memory every "
                   "step; the library overlaps the uploads and read-backs with the steps on two copy streams; "
                   "measured right after the headline region"}, i0 + i_next


def time_copies_alone(h_inputs, hx, dev):
    """The e2e loop's host copies with no compute running, on this machine: one
    step's inputs host -> device and the state device -> host (pinned
    buffers, torch copies into a scratch device buffer), median of 3.  When
    they take longer than a step, the e2e loop is bound by the host side."""
    d_in = [torch.empty_like(t, device=dev) for t in h_inputs]
    d_x = torch.empty(hx.shape, dtype=hx.dtype, device=dev)
    out = {}
    for name, fn in (("h2d", lambda: [d.copy_(h, non_blocking=True) for d, h in zip(d_in, h_inputs)]),
                     ("d2h", lambda: hx.copy_(d_x, non_blocking=True))):
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        nbytes = sum(t.numel() * t.element_size() for t in h_inputs) if name == "h2d" else hx.numel() * hx.element_size()
        out[name] = {"ms": round(ms, 3), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    del d_in, d_x
    return out


def run_long(args, w: I.Workload, world: int, rank: int, local: int):
    """Long streaming session: w.B sessions batched, args.chunks consecutive
    chunks of w.steps denoising steps each, the boundary rolled every chunk.
    Reports the attention throughput over the whole run, sustained latent
    frames/s, nearest-rank p50/p99 of the per-chunk latency, and whether the
    device's free memory stayed constant from chunk to chunk."""
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    seed = 1 + rank
    dts = S.flow_time_grid(w.steps, w.shift)
    sets = []
    for c in range(2):  # two resident input sets alternate between steps
        st = I.step_inputs(w, seed, c, 0)
        sets.append(tuple(t.to(dev) for t in (st.q, st.k, st.v)))
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).to(dev)
    x = I.state_x(w, seed).to(dev)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base)
    cs.set_reference(rk.to(dev), rv.to(dev))
    def chunk(i0):
        for s in range(w.steps):
            q, k, v = sets[(i0 + s) & 1]
            cs.step(q, k, v, wo, x, dts[s], s == w.steps - 1)
        cs.end_chunk()

    for c in range(max(1, args.warmup // w.steps + 1)):  # warm-up chunks
        chunk(0)
    cs.sync()
    n = args.chunks
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    free = []
    l0 = S.savgb_kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for c in range(n):
            chunk(c * w.steps)
            ev[c + 1].record(stream)
            if c % 8 == 7:
                free.append(torch.cuda.mem_get_info(dev)[0])  # synchronising query, outside the events
        torch.cuda.synchronize()
    launches = S.savgb_kernel_launches() - l0
    barrier(world)
    cs.sync()
    per_chunk = sorted(ev[c].elapsed_time(ev[c + 1]) for c in range(n))
    total_ms = max_over_ranks(world, ev[0].elapsed_time(ev[n]))
    nearest = lambda q: per_chunk[max(0, math.ceil(q * len(per_chunk)) - 1)]
    info = cs.info()
    cs.close()
    attn = w.attn_flops(True) * w.steps * n
    return {
        "metric": METRIC,
        "value": round(whole_job_rate(world, attn, total_ms) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": n * w.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / (n * w.steps), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v/ref, W_o ~ N(0,1/hid), x ~ N(0,1))",
        "config": {"workload": describe(w) + f", {n} consecutive chunks", "parallelism": f"replicas x{world}",
                   "global_batch": world * w.B,
                   "l2": "inputs larger than L2: two alternating input sets of "
                         f"{3 * w.B * w.n_q * w.hid * 2 / 1e6:.0f} MB"},
        "sustained_latent_frames_per_s": round(whole_job_rate(world, w.B * w.F * n, total_ms), 2),
        "chunk_latency_ms": {"p50": round(nearest(0.50), 3), "p99": round(nearest(0.99), 3),
                             "min": round(per_chunk[0], 3), "max": round(per_chunk[-1], 3)},
        "memory": {"arena_bytes": info["arena_bytes"], "free_bytes_samples": len(free),
                   "free_bytes_constant": len(set(free)) <= 1},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None, "cpu_baseline": None, "roofline": None,
    }


def run_interp(args, w: I.Workload, world: int, rank: int, local: int):
    """Interpolation-chunk steps of a base-shaped stream: N0 and N1 are run
    first, then K timed steps of the pending I chunk (its F-2 interior frames
    attend over [reference | two anchor frames | interior])."""
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    seed = 1 + rank
    dts = S.flow_time_grid(w.steps, w.shift)
    st = I.step_inputs(w, seed, 0, 0)
    q, k, v = (t.to(dev) for t in (st.q, st.k, st.v))
    rk, rv = I.reference_kv(w, seed)
    wo = I.out_proj_weight(w, seed).to(dev)
    x = I.state_x(w, seed).to(dev)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base, interp_chunks=True)
    cs.set_reference(rk.to(dev), rv.to(dev))
    for c in range(2):  # N0, N1 (one step each is enough to fill the anchors)
        cs.step(q, k, v, wo, x, dts[0], True)
        cs.end_chunk()
    isets = []
    for c in range(2):
        si = I.istep_inputs(w, seed, c, 0)
        isets.append(tuple(t.to(dev) for t in (si.q, si.k, si.v)))
    n_int = (w.F - 2) * w.frame_tokens
    xi = torch.zeros((w.B * n_int, w.hid), dtype=torch.float32, device=dev)
    for i in range(args.warmup):
        cs.istep(*isets[i & 1], wo, xi, dts[i % w.steps])
    cs.sync()
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        l0 = S.savgb_kernel_launches()
        a.record(stream)
        for i in range(args.steps):
            cs.istep(*isets[i & 1], wo, xi, dts[i % w.steps])
        b.record(stream)
        torch.cuda.synchronize()
        launches = S.savgb_kernel_launches() - l0
    barrier(world)
    cs.sync()
    cs.close()
    ms = max_over_ranks(world, a.elapsed_time(b)) / args.steps
    n_kv = w.n_ref + 2 * w.frame_tokens + n_int
    flops = 4.0 * w.B * w.H * n_int * n_kv * w.D
    return {
        "metric": METRIC,
        "value": round(whole_job_rate(world, flops, ms) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v/ref, W_o ~ N(0,1/hid))",
        "config": {"workload": f"interpolation chunk of {describe(w)}: {n_int} interior queries over "
                               f"{w.n_ref} ref + {2 * w.frame_tokens} anchor + {n_int} interior kv tokens",
                   "parallelism": f"replicas x{world}", "global_batch": world * w.B,
                   "l2": "two alternating input sets larger than L2"},
        "latent_frames_per_s": round(whole_job_rate(world, w.B * (w.F - 2), ms), 1),
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None, "cpu_baseline": None, "roofline": None,
    }


def run_block(args, w: I.Workload, world: int, rank: int, local: int):
    """Block steps of a base-shaped stream: the chunk's q, k, v are projected
    from the state x by the QKV GEMM (RoPE of q, k in its epilogue), then
    attention and W_o + Euler.  One priming chunk end gives every timed step a
    boundary."""
    import __graft_entry__ as g
    g.build()
    from streaming_avatar_video_gb300 import savgb as S

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    seed = 1 + rank
    dts = S.flow_time_grid(w.steps, w.shift)
    rk, rv = I.reference_kv(w, seed)
    wqkv = I.qkv_weight(w, seed).to(dev)
    wo = I.out_proj_weight(w, seed).to(dev)
    x = I.state_x(w, seed).to(dev)
    cs = S.ChunkStream(w.B, w.H, w.D, w.F, w.grid_h, w.grid_w, w.ref_frames, w.boundary_frames, w.ref_t,
                       w.rope_base, qkv_block=True)
    cs.set_reference(rk.to(dev), rv.to(dev))
    cs.block_step(wqkv, wo, x, dts[0], True)
    cs.end_chunk()
    state = {"i": 0}

    def one(events=None):
        i = state["i"]
        s_ = i % w.steps
        last = s_ == w.steps - 1
        if events is not None:
            cs.set_step_events(events)
        cs.block_step(wqkv, wo, x, dts[s_], last)
        if last:
            cs.end_chunk()
        state["i"] = i + 1

    for _ in range(args.warmup):
        one()
    cs.sync()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ai, bi = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # the steps alone, then a second region with per-stage events
        l0 = S.savgb_kernel_launches()
        barrier(world)
        torch.cuda.synchronize()
        a.record(stream)
        for k_ in range(args.steps):
            one()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        launches = S.savgb_kernel_launches() - l0
        barrier(world)
        torch.cuda.synchronize()
        ai.record(stream)
        for k_ in range(args.steps):
            one(ev[k_])
        bi.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    cs.sync()
    cs.close()
    ms = max_over_ranks(world, a.elapsed_time(b)) / args.steps
    ms_instr = max_over_ranks(world, ai.elapsed_time(bi)) / args.steps
    qkv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    wo_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    attn = w.attn_flops(True)
    qkv_flops = 2.0 * w.B * w.n_q * w.hid * 3 * w.hid
    total = attn + qkv_flops + w.wo_flops()
    return {
        "metric": METRIC,
        "value": round(whole_job_rate(world, attn, ms) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded x ~ N(0,1), W_qkv, W_o ~ N(0,1/hid), reference ~ N(0,1))",
        "config": {"workload": "DiT attention block steps of " + describe(w),
                   "parallelism": f"replicas x{world}", "global_batch": world * w.B,
                   "l2": "state and operands larger than L2"},
        "latent_frames_per_s": round(whole_job_rate(world, w.B * w.F, ms), 1),
        "block_tflops": round(whole_job_rate(world, total, ms) / 1e12, 1),
        "kernels_timed_region": {"steps": args.steps, "ms_per_step": round(ms_instr, 4),
                                 "what": "a second K-step region with CUDA events around each stage of every step"},
        "kernels_ms": {"to_bf16+qkv_rope_project": round(qkv_ms, 4), "chunk_attention": round(attn_ms, 4),
                       "out_proj_euler": round(wo_ms, 4)},
        "kernel_rates": {"qkv_tflops": round(qkv_flops / (qkv_ms * 1e-3) / 1e12, 1),
                         "chunk_attention_tflops": round(attn / (attn_ms * 1e-3) / 1e12, 1),
                         "out_proj_euler_tflops": round(w.wo_flops() / (wo_ms * 1e-3) / 1e12, 1)},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None, "cpu_baseline": None, "roofline": None,
    }


# ------------------------------------------------------------- oracle arm

class OracleSample:
    """The fp64 CPU oracle on a bounded sample of one step of ``w``.

    Untimed set-up: the step's inputs and the rotated reference, boundary and
    chunk keys (the keys every query row needs).  Timed: RoPE of ``frames``
    latent frames of q and k, then attention over the full key/value set,
    W_o and the Euler update for ``rows`` random query rows of every session
    and head.  Both parts scale linearly (RoPE in frames, the rest in rows),
    so the per-step time is extrapolated from the sample."""

    def __init__(self, w: I.Workload, seed: int = 1):
        import oracle as O
        self.O, self.w = O, w
        st = I.step_inputs(w, seed, 0, 0)
        rk, rv = I.reference_kv(w, seed)
        bk, bv = I.boundary_kv(w, seed)
        self.wo = I.out_proj_weight(w, seed).double().numpy()
        self.x = I.state_x(w, seed).numpy().astype(np.float64)
        self.q, self.k, self.v = (t.double().numpy() for t in (st.q, st.k, st.v))
        self.segs = [
            (O.rope3d(rk.double().numpy(), w.ref_frames, w.grid_h, w.grid_w, w.ref_t, w.rope_base),
             rv.double().numpy()),
            (O.rope3d(bk.double().numpy(), w.boundary_frames, w.grid_h, w.grid_w, -w.boundary_frames,
                      w.rope_base) if w.n_b else np.zeros((w.B, 0, w.H, w.D)), bv.double().numpy()),
            (O.rope3d(self.k, w.F, w.grid_h, w.grid_w, 0, w.rope_base), self.v),
        ]
        self.q_rot = O.rope3d(self.q, w.F, w.grid_h, w.grid_w, 0, w.rope_base)
        self.dt = O.time_grid(w.steps, w.shift)[0]
        self.rng = np.random.default_rng(seed)

    def run(self, rows: int, frames: int):
        O, w = self.O, self.w
        rows = min(rows, w.n_q)
        frames = min(frames, w.F)
        sel = np.sort(self.rng.choice(w.n_q, size=rows, replace=False))
        nf = frames * w.frame_tokens
        t0 = time.perf_counter()
        O.rope3d(self.q[:, :nf], frames, w.grid_h, w.grid_w, 0, w.rope_base)
        O.rope3d(self.k[:, :nf], frames, w.grid_h, w.grid_w, 0, w.rope_base)
        t1 = time.perf_counter()
        o = O.attention(self.q_rot[:, sel], self.segs)
        flat_rows = (np.arange(w.B)[:, None] * w.n_q + sel[None, :]).reshape(-1)
        vel = O.out_proj(o.reshape(-1, w.hid), self.wo)
        O.euler_update(self.x[flat_rows], vel, self.dt)
        t2 = time.perf_counter()
        per_step = (t1 - t0) * (w.F / frames) + (t2 - t1) * (w.n_q / rows)
        desc = (f"oracle on {rows} of {w.n_q} query rows x {w.B} sessions x {w.H} heads over all "
                f"{w.n_kv} kv tokens, + RoPE of {frames} of {w.F} frames of q and k; per-step time "
                f"extrapolated linearly (rows, frames)")
        return t2 - t0, per_step, desc

    def calibrated(self, budget_s: float):
        """Rows and frames whose sample takes about ``budget_s`` seconds."""
        secs, _, _ = self.run(16, 1)
        rows = int(max(8, min(self.w.n_q, 16 * budget_s / max(secs, 1e-3))))
        frames = 1 if budget_s < 5 else self.w.F
        return rows, frames


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model, from lscpu, else /proc/cpuinfo, else the machine type."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine() or "unknown"


def cpu_baseline(w: I.Workload, budget_s: float):
    smp = OracleSample(w)
    rows, frames = smp.calibrated(budget_s)
    secs, per_step, desc = smp.run(rows, frames)
    return {"value": round(w.attn_flops(True) / per_step / 1e12, 6), "unit": "TFLOP/s",
            "cores": cpu_cores(), "cpu_model": cpu_model(), "kind": "oracle", "sample": desc,
            "sample_seconds": round(secs, 2), "extrapolated": True,
            "extrapolated_s_per_step": round(per_step, 2),
            "threads": "numpy BLAS default (all affinity cores)"}


def run_reference(args, w: I.Workload, world: int, rank: int):
    """The reference arm: the fp64 oracle as it stands, on the host cores.
    Each of the W + K "steps" is one bounded sample of the step (rows and
    frames as OracleSample.run), so the whole run ends within minutes; its
    time is extrapolated linearly to a full step, and the JSON says so in
    keys: extrapolated, samples, ms_per_sample next to the extrapolated
    ms_per_step.  steps / warmup are the driver's K / W, counted in samples."""
    if rank != 0:
        return None
    smp = OracleSample(w)
    budget = min(20.0, getattr(args, "cpu_seconds", 20.0), max(0.05, 100.0 / (args.steps + args.warmup)))
    rows, frames = smp.calibrated(budget)
    per, walls = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        wall, per_step, desc = smp.run(rows, frames)
        if i >= args.warmup:
            per.append(per_step)
            walls.append(wall)
    ms = 1e3 * statistics.mean(per)
    value = w.attn_flops(True) / (ms * 1e-3) / 1e12
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "steps_are": "bounded samples of the step, each extrapolated to a full step (see samples, ms_per_sample)",
        "extrapolated": True, "samples": len(per),
        "ms_per_sample": round(1e3 * statistics.mean(walls), 2),
        "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v/ref, W_o ~ N(0,1/hid), x ~ N(0,1))",
        "config": config_of(w, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": desc, "extrapolated": True},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def nested(res: dict) -> dict:
    """The figures of a second workload, nested in the headline line."""
    keys = ("value", "unit", "ms_per_step", "latent_frames_per_s", "pct_of_bf16_peak", "kernels_timed_region",
            "kernels_ms", "kernel_rates", "clock_normalised", "roofline", "softmax_exp_forms", "gpu_launches",
            "clocks", "e2e", "config")
    return {k: res.get(k) for k in keys}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="default",
                    choices=["default", "base", "sr", "sr1", "long", "ibase", "block", "small", "tiny"],
                    help="default: the SR-shaped chunk as the headline; the base-DiT chunk, the long session, the "
                         "interpolation chunk and the DiT block nested under their names")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-exp-forms", action="store_true", help="skip the packed / fp32 exponential comparison")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="default run: skip the nested long-session, interpolation-chunk and DiT-block workloads")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target length of the oracle's timed sample")
    ap.add_argument("--chunks", type=int, default=64, help="chunks of the long-session run (--config long)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    head = "sr" if args.config == "default" else args.config
    w = I.WORKLOADS["base" if head in ("ibase", "block") else head]
    # the reference arm runs on the host cores alone: its ranks need no GPU
    world, rank, local = dist_setup("gloo" if args.impl == "reference" else "nccl")
    if args.impl == "reference":
        res = run_reference(args, w, world, rank)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if head in ("long", "ibase", "block"):
        fn = {"long": run_long, "ibase": run_interp, "block": run_block}[head]
        res = fn(args, w, world, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res = run_ours(args, w, world, rank, local)
    if args.config == "default":
        res["base"] = nested(run_ours(args, I.WORKLOADS["base"], world, rank, local))
        if not args.no_extra_workloads:
            # the 1-step SR chunk: every step ends a chunk and rolls the boundary
            sub_args = argparse.Namespace(**vars(args))
            sub_args.no_e2e, sub_args.no_exp_forms = True, True
            res["sr1"] = nested(run_ours(sub_args, I.WORKLOADS["sr1"], world, rank, local))
            # the other configurations, each with its own timed region and clocks
            sub = ("value", "unit", "ms_per_step", "steps", "latent_frames_per_s", "sustained_latent_frames_per_s",
                   "chunk_latency_ms", "memory", "block_tflops", "kernels_ms", "kernel_rates", "gpu_launches",
                   "clocks", "config")
            for name, fn in (("long", run_long), ("ibase", run_interp), ("block", run_block)):
                r = fn(args, I.WORKLOADS["long" if name == "long" else "base"], world, rank, local)
                res[name] = {k: r[k] for k in sub if k in r}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
