"""Benchmark of the exact tiled attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
  1. fused RMSNorm on X[4096, 1024] (bf16, eps 1e-6),
  2. causal GQA prefill B=2, Hq=32, Hkv=8, T=8192, d=128 (bf16, scale 1/sqrt(128)),
  3. flash-decoding B=16, Hq=32, Hkv=8, d=128 over a bf16 KV cache with
     per-sequence lengths drawn uniformly in [8192, 32768] (split-KV + combine).
All inputs are resident in HBM before the timed region. The headline value is
the causal-prefill throughput in TFLOP/s (algorithmic FLOPs: 4d per visible
query/key pair); the decode KV-stream GB/s and the RMSNorm GB/s are reported
beside it. Kernel times come from CUDA events recorded on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the float64 CPU oracle is timed instead, on a bounded
sample of the same workload (the oracle is a deliberately slow definition, so
this is a reported baseline, not a target).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "attention TFLOPS (causal prefill) & decode KV-stream GB/s, as % of GB300 roofline"
PREFILL = W.GQA_LLAMA
DECODE = W.DECODE_LLAMA
NORM = W.NORM_QWEN
WORKLOAD = (f"{PREFILL.name} + {DECODE.name} + {NORM.name}")

# DRAM bytes (read + write) of one attn_fwd_kernel<128> launch on the prefill workload, from the
# ncu capture summarised in profiles/attn_fwd_kernel_d128_causal_gqa_B2_Hq32_Hkv8_T8192.md, with
# the SHA-256 of the kernel's sources (prefill.cu and common.cuh) it was taken with: the figure is
# reported only while those sources are unchanged.
PREFILL_TRAFFIC = {"bytes": 301086208 + 84741376,
                   "sources_sha256": "c685f32cca8987fdfe871078fe20a8e78894b86cec5b727e6b6552f30c9a6827"}
PREFILL_SOURCES = ("prefill.cu", "common.cuh")


def prefill_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for name in PREFILL_SOURCES:
        with open(os.path.join(ROOT, "exact_tiled_attention_attn_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def prefill_traffic():
    if PREFILL_TRAFFIC["bytes"] is None:
        return None
    return PREFILL_TRAFFIC["bytes"] if prefill_sources_sha256() == PREFILL_TRAFFIC["sources_sha256"] else None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


def decode_kernels(splits: int, eb: int) -> str:
    cache = " (E4M3 cache)" if eb == 1 else ""
    if splits == 0:
        return f"decode_balanced_kernel<128,{eb}>{cache} + decode_balanced_merge_kernel<128>"
    return f"decode_split_mma_kernel<128,{eb}>{cache} + decode_combine_kernel<128>"


# ----------------------------------------------------------------------------- clocks

def summarise_clock_samples(samples, t0: float, t1: float, source: str):
    """Median SM clock, highest max clock and the union of the named clock-event reasons over
    the samples (wall time, sm MHz, max MHz, set of reason names) taken between t0 and t1."""
    sm, smax, reasons = [], [], set()
    for ts, mhz, max_mhz, names in samples:
        if t0 <= ts <= t1:
            sm.append(float(mhz))
            smax.append(float(max_mhz))
            reasons.update(names)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
            "reasons": sorted(reasons), "source": source}


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*) and the names reported for them.
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}


def nvml_reason_names(mask: int):
    return {name for bit, name in NVML_REASONS.items() if mask & bit}


class NvmlClockSampler:
    """Polls the SM clock and the clock-event reasons through NVML every `period_s` in a thread.

    Read-only queries (nvmlDeviceGetClockInfo, nvmlDeviceGetMaxClockInfo,
    nvmlDeviceGetCurrentClocksEventReasons); a timed region of a few tens of milliseconds still
    holds several samples, which the 200 ms nvidia-smi loop cannot give. `lib` is the loaded
    libnvidia-ml (a stand-in object in the CPU tests). Raises OSError when NVML is unusable.
    """

    CLOCK_SM = 1

    def __init__(self, uuid: str, lib=None, period_s: float = 0.002):
        import ctypes
        self.ct = ctypes
        self.lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
            self.lib.nvmlShutdown()
            raise OSError("no NVML device with uuid " + uuid)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        if self.reasons_fn is None:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _sample(self):
        ct = self.ct
        mhz, max_mhz, mask = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.handle, self.CLOCK_SM, ct.byref(mhz)) != 0:
            return None
        if self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.CLOCK_SM, ct.byref(max_mhz)) != 0:
            return None
        if self.reasons_fn(self.handle, ct.byref(mask)) != 0:
            return None
        return (time.time(), mhz.value, max_mhz.value, nvml_reason_names(mask.value))

    def _run(self):
        while not self.stop_flag.is_set():
            s = self._sample()
            if s is not None:
                self.samples.append(s)
            self.stop_flag.wait(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self, t0: float, t1: float):
        self.stop_flag.set()
        if self.thread is not None:
            self.thread.join(timeout=2)
        self.lib.nvmlShutdown()
        return summarise_clock_samples(self.samples, t0, t1, f"nvml every {self.period * 1e3:g} ms")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms in a subprocess."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index_or_uuid):
        self.dev = device_index_or_uuid
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    @staticmethod
    def parse(lines):
        """(wall time, csv line) pairs -> samples as summarise_clock_samples takes them."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        out = []
        for ts, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                mhz, max_mhz = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            out.append((ts, mhz, max_mhz, {n for n, v in zip(names, parts[4:8]) if v.lower() == "active"}))
        return out

    def stop(self, t0: float, t1: float):
        """Stop sampling; summarise the samples that arrived between t0 and t1 (wall time)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        return summarise_clock_samples(self.parse(self.lines), t0, t1, "nvidia-smi every 200 ms")


def make_clock_sampler(uuid, local_index):
    """NVML polling when the library answers for this device, else the nvidia-smi loop."""
    if uuid:
        try:
            return NvmlClockSampler(uuid)
        except (OSError, AttributeError):
            pass
    return ClockSampler(uuid if uuid else local_index)


# ----------------------------------------------------------------------------- GPU arm

def _dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of per-rank numbers over the default process group.

    Every rank gets the maximum (the slowest rank sets the whole job's time). With
    no process group, or a single rank, the values come back unchanged.
    """
    import torch
    import torch.distributed as dist
    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(a) for a in t.tolist()]


def whole_job_rate(work_per_rank: float, ms_max: float, world: int) -> float:
    """Units per second of the whole job: every rank did `work_per_rank` units, and the
    job took as long as its slowest rank (`ms_max`)."""
    return world * work_per_rank / (ms_max * 1e-3)


def run_gpu(args):
    import torch
    import exact_tiled_attention_attn_gb300 as attn
    from exact_tiled_attention_attn_gb300.build import build

    world, rank, local = _dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build()
    attn.lib()

    # ---- inputs (seeded, generated on the host, copied once to HBM)
    q, k, v = W.attention_inputs(PREFILL)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    od = torch.empty_like(qd)
    lsed = torch.empty(PREFILL.B, PREFILL.Hq, PREFILL.T, dtype=torch.float32, device=dev)
    x, w = W.norm_inputs(NORM)
    xd, wd = x.to(dev), w.to(dev)
    yd = torch.empty_like(xd)
    dq, dkc, dvc, dsl = W.decode_inputs(DECODE)
    dqd, dkcd, dvcd, dsld = dq.to(dev), dkc.to(dev), dvc.to(dev), dsl.to(dev)
    del dkc, dvc
    # 0 = the balanced schedule (equal key ranges over persistent CTAs, then a merge of the cut
    # segments); N >= 1 = flash-decoding with N splits per sequence
    splits = args.splits if args.splits is not None else 0
    ws = torch.empty(attn.decode_workspace_size(DECODE.B, DECODE.Hq, DECODE.d, splits), dtype=torch.uint8,
                     device=dev)
    dod = torch.empty_like(dqd)
    dlse = torch.empty(DECODE.B, DECODE.Hq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        attn.rmsnorm(xd, wd, eps=NORM.eps, out=yd)
        if ev is not None:
            ev[1].record(stream)
        attn.fwd(qd, kd, vd, causal=True, scale=PREFILL.scale, out=od, lse=lsed)
        if ev is not None:
            ev[2].record(stream)
        attn.decode(dqd, dkcd, dvcd, dsld, scale=DECODE.scale, num_splits=splits, workspace=ws, out=dod,
                    lse=dlse)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        uuid = None
    sampler = make_clock_sampler(uuid, local)
    sampler.start()
    time.sleep(0.4)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = attn.kernel_launches()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    launches = attn.kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(wall0, wall1)
    assert attn.last_device_error() == 0

    total_ms = t_start.elapsed_time(t_end)
    norm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    dec_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    total_ms, fwd_ms, dec_ms, norm_ms = max_over_ranks([total_ms, fwd_ms, dec_ms, norm_ms], dev)

    peaks = _peaks()
    flops = PREFILL.flops()
    sum_l = int(dsl.sum().item())
    dec_bytes = (4 * DECODE.Hkv * DECODE.d * sum_l + 2 * DECODE.B * DECODE.Hq * DECODE.d * 2
                 + DECODE.B * DECODE.Hq * 4 + DECODE.B * 4)
    norm_bytes = NORM.hbm_bytes()
    prefill_tflops = flops / (fwd_ms * 1e-3) / 1e12
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    norm_gbs = norm_bytes / (norm_ms * 1e-3) / 1e9
    value = whole_job_rate(flops, fwd_ms, world) / 1e12

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        lh = torch.empty(lsed.shape, dtype=torch.float32).pin_memory()
        qd2, kd2, vd2 = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)

        def e2e_step():
            qd2.copy_(qh, non_blocking=True)
            kd2.copy_(kh, non_blocking=True)
            vd2.copy_(vh, non_blocking=True)
            o2, l2 = attn.fwd(qd2, kd2, vd2, causal=True, scale=PREFILL.scale, out=od, lse=lsed)
            oh.copy_(o2, non_blocking=True)
            lh.copy_(l2, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        # up to 30 steps: the pipelined form below fills and drains once per timed run, and a
        # serving loop runs many steps (10 steps: 1.247 ms per step, 30 steps: 1.167 ms)
        n_e2e = max(3, min(args.steps, 30))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        serial_ms = max_over_ranks([a.elapsed_time(b) / n_e2e], dev)[0]
        h2d = (q.numel() + k.numel() + v.numel()) * 2
        d2h = q.numel() * 2 + lsed.numel() * 4

        # The same steps pipelined the way a serving loop runs them: two sets of device buffers,
        # the host-to-device copies of step i + 1 on one stream and the device-to-host copies of
        # step i - 1 on another while step i computes; every step still moves all of its bytes.
        bufs = [(qd2, kd2, vd2, od, lsed),
                (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd), torch.empty_like(od),
                 torch.empty_like(lsed))]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]

        def pipelined(nsteps):
            for i in range(nsteps):
                bi = i & 1
                qb, kb, vb, ob, lb = bufs[bi]
                with torch.cuda.stream(s_in):
                    if used[bi]:
                        s_in.wait_event(comp_done[bi])   # step i - 2 has read q, k, v of this set
                    qb.copy_(qh, non_blocking=True)
                    kb.copy_(kh, non_blocking=True)
                    vb.copy_(vh, non_blocking=True)
                    in_done[bi].record(s_in)
                stream.wait_event(in_done[bi])
                if used[bi]:
                    stream.wait_event(out_done[bi])      # step i - 2's O and LSE have been read back
                attn.fwd(qb, kb, vb, causal=True, scale=PREFILL.scale, out=ob, lse=lb)
                comp_done[bi].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[bi])
                    oh.copy_(ob, non_blocking=True)
                    lh.copy_(lb, non_blocking=True)
                    out_done[bi].record(s_out)
                used[bi] = True

        pipelined(max(2, args.warmup))
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_stream(stream)
        pipelined(n_e2e)
        stream.wait_stream(s_out)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks([a.elapsed_time(b) / n_e2e], dev)[0]
        e2e = {"value": round(whole_job_rate(flops, e2e_ms, world) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "steps": n_e2e,
               "how": "pinned host buffers; H2D, attn_fwd and D2H of consecutive steps on three streams with "
                      "two device buffer sets; the timed steps include the pipeline's one fill and drain",
               "serial": {"value": round(whole_job_rate(flops, serial_ms, world) / 1e12, 2),
                          "ms_per_step": round(serial_ms, 4),
                          "how": "H2D, attn_fwd, D2H of each step one after another on one stream"}}
        del bufs

    # ---- the other two prefill configurations, each timed on its own outside the step: every
    #      launch between two events, L2 flushed before it (the causal GQA B1 inputs, 34 MB, fit
    #      in L2); the median launch is reported
    prefill_other = {}
    if not args.no_prefill_configs:
        flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
        for key, shp in (("prefill_c2", W.MHA_GPT2), ("prefill_c3", W.GQA_QWEN)):
            pq, pk, pv = [t.to(dev) for t in W.attention_inputs(shp)]
            po = torch.empty_like(pq)
            pl = torch.empty(shp.B, shp.Hq, shp.T, dtype=torch.float32, device=dev)
            pws = torch.empty(attn.fwd_workspace_size(shp.d), dtype=torch.uint8, device=dev)
            for _ in range(3):
                attn.fwd(pq, pk, pv, causal=shp.causal, scale=shp.scale, out=po, lse=pl, workspace=pws)
            n_launch0 = attn.kernel_launches()
            attn.fwd(pq, pk, pv, causal=shp.causal, scale=shp.scale, out=po, lse=pl, workspace=pws)
            launches_per_call = attn.kernel_launches() - n_launch0
            tms = []
            for _ in range(20):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                attn.fwd(pq, pk, pv, causal=shp.causal, scale=shp.scale, out=po, lse=pl, workspace=pws)
                b.record(stream)
                torch.cuda.synchronize()
                tms.append(a.elapsed_time(b))
            assert attn.last_device_error() == 0
            tms.sort()
            p_ms = max_over_ranks([tms[len(tms) // 2]], dev)[0]
            p_tf = shp.flops() / (p_ms * 1e-3) / 1e12
            prefill_other[key] = {"value": round(p_tf, 2), "unit": "TFLOP/s", "bound": "tensor",
                                  "peak": peaks["bf16"], "frac": round(p_tf / peaks["bf16"], 4),
                                  "ms": round(p_ms, 4), "ms_p10_p90": [round(tms[2], 4), round(tms[-3], 4)],
                                  "flops_per_launch": shp.flops(), "workload": shp.name,
                                  "kernel": f"attn_fwd_kernel<{shp.d}>" + (
                                      f" + attn_fwd_merge_kernel<{shp.d}> (last round's units split along the keys)"
                                      if launches_per_call == 2 else ""),
                                  "launches_per_call": launches_per_call,
                                  "timing": "median of 20 calls, each between two events, L2 flushed before it"}
            del pq, pk, pv, po, pl, pws
        del flush

    # ---- RMSNorm at growing T: the workload's 16.8 MB is launch- and latency-bound,
    #      the sweep shows the kernel's sustained bandwidth (L2 flushed before each launch)
    norm_sweep = []
    if not args.no_e2e:
        flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
        for Ts in (4096, 65536, 262144):
            xs = torch.randn(Ts, NORM.D, device=dev).to(torch.bfloat16)
            ys = torch.empty_like(xs)
            tms = []
            for _ in range(8):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                attn.rmsnorm(xs, wd, eps=NORM.eps, out=ys)
                b.record(stream)
                torch.cuda.synchronize()
                tms.append(a.elapsed_time(b))
            tms.sort()
            bytes_s = 4 * Ts * NORM.D + 2 * NORM.D
            norm_sweep.append({"T": Ts, "us": round(1e3 * tms[len(tms) // 2], 2),
                               "GB/s": round(bytes_s / (tms[len(tms) // 2] * 1e-3) / 1e9, 1)})
            del xs, ys
        del flush

    # ---- RMSNorm X[4096, 1024] timed the way a kernel this short is timed: a CUDA graph of
    #      back-to-back launches over 32 distinct (x, y) pairs (537 MB, so every launch reads x
    #      from HBM), divided by the launches; the in-step number above is one launch between
    #      two events and carries the launch gap
    nbuf, reps = 32, 3
    xs = [torch.randn(NORM.T, NORM.D, device=dev).to(torch.bfloat16) for _ in range(nbuf)]
    ys = [torch.empty_like(xs[0]) for _ in range(nbuf)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            for i in range(nbuf):
                attn.rmsnorm(xs[i], wd, eps=NORM.eps, out=ys[i])
    torch.cuda.synchronize()
    gms = []
    for _ in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        gms.append(a.elapsed_time(b) / (reps * nbuf))
    assert attn.last_device_error() == 0
    g_ms = max_over_ranks([sorted(gms)[1]], dev)[0]
    norm_graph = {"launches": reps * nbuf, "buffers": nbuf, "us_per_launch": round(1e3 * g_ms, 3),
                  "GB/s": round(norm_bytes / (g_ms * 1e-3) / 1e9, 1),
                  "frac": round(norm_bytes / (g_ms * 1e-3) / 1e9 / peaks["hbm"], 4)}
    del g, xs, ys

    # ---- residual-add RMSNorm on the same X[4096, 1024] (h = bf16(x + r), y = RMSNorm(h) w): reads
    #      x and r, writes h and y; L2 flushed before each launch
    res_line = None
    if not args.no_e2e:
        flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
        rd = torch.randn(NORM.T, NORM.D, device=dev).to(torch.bfloat16)
        hd = torch.empty_like(xd)
        tms = []
        for _ in range(8):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            attn.rmsnorm_residual(xd, rd, wd, eps=NORM.eps, out=yd, h=hd)
            b.record(stream)
            torch.cuda.synchronize()
            tms.append(a.elapsed_time(b))
        tms.sort()
        r_ms = max_over_ranks([tms[len(tms) // 2]], dev)[0]
        r_bytes = 8 * NORM.T * NORM.D + 2 * NORM.D
        del flush, rd, hd
        # the same graph form as the plain RMSNorm: back-to-back launches over 16 distinct
        # (x, r, y, h) sets (537 MB), so every launch reads x and r from HBM
        nset, rreps = 16, 3
        sets = [(torch.randn(NORM.T, NORM.D, device=dev).to(torch.bfloat16),
                 torch.randn(NORM.T, NORM.D, device=dev).to(torch.bfloat16),
                 torch.empty(NORM.T, NORM.D, dtype=torch.bfloat16, device=dev),
                 torch.empty(NORM.T, NORM.D, dtype=torch.bfloat16, device=dev)) for _ in range(nset)]
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(rreps):
                for xs_, rs_, ys_, hs_ in sets:
                    attn.rmsnorm_residual(xs_, rs_, wd, eps=NORM.eps, out=ys_, h=hs_)
        torch.cuda.synchronize()
        grs = []
        for _ in range(4):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            gr.replay()
            b.record(stream)
            torch.cuda.synchronize()
            grs.append(a.elapsed_time(b) / (rreps * nset))
        assert attn.last_device_error() == 0
        rg_ms = max_over_ranks([sorted(grs)[1]], dev)[0]
        del gr, sets
        res_line = {"value": round(r_bytes / (rg_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "bound": "hbm",
                    "peak": peaks["hbm"], "frac": round(r_bytes / (rg_ms * 1e-3) / 1e9 / peaks["hbm"], 4),
                    "us": round(1e3 * rg_ms, 3), "bytes_per_launch": r_bytes, "workload": "X, R [4096, 1024]",
                    "timing": f"CUDA graph of {rreps * nset} back-to-back launches over {nset} distinct "
                              "(x, r, y, h) sets (537 MB), divided by the launches",
                    "single_launch": {"us": round(1e3 * r_ms, 2),
                                      "GB/s": round(r_bytes / (r_ms * 1e-3) / 1e9, 1),
                                      "timing": "one launch between two events, L2 flushed before it"}}

    # ---- the bf16 decode of the step, 20 launches back to back (consecutive decode steps of a
    #      serving loop; the in-step number above follows the prefill, whose writes are still
    #      in L2)
    nb = 20
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(nb):
        attn.decode(dqd, dkcd, dvcd, dsld, scale=DECODE.scale, num_splits=splits, workspace=ws, out=dod, lse=dlse)
    b.record(stream)
    torch.cuda.synchronize()
    assert attn.last_device_error() == 0
    db_ms = max_over_ranks([a.elapsed_time(b) / nb], dev)[0]
    dec_b2b = {"value": round(dec_bytes / (db_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
               "frac": round(dec_bytes / (db_ms * 1e-3) / 1e9 / peaks["hbm"], 4), "ms": round(db_ms, 4),
               "timing": f"{nb} launches back to back between two events"}

    # ---- FP8 (E4M3) KV-cache decode on the same workload (its own timing, outside the step):
    #      the cache is quantised once on the GPU, then only the 1-byte codes are streamed
    dec8 = None
    if not args.no_fp8:
        kq, ks = attn.kv_quantize_fp8(dkcd)
        vq, vs = attn.kv_quantize_fp8(dvcd)
        for _ in range(3):
            attn.decode_fp8(dqd, kq, vq, ks, vs, dsld, scale=DECODE.scale, num_splits=splits, workspace=ws,
                            out=dod, lse=dlse)
        torch.cuda.synchronize()
        n8 = 20
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n8):
            attn.decode_fp8(dqd, kq, vq, ks, vs, dsld, scale=DECODE.scale, num_splits=splits, workspace=ws,
                            out=dod, lse=dlse)
        b.record(stream)
        torch.cuda.synchronize()
        assert attn.last_device_error() == 0
        d8_ms = max_over_ranks([a.elapsed_time(b) / n8], dev)[0]
        d8_bytes = (2 * DECODE.Hkv * DECODE.d * sum_l + 2 * DECODE.B * DECODE.Hq * DECODE.d * 2
                    + DECODE.B * DECODE.Hq * 4 + DECODE.B * 4 + 2 * DECODE.B * DECODE.Hkv * 4)
        d8_gbs = d8_bytes / (d8_ms * 1e-3) / 1e9
        dec8 = {"value": round(d8_gbs, 1), "unit": "GB/s", "bound": "hbm", "peak": peaks["hbm"],
                "frac": round(d8_gbs / peaks["hbm"], 4), "ms": round(d8_ms, 4), "bytes_per_launch": d8_bytes,
                "vs_bf16_decode_time": round(dec_ms / d8_ms, 3),
                "kernels": decode_kernels(splits, 1),
                "timing": f"{n8} launches back to back between two events",
                "num_splits": splits}
        del kq, vq

    # ---- short-context decode (B16 Hq32 Hkv8 d128, L ~ U[1024, 2048]): launch overhead is visible here;
    #      20 steps launched one by one vs the same 20 steps captured once in a CUDA graph and replayed
    short = None
    if not args.no_e2e:
        sshp = W.DecodeShape("short", DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.d, 1024, 2048, DECODE.seed)
        sq, skc, svc, ssl = [t.to(dev) for t in W.decode_inputs(sshp)]
        sS = splits  # the balanced schedule by default (graph replay: 23.3 us per step against 24.7 with 2 splits)
        sws = torch.empty(attn.decode_workspace_size(sshp.B, sshp.Hq, sshp.d, sS), dtype=torch.uint8, device=dev)
        so, sl_ = torch.empty_like(sq), torch.empty(sshp.B, sshp.Hq, dtype=torch.float32, device=dev)
        nstep = 20

        def short_steps():
            for _ in range(nstep):
                attn.decode(sq, skc, svc, ssl, scale=sshp.scale, num_splits=sS, workspace=sws, out=so, lse=sl_)

        for _ in range(3):
            short_steps()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(stream)
        short_steps()
        b.record(stream)
        torch.cuda.synchronize()
        host_eager = (time.perf_counter() - t0) / nstep
        eager_ms = a.elapsed_time(b) / nstep
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            short_steps()
        g.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        host_graph = (time.perf_counter() - t0) / nstep
        graph_ms = a.elapsed_time(b) / nstep
        s_bytes = 4 * sshp.Hkv * sshp.d * int(ssl.sum().item())
        short = {"workload": "flash-decoding B16 Hq32 Hkv8 d128 L~U[1024,2048]", "num_splits": sS,
                 "kernels": decode_kernels(sS, 2),
                 "eager_us_per_step": round(1e3 * eager_ms, 2), "graph_us_per_step": round(1e3 * graph_ms, 2),
                 "eager_GB/s": round(s_bytes / (eager_ms * 1e-3) / 1e9, 1),
                 "graph_GB/s": round(s_bytes / (graph_ms * 1e-3) / 1e9, 1),
                 "host_wall_us_per_step_eager": round(1e6 * host_eager, 2),
                 "host_wall_us_per_step_graph": round(1e6 * host_graph, 2)}
        del g, sq, skc, svc, sws

    # ---- backward pass on the prefill workload (its own timing, outside the step). Algorithmic
    #      FLOPs: the 5 GEMMs of the gradients, 2.5x the forward's (the kernels recompute S and
    #      dP for dQ: 7 GEMMs executed)
    bwd_line = None
    if not args.no_bwd:
        dod = W.grad_output(PREFILL.B, PREFILL.Hq, PREFILL.T, PREFILL.d, PREFILL.seed).to(dev)
        gq, gk, gv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        bws = torch.empty(attn.lib().attn_bwd_workspace_size(PREFILL.B, PREFILL.Hq, PREFILL.T), dtype=torch.uint8,
                          device=dev)
        attn.fwd(qd, kd, vd, causal=True, scale=PREFILL.scale, out=od, lse=lsed)

        def bwd_once():
            attn.bwd(qd, kd, vd, od, lsed, dod, causal=True, scale=PREFILL.scale, dq=gq, dk=gk, dv=gv, workspace=bws)

        for _ in range(3):
            bwd_once()
        torch.cuda.synchronize()
        # three timed regions of nb calls each; the median region is reported (a single region of
        # back-to-back calls is exposed to a transient clock drop)
        nb = 8
        regions = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(nb):
                bwd_once()
            b.record(stream)
            torch.cuda.synchronize()
            regions.append(a.elapsed_time(b) / nb)
        assert attn.last_device_error() == 0
        regions.sort()
        b_ms = max_over_ranks([regions[1]], dev)[0]
        b_flops = 2.5 * flops
        b_tf = b_flops / (b_ms * 1e-3) / 1e12
        bwd_line = {"value": round(b_tf, 2), "unit": "TFLOP/s", "bound": "tensor", "peak": peaks["bf16"],
                    "frac": round(b_tf / peaks["bf16"], 4), "ms": round(b_ms, 4), "flops_per_launch": b_flops,
                    "ms_regions": [round(x, 4) for x in regions],
                    "timing": f"median of 3 regions of {nb} calls back to back, each between two events",
                    "workload": PREFILL.name,
                    "kernels": "bwd_delta_kernel<128> + bwd_dkdv_kernel<128> + bwd_dq_kernel<128>"}
        del dod, gq, gk, gv, bws

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_heads)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16; decode lengths ~U[8192,32768] seed 1004)",
            "config": {"workload": WORKLOAD, "prefill_ms": round(fwd_ms, 4), "decode_ms": round(dec_ms, 4),
                       "rmsnorm_ms": round(norm_ms, 4), "decode_num_splits": splits,
                       "decode_sum_lengths": sum_l,
                       "l2": "inputs larger than L2: prefill reads 201 MB, decode streams "
                             f"{dec_bytes / 1e9:.2f} GB between reuses of any buffer",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel<128>",
                         "achieved": round(prefill_tflops, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": round(prefill_tflops / peaks["bf16"], 4),
                         "traffic": args.traffic if args.traffic is not None else prefill_traffic(),
                         "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                         "algorithmic_bytes": PREFILL.hbm_bytes(),
                         "peak_source": f"{peaks['source']} bf16 (burst)",
                         "flops_per_launch": flops},
            "decode": {"value": round(dec_gbs, 1), "unit": "GB/s", "bound": "hbm", "peak": peaks["hbm"],
                       "frac": round(dec_gbs / peaks["hbm"], 4), "bytes_per_launch": dec_bytes,
                       "kernels": decode_kernels(splits, 2),
                       "num_splits": splits,
                       "timing": "one launch inside the step, after the prefill (between two events)",
                       "back_to_back": dec_b2b},
            "rmsnorm": {"value": norm_graph["GB/s"], "unit": "GB/s", "bound": "hbm", "peak": peaks["hbm"],
                        "frac": norm_graph["frac"], "bytes_per_launch": norm_bytes,
                        "timing": "a kernel this short is timed as a CUDA graph of back-to-back launches over "
                                  "32 distinct (x, y) pairs (537 MB, x always read from HBM), divided by the "
                                  "launches",
                        "graph_back_to_back": norm_graph,
                        "single_launch_in_step": {"value": round(norm_gbs, 1), "us": round(1e3 * norm_ms, 2),
                                                  "frac": round(norm_gbs / peaks["hbm"], 4),
                                                  "timing": "one launch between two events inside the step"},
                        "sweep_D1024": norm_sweep},
            "prefill_c2": prefill_other.get("prefill_c2"),
            "prefill_c3": prefill_other.get("prefill_c3"),
            "decode_fp8": dec8,
            "rmsnorm_residual": res_line,
            "decode_short_context": short,
            "backward": bwd_line,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS = {}


def _oracle_inputs():
    """float64 copies of the prefill workload's inputs (generated once per process)."""
    if not _ORACLE_INPUTS:
        q, k, v = W.attention_inputs(PREFILL)
        _ORACLE_INPUTS.update(q=q, k=k, v=v)
    return _ORACLE_INPUTS["q"], _ORACLE_INPUTS["k"], _ORACLE_INPUTS["v"]


def _oracle_sample(heads):
    """The oracle on every query row of the given (batch, head) pairs of the prefill workload.

    Returns (flops, seconds); only the oracle call is timed.
    """
    import oracle
    q, k, v = _oracle_inputs()
    g = PREFILL.Hq // PREFILL.Hkv
    T = PREFILL.T
    rows = np.arange(T)
    flops, dt = 0.0, 0.0
    for b, h in heads:
        qh = W.to_f64(q[b, h])[None, None]
        kh = W.to_f64(k[b, h // g])[None, None]
        vh = W.to_f64(v[b, h // g])[None, None]
        t0 = time.perf_counter()
        oracle.attention_rows(qh, kh, vh, 0, 0, rows, True, PREFILL.scale)
        dt += time.perf_counter() - t0
        flops += 4.0 * PREFILL.d * T * (T + 1) / 2
    return flops, dt


def cpu_baseline(n_heads: int):
    heads = [(0, h) for h in range(n_heads)]
    flops, dt = _oracle_sample(heads)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"float64 three-pass oracle on all {PREFILL.T} causal query rows of {n_heads} of the "
                      f"{PREFILL.B * PREFILL.Hq} (batch, head) pairs of the prefill workload (d={PREFILL.d}); "
                      f"{flops / 1e9:.1f} GFLOP in {dt:.2f} s; numpy BLAS with its default threads "
                      "(all host cores)"}


def _oracle_rows(b: int, h: int, rows: int):
    """The oracle on the last `rows` causal query rows of one (batch, head) pair. Returns (flops, s)."""
    import oracle
    q, k, v = _oracle_inputs()
    g = PREFILL.Hq // PREFILL.Hkv
    T = PREFILL.T
    sel = np.arange(T - rows, T)
    qh = W.to_f64(q[b, h])[None, None]
    kh = W.to_f64(k[b, h // g])[None, None]
    vh = W.to_f64(v[b, h // g])[None, None]
    t0 = time.perf_counter()
    oracle.attention_rows(qh, kh, vh, 0, 0, sel, True, PREFILL.scale)
    return 4.0 * PREFILL.d * float(np.sum(sel + 1)), time.perf_counter() - t0


def run_reference(args):
    world, rank, _ = _dist_setup()
    if rank != 0:
        return
    _oracle_inputs()
    # Size each step's sample so the whole run stays near --ref-seconds of oracle time.
    _, t_cal = _oracle_rows(0, 0, 256)
    per_step = args.ref_seconds / (args.steps + args.warmup)
    rows = int(max(16, min(PREFILL.T, 256 * per_step / max(t_cal, 1e-6))))
    for i in range(args.warmup):
        _oracle_rows(0, i % PREFILL.Hq, rows)
    tot_f, tot_t = 0.0, 0.0
    for i in range(args.steps):
        f, t = _oracle_rows(i // PREFILL.Hq % PREFILL.B, i % PREFILL.Hq, rows)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    sample = (f"each step: float64 three-pass oracle on the last {rows} causal query rows (of {PREFILL.T}) of one "
              "(batch, head) pair of the prefill workload; numpy BLAS with its default threads")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_t / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 decoded to float64)",
        "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--splits", type=int, default=None,
                    help="decode split count; 0 (the default) = the balanced schedule")
    ap.add_argument("--cpu-heads", type=int, default=8, help="(batch, head) pairs in the CPU-baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="approximate oracle time of a whole --impl reference run")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per prefill launch from an ncu capture, if known for this build")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 KV-cache decode line")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward-pass line")
    ap.add_argument("--no-prefill-configs", action="store_true",
                    help="skip the lines for the non-causal MHA and the causal GQA B1 prefill configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
