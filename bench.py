#!/usr/bin/env python
"""Training-step throughput of the B300 GPT-2 library (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one whole training step -- forward of every layer, fused softmax +
cross-entropy, zero_grad, backward of every layer, AdamW over the flat buffer -- on
one fresh batch of the GPT-2 124M bf16 workload (B=16, T=1024, 16384 tokens, Zipf
s=1.1 token stream, lr 6e-4, wd 0.1).  Weights are random-init from the seeded
recipe; batches are synthetic and resident in HBM before timing starts.

For N > 1 (torchrun) every rank trains its own replica on its own data (weak
scaling, no collective): the data-parallel gradient exchange is not built, because
every run of this library has one GPU.  ``--impl reference`` times the CPU oracle (the
deliberately slow plain program) on the host cores, on a bounded sample of the same
workload.
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

WORKLOAD = "gpt2_124m_bf16_b16_t1024"
METRIC = "GPT-2 124M train tokens/sec (fwd+bwd+AdamW) on 1 B300; MFU; kernel % roofline"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--optimizer", choices=["adamw", "muon"], default="adamw",
                    help="muon: Muon (5 Newton-Schulz steps) on the block matrices, AdamW on the rest")
    ap.add_argument("--windows", type=int, default=5,
                    help="timed windows of K steps (the first is the headline; all give the spread)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ------------------------------------------------------------------------ model flops
def mfu_flops_per_token(shape, T):
    """6N + 12 L C T per token, N = real parameter count (V token rows)."""
    C, L = shape.channels, shape.num_layers
    N = (shape.vocab_size * C + shape.max_seq_len * C
         + L * (12 * C * C + 13 * C) + 2 * C)
    return 6.0 * N + 12.0 * L * C * T, N


# ------------------------------------------------------------------------ clocks
class _Nvml:
    """The few NVML calls the clock sampler needs, through ctypes on the driver's
    libnvidia-ml (present wherever the GPU driver is)."""
    CLOCK_SM = 1
    REASONS = (("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40),
               ("sw_power_cap", 0x4), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, cuda_index):
        import ctypes
        import torch
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        pr = torch.cuda.get_device_properties(cuda_index)
        bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
        self.h = ctypes.c_void_p()
        rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h))
        if rc != 0:
            n = ctypes.c_uint(0)
            self.lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
            if n.value != 1 or self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                raise RuntimeError(f"no NVML handle for {bus.decode()} (rc {rc})")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def max_sm(self):
        v = self.c.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.c.byref(v))
        return float(v.value)

    def sample(self):
        c = self.c
        sm, pw, rs = c.c_uint(0), c.c_uint(0), c.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, c.byref(sm)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(pw))
        self.reasons_fn(self.h, c.byref(rs))
        return float(sm.value), pw.value / 1000.0, {n for n, b in self.REASONS if rs.value & b}


class ClockSampler:
    """SM clock, power and clock-event reasons of this process's GPU, sampled every 20 ms
    through NVML (ctypes on libnvidia-ml; the GPU is found by its PCI bus id, so the NVML
    index need not match the CUDA one) from a background thread while the timed region
    runs; nvidia-smi at 200 ms when NVML cannot be opened."""

    NV_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index):
        self.cuda_index = cuda_index
        self.samples = []          # (sm_mhz, max_mhz, power_w, set of reasons, host time)
        self.stop_ev = threading.Event()
        self.t = None
        self.proc = None
        self.nv = None
        self.note = None
        try:
            self.nv = _Nvml(cuda_index)
        except Exception as e:
            self.nv = None
            self.note = f"NVML unavailable ({e!r:.160}); nvidia-smi at 200 ms"

    def _poll_nvml(self):
        mx = self.nv.max_sm()
        while not self.stop_ev.is_set():
            try:
                r = self.nv.sample()
                if r is not None:
                    self.samples.append((r[0], mx, r[1], r[2], time.perf_counter()))
            except Exception:
                pass
            self.stop_ev.wait(0.02)

    def _read_smi(self):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.proc.stdout:
            f = [x.strip() for x in line.strip().split(",")]
            if len(f) < 9:
                continue
            try:
                rs = {n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")}
                self.samples.append((float(f[1]), float(f[2]), float(f[3]), rs, time.perf_counter()))
            except ValueError:
                continue

    def start(self):
        if self.nv is not None:
            self.t = threading.Thread(target=self._poll_nvml, daemon=True)
            self.t.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={self.NV_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read_smi, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def window(self, t0, t1):
        """Median SM clock and the reasons seen between host times t0 and t1."""
        w = [x for x in self.samples if t0 <= x[4] <= t1]
        if not w:
            return {"sm_mhz": None, "samples": 0, "reasons": []}
        return {"sm_mhz": statistics.median(x[0] for x in w), "samples": len(w),
                "reasons": sorted(set().union(*[x[3] for x in w]))}

    def stop(self):
        self.stop_ev.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=5)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0,
                    "source": self.note or "nvml"}
        sm = [x[0] for x in self.samples]
        reasons = set().union(*[x[3] for x in self.samples])
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                "sm_max_mhz": max(x[1] for x in self.samples),
                "power_w_median": statistics.median(x[2] for x in self.samples),
                "power_w_max": max(x[2] for x in self.samples),
                "samples": len(sm), "source": "nvml, 20 ms" if self.nv is not None else self.note,
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------ ncu traffic
TRAFFIC_PROFILE = os.path.join("profiles", "matmul_dram_traffic_gpt2_124m_bf16_b16_t1024.md")


def matmul_traffic(workload):
    """DRAM bytes per matmul launch from the committed ncu summary of this workload, or
    (None, why) when there is none or the kernel's sources changed since the capture."""
    import hashlib
    if workload != WORKLOAD:
        return None, "no capture for this workload"
    try:
        with open(os.path.join(ROOT, TRAFFIC_PROFILE)) as f:
            kv = dict(l.split(":", 1) for l in f.read().splitlines() if l.startswith(
                ("traffic_bytes_per_launch:", "kernel_sources:", "sources_sha256:")))
        h = hashlib.sha256()
        for src in kv["kernel_sources"].split():
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
    except (OSError, KeyError, ValueError) as e:
        return None, f"no traffic capture ({e!r:.80})"
    if h.hexdigest() != kv["sources_sha256"].strip():
        return None, "the matmul kernel changed since the DRAM counters were taken"
    return float(kv["traffic_bytes_per_launch"]), f"{TRAFFIC_PROFILE} (ncu dram__bytes_read.sum + dram__bytes_write.sum, mean per launch of the family in one step)"


# ------------------------------------------------------------------------ CPU oracle leg
def oracle_tokens_per_s(w, sample_B, sample_T, steps, warmup=0, seed_offset=0):
    """Time the CPU oracle (float32, as the pages' program) on a bounded sample of the
    workload: `steps` whole training steps at (sample_B, sample_T)."""
    import numpy as np
    from oracle import gpt2_oracle as O
    from step_gpt_train_03_b300 import synth
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    o = O.from_shape(w.shape, np.float32)
    o.keep_preatt = False
    o.load(synth.init_params(w.shape, w.seed))
    batches = synth.zipf_batches(w.shape.vocab_size, sample_B, sample_T, warmup + steps, w.seed + 100 + seed_offset)
    per = []
    for i, (tok, tgt) in enumerate(batches):
        t0 = time.perf_counter()
        o.step(tok, tgt, w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, i + 1)
        dt = time.perf_counter() - t0
        if i >= warmup:
            per.append(dt)
    total = sum(per)
    return sample_B * sample_T * len(per) / total, cores, total, per


def reference_arm(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from step_gpt_train_03_b300 import synth
    w = synth.WORKLOADS[args.workload]
    # each step a bounded sample (one sequence), shorter as the step count grows, so the
    # whole run stays within a few minutes of host time
    n = args.steps + args.warmup
    sB, sT = 1, min(512 if n <= 13 else 256 if n <= 26 else 128, w.shape.max_seq_len)
    tps, cores, total, per = oracle_tokens_per_s(w, sB, sT, args.steps, args.warmup)
    sample = (f"{args.steps} timed whole steps (after {args.warmup} warm-up) of the fp32 CPU oracle "
              f"on the {w.name} model at B={sB}, T={sT} ({sB * sT} tokens each)")
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / len(per),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Zipf s=1.1 token stream, random-init weights)",
        "config": {"workload": w.name, "global_batch": w.B, "seq_len": w.T, "parallelism": "none (CPU)"},
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------ our arm
def ours(args):
    import numpy as np
    import torch
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    from step_gpt_train_03_b300 import build, synth
    if rank == 0:
        build.build()
    barrier()
    from step_gpt_train_03_b300 import gpt2lib as G

    w = synth.WORKLOADS[args.workload]
    B, T = w.B, w.T
    BT = B * T
    stream = torch.cuda.Stream()
    prec = w.precision                      # "bf16" (fp32 master weights) or "fp32"
    m = G.GPT2(w.shape, B, T, prec, stream=stream)
    m.load_params(synth.init_params(w.shape, w.seed))
    n_batches = args.warmup + args.steps
    host = synth.zipf_batches(w.shape.vocab_size, B, T, n_batches, w.seed + 7919 * rank)
    toks = torch.as_tensor(np.stack([b[0] for b in host])).cuda()
    tgts = torch.as_tensor(np.stack([b[1] for b in host])).cuda()
    hp = (w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    torch.cuda.synchronize()

    def step(i, t):
        if args.optimizer == "muon":
            # forward, backward, then Muon + AdamW: one CUDA graph launch once captured
            m.step_muon_device(toks[i], tgts[i], 0.02, 0.95, 5, *hp, t, want_loss=False)
            return
        # the library's whole-step call: one CUDA graph launch once the shape is captured
        m.step_device(toks[i], tgts[i], *hp, t, want_loss=False)

    # warm-up (W >= 3 steps): one untraced step (the first step of the shape: lazy set-up,
    # kernel by kernel), then W-2 steps traced in full (every kernel class's share of a
    # warm step, launched kernel by kernel), then one untraced step that captures the
    # step graph the timed region replays
    n_traced = max(1, args.warmup - 2)
    G.profile_enable([])
    with torch.cuda.stream(stream):
        step(0, 1)
    stream.synchronize()
    G.profile_enable(None)
    G.profile_reset()
    with torch.cuda.stream(stream):
        for i in range(1, 1 + n_traced):
            step(i % n_batches, i + 1)
    stream.synchronize()
    m.check()
    warm_prof = G.profile_read()
    G.profile_reset()
    G.profile_enable([])
    with torch.cuda.stream(stream):
        for i in range(1 + n_traced, max(args.warmup, 2 + n_traced)):
            step(i % n_batches, i + 1)
    stream.synchronize()
    m.check()
    shares = {k: v["ms"] for k, v in warm_prof.items()}
    total_ms = sum(shares.values()) or 1.0
    # the dominant kernel: the class family with the largest traced time
    families = {"matmul": ["matmul_forward", "matmul_backward_dx", "matmul_backward_dw"]}
    fam_ms = {"matmul": sum(shares[c] for c in families["matmul"])}
    for c, v in shares.items():
        if c not in families["matmul"]:
            fam_ms[c] = v
    dominant = max(fam_ms, key=fam_ms.get)
    dom_classes = families.get(dominant, [dominant])
    # the timed region: K untraced steps (the headline), then more windows of K steps
    # each, timed the same way, for the run-to-run spread
    G.profile_enable([])
    clocks = ClockSampler(local_rank)
    launches0 = G.kernel_launches()
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    win_ms, win_clk = [], []
    t_next = max(args.warmup, 2 + n_traced)
    for wi in range(max(1, args.windows)):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if wi > 0:
            barrier()
            torch.cuda.synchronize()
        h0 = time.perf_counter()
        start.record(stream)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                step((args.warmup + i) % n_batches, t_next + 1)
                t_next += 1
        end.record(stream)
        end.synchronize()
        torch.cuda.synchronize()
        h1 = time.perf_counter()
        win_ms.append(start.elapsed_time(end))
        win_clk.append(clocks.window(h0, h1))
        if wi == 0:
            barrier()
            launches = G.kernel_launches() - launches0
    clk = clocks.stop()
    clk["headline_window"] = win_clk[0]
    ms = win_ms[0]
    m.check()
    # the roofline pass: the same K steps again, CUDA events around every launch of the
    # dominant kernel family on the step's stream (events between launches add gaps, so
    # this pass is kept out of the headline)
    G.profile_enable(dom_classes)
    G.profile_reset()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            step(args.warmup + i, t_next + 1)
            t_next += 1
    t_end.record(stream)
    t_end.synchronize()
    ms_traced = t_start.elapsed_time(t_end)
    m.check()
    live = G.profile_read()
    G.profile_enable([])
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = BT * args.steps * world / (ms / 1000.0)

    # end-to-end through the public step call: pinned host tokens in, loss out, per step
    e2e = None
    if not args.no_e2e and args.optimizer == "adamw":
        th = torch.as_tensor(np.stack([b[0] for b in host])).pin_memory()
        gh = torch.as_tensor(np.stack([b[1] for b in host])).pin_memory()
        m.set_stream(stream)
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            m.step_host(th[args.warmup + i], gh[args.warmup + i], *hp, t_next + 1)
            t_next += 1
        e2e_s = time.perf_counter() - t0
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([e2e_s], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_s = float(t.item())
        e2e = {"value": BT * args.steps * world / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": 2 * BT * 4, "d2h_bytes_per_step": 4,
               "call": "gpt2_step_host"}

    if rank != 0:
        return 0

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        src = "measured"
    except OSError:
        peaks = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
        src = "fallback"
    d_ms = sum(live[c]["ms"] for c in dom_classes)
    d_n = sum(live[c]["launches"] for c in dom_classes)
    d_fl = sum(live[c]["flops"] for c in dom_classes)
    d_by = sum(live[c]["bytes"] for c in dom_classes)
    sm_med = clk.get("sm_mhz")
    sm_max = clk.get("sm_max_mhz") or peaks.get("sm_max_mhz", 2032.0)
    timing = (f"CUDA events around each launch on the step's stream, over a second timed pass "
              f"of the same {args.steps} steps ({ms_traced / args.steps:.3f} ms/step with the events)")
    if d_fl > 0:
        achieved = d_fl / (d_ms / 1e3) / 1e12
        if prec in ("bf16", "fp8"):
            # primary: the burst peak (measured at ~full clock, as these kernels run);
            # beside it the sustained peak (measured at a lower, power-capped clock) and
            # the burst peak scaled to the SM clock seen during the headline window
            bound, peak = "tensor", peaks["bf16_tflops"]
            extra = {"frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "peak_sustained": peaks["bf16_tflops_sustained"],
                     "frac_clock_normalised": (achieved / (peak * sm_med / sm_max)) if sm_med else None,
                     "clock_normalisation": f"peak x {sm_med} / {sm_max} MHz (median SM clock of the headline window)"}
            peak_src = f"{src} bf16 burst (cuBLAS 8192^3, best of 10)"
            if prec == "fp8":
                peak_src += ("; the fp8 workload's matmul family mixes e4m3 (qkv, fc forward; nominal rate 2x bf16) "
                             "and bf16 products, reported against the bf16 peak")
        else:
            # the fp32 path's matmuls run on the FP32 FMA units: 148 SMs x 128 lanes x 2 flops
            # at the 2032 MHz maximum SM clock
            bound, peak = "alu", 148 * 128 * 2 * 2.032e9 / 1e12
            extra = {}
            peak_src = "derived: 148 SMs x 128 FP32 lanes x 2 flop/FMA x 2.032 GHz"
        traffic, traffic_src = matmul_traffic(args.workload) if dominant == "matmul" else (None, "no capture")
        roof = {"kernel": dominant, "bound": bound, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, **extra, "traffic": traffic,
                "traffic_measured": False, "traffic_source": traffic_src,
                "peak_source": peak_src,
                "launches": d_n, "avg_launch_ms": d_ms / max(d_n, 1),
                "share_of_traced_step": fam_ms[dominant] / total_ms, "timing": timing}
    else:
        achieved = d_by / (d_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dominant, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": None, "traffic_measured": False,
                "peak_source": f"{src} copy bandwidth",
                "launches": d_n, "avg_launch_ms": d_ms / max(d_n, 1),
                "share_of_traced_step": fam_ms[dominant] / total_ms, "timing": timing}
    fpt, nparams = mfu_flops_per_token(w.shape, T)
    step_s = ms / 1000.0 / args.steps
    mfu = fpt * BT / step_s / 1e12
    kernels = {k: {"ms_per_step": v["ms"] / n_traced,
                   "share": v["ms"] / total_ms,
                   "tflops": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["flops"] and v["ms"] else None,
                   "gbs": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["bytes"] and v["ms"] else None}
               for k, v in warm_prof.items() if v["launches"]}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        sB, sT = 1, min(1024, w.shape.max_seq_len)
        tps, cores, total, per = oracle_tokens_per_s(w, sB, sT, 1)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"one whole step (fwd+bwd+AdamW) of the fp32 CPU oracle on the {w.name} model "
                         f"at B={sB}, T={sT} ({sB * sT} tokens), {total:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": {"bf16": "bf16", "fp8": "fp8", "fp32": "f32"}[prec],
        "data": "synthetic (seeded Zipf s=1.1 int32 token stream, fresh batch per step; random-init weights)",
        "config": {"workload": w.name,
                   "shape": (f"L={w.shape.num_layers}, C={w.shape.channels}, NH={w.shape.num_heads}, "
                             f"V={w.shape.vocab_size} padded to {w.shape.padded_vocab_size}"),
                   "global_batch": B * world, "seq_len": T,
                   "parallelism": "replicas only" if world > 1 else "single GPU",
                   "optimizer": ("Muon (momentum 0.95, 5 Newton-Schulz steps, lr 0.02) on the block matrices, AdamW "
                                 "on the rest" if args.optimizer == "muon" else "AdamW"),
                   "precision": {"bf16": "bf16 weights/activations, fp32 master weights and AdamW state",
                                 "fp8": ("e4m3 qkv and fc forward products (row-scaled layernorm outputs, tensor-scaled "
                                         "weights); bf16 elsewhere; fp32 master weights and AdamW state"),
                                 "fp32": "fp32 throughout"}[prec],
                   "l2": "no flush: the step's working set (GBs of activations) is far larger than the 126 MB L2"},
        "clocks": clk,
        "windows": {"n": len(win_ms), "steps_each": args.steps,
                    "ms_per_step": [x / args.steps for x in win_ms],
                    "tokens_per_s_median": statistics.median(BT * args.steps * world / (x / 1e3) for x in win_ms),
                    "tokens_per_s_min": min(BT * args.steps * world / (x / 1e3) for x in win_ms),
                    "tokens_per_s_max": max(BT * args.steps * world / (x / 1e3) for x in win_ms),
                    "sm_mhz_median": [c["sm_mhz"] for c in win_clk],
                    "note": "the headline value is the first window; the others repeat it for the spread"},
        "gpu_launches": launches,
        "e2e": e2e,
        "mfu": {"model_flops_per_step": fpt * BT, "num_parameters": nparams,
                "tflops": mfu, "vs_measured_burst": mfu / peaks["bf16_tflops"],
                "vs_measured_sustained": mfu / peaks["bf16_tflops_sustained"]},
        "roofline": roof,
        "kernels": kernels,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    return ours(args)


if __name__ == "__main__":
    sys.exit(main())
