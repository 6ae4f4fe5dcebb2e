"""Benchmark: exact attention forward + backward through libfa on GB300.

One step = the whole hot path over one batch: fa_fwd (O, lse), then the
backward's three kernels (D preprocess, dK/dV/dQ kernel, dQ conversion).
Default inputs are seeded synthetic tensors shaped like the long-context
causal workload (B=1, H=16, N=16384, d=128, bf16, values N(0,1) x 0.5); Q, K,
V, dO are 256 MiB together, larger than the 129 MB L2, so no flush is needed.

Prints ONE JSON line (rank 0).  Metric: attention fwd+bwd TFLOP/s with the
FLOP convention fwd = 4 B H N^2 d (halved for causal), bwd = 2.5 x fwd.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference] [--no-extras]

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only under torchrun).  Multi-GPU runs are
independent replicas (every (batch, head) is independent; no collective).
"""
import argparse
import json
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

from workloads import WORKLOADS, generate, flops, sha256  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, causal, 1 GB300) and % of dense bf16 peak"
DEFAULT_WORKLOAD = "long_causal_d128"
# DRAM bytes (read + write) of one launch on the default workload, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of the current
# version of each kernel: the combined backward kernel that fa_bwd launches
# after its preprocess, and the standalone dK/dV kernel; set to None whenever
# a kernel changes until it is captured again.
DRAM_BYTES = {"long_causal_d128": {"bwd_combined": 808603392 + 189961216,
                                   "bwd_dkdv": 380701952 + 103244032}}
# Tensor-pipe activity of each kernel on the default workload: the fraction of
# elapsed cycles the tensor pipe was active (sm__pipe_tensor_cycles_active,
# pct_of_peak_sustained_elapsed) in one-kernel ncu captures of the current
# kernels; set to None whenever a kernel changes until it is captured again.
TENSOR_PIPE_ACTIVE = {"long_causal_d128": {"fwd": 0.649, "bwd_preprocess": 0.0,
                                           "bwd_combined": 0.654, "bwd_dkdv": 0.607,
                                           "bwd_dq": 0.696}}
# the kernels a timed step launches (the work-order kernel aside)
STEP_KERNELS = ("fwd", "bwd_preprocess", "bwd_combined")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def kept_fraction(block_mask):
    if block_mask is None:
        return None
    return float(np.asarray(block_mask, np.float64).mean())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

NVML_CLOCK_SM = 1
# clock event reason bits of NVML that the timing rules look at
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def load_nvml():
    """NVML (the library that ships with the NVIDIA driver), or None."""
    import ctypes
    for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            pass
    return None


class NvmlSampler:
    """Polls one GPU's SM clock, clock event reasons and power through NVML
    (read-only queries) from a host thread every `period_s`; stop(t0, t1)
    summarises the samples whose host time (time.perf_counter) lies in
    [t0, t1], the timed region.  A timed region of a few tens of ms still gets
    dozens of samples, where nvidia-smi's loop would give one or none."""

    def __init__(self, uuid=None, index=0, lib=None, period_s=0.001):
        self.uuid, self.index, self.lib, self.period_s = uuid, index, lib, period_s
        self.samples = []
        self.max_mhz = None
        self.driver = None
        self.thread = None
        self.done = threading.Event()

    def start(self):
        """True when NVML answered and polling has started."""
        import ctypes
        lib = self.lib
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = bool(self.uuid) and lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(),
                                                               ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) == 0
        if not ok:
            lib.nvmlShutdown()
            return False
        self.handle = h
        try:
            buf = ctypes.create_string_buffer(96)
            if lib.nvmlSystemGetDriverVersion(buf, ctypes.c_uint(96)) == 0:
                self.driver = buf.value.decode(errors="replace")
        except (AttributeError, ctypes.ArgumentError, OSError, ValueError):
            pass  # a report field must not end the run
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(NVML_CLOCK_SM), ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self.reasons_fn = None
        for name in ("nvmlDeviceGetCurrentClocksEventReasons",
                     "nvmlDeviceGetCurrentClocksThrottleReasons"):
            try:
                self.reasons_fn = getattr(lib, name)
                break
            except AttributeError:
                pass
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        return True

    def _poll(self):
        import ctypes
        lib, h = self.lib, self.handle
        while not self.done.is_set():
            t = time.perf_counter()
            sm, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
            a = lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(NVML_CLOCK_SM), ctypes.byref(sm))
            b = self.reasons_fn(h, ctypes.byref(rs)) if self.reasons_fn is not None else -1
            c = lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            self.samples.append((t, float(sm.value) if a == 0 else None,
                                 int(rs.value) if b == 0 else None,
                                 pw.value / 1000.0 if c == 0 else None))
            time.sleep(self.period_s)

    def stop(self, t0, t1):
        self.done.set()
        if self.thread is not None:
            self.thread.join(timeout=5)
            self.lib.nvmlShutdown()
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        sm = [x[1] for x in inside if x[1] is not None]
        power = [x[3] for x in inside if x[3] is not None]
        reasons, bits = set(), 0
        for x in inside:
            if x[2] is not None:
                bits |= x[2]
                reasons.update(n for bit, n in NVML_REASONS.items() if x[2] & bit)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_min_mhz": min(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons),
                "reason_bits_seen": hex(bits), "samples": len(sm),
                "source": "NVML polled every %g ms from the host; samples inside the timed "
                          "region only" % (1e3 * self.period_s)}


def device_uuid(dev):
    """NVML's name of a torch CUDA device ("GPU-..."), or None."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


def device_info(dev, driver):
    """The GPU's name, the NVIDIA driver version (from NVML, or None) and the CUDA
    runtime torch was built with; never raises."""
    import torch
    try:
        name = torch.cuda.get_device_name(dev)
    except Exception:  # noqa: BLE001  (a report field must not end the run)
        name = None
    return {"name": name, "driver": driver, "cuda_runtime": torch.version.cuda}


class ClockSampler:
    """nvidia-smi's query loop: the fallback when NVML cannot be loaded."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# replicas: every rank runs the whole workload on its own GPU; the job's time
# is the slowest rank's, its work the sum over ranks
# ---------------------------------------------------------------------------

def max_over_ranks(elapsed_ms, dist, device):
    """Timed-region duration of the job: the max over ranks (dist = None: one rank)."""
    if dist is None:
        return elapsed_ms
    import torch
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(step_flops, steps, elapsed_ms, world):
    """TFLOP/s of the whole job: `world` replicas each did `steps` steps."""
    return world * step_flops * steps / (elapsed_ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank, world, local_rank):
    import torch
    import exact_attention_88_gb300 as fa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOADS[args.workload]
    case = generate(w, seed=0, samples=1)
    to_dev = lambda n: torch.from_numpy(case[n + "_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v, do = (to_dev(n) for n in ("q", "k", "v", "do"))
    B, H, N, d = w.B, w.H, w.N, w.d
    scale = w.scale
    kv_len = None if case["kv_len"] is None else torch.from_numpy(case["kv_len"]).to(dev)
    bmask = None if case["block_mask"] is None else torch.from_numpy(case["block_mask"]).to(dev)
    # block-sparse: the mask's work order (query tiles, key tiles, pairs, most
    # work first), recomputed inside every timed step
    order = None
    if bmask is not None:
        order = torch.empty(fa.fa_block_mask_order_len(bmask.shape[0]), dtype=torch.int32,
                            device=dev)
    mask = fa.make_mask(kv_len, bmask, tile_order=order)
    # fused dropout (--dropout p): the same kernels with the mask drawn in them
    opt = fa.make_options(None, args.dropout, 0x5EED, 1) if args.dropout else None
    kept = kept_fraction(case["block_mask"])
    fwd_flops, step_flops = flops(w, kept)
    # secondary FLOP figures, labelled: dense-equivalent for block-sparse (every
    # tile counted), effective for key padding (sum_b N * kv_len[b] instead of
    # B * N^2)
    dense_step_flops = flops(w)[1]
    eff_step_flops = None
    if case["kv_len"] is not None:
        eff_step_flops = step_flops * float(np.sum(np.minimum(case["kv_len"], N))) / (B * N)
    inputs_sha256 = {n: sha256(case[n + "_bits"]) for n in ("q", "k", "v", "do")}
    if case["kv_len"] is not None:
        inputs_sha256["kv_len"] = sha256(case["kv_len"])
    if case["block_mask"] is not None:
        inputs_sha256["block_mask"] = sha256(case["block_mask"])

    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    rows = B * H * N
    D = ws[: rows * 4].view(torch.float32)
    stream = torch.cuda.current_stream(dev)

    kernels = (["mask_order"] if order is not None else []) + [
        "fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq", "bwd"]
    ev = {n: [] for n in kernels}

    # A timed step is the public calls: fa_fwd_ex, then fa_bwd_ex (the D
    # preprocess, then dK/dV and dQ in one launch whose dQ CTAs fill the SMs the
    # last dK/dV CTAs leave idle).  The per-kernel pass times the same kernels
    # through the one-step calls, each between CUDA events on the stream, and
    # fa_bwd_ex as the step runs it: its time less the preprocess launch's is
    # the combined kernel's.
    def step(record):
        def mark(name, fn):
            if record:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev[name].append((a, b))
            else:
                fn()
        if order is not None:
            mark("mask_order", lambda: fa.fa_block_mask_order(bmask, bmask.shape[0], w.causal,
                                                              order, stream))
        mark("fwd", lambda: fa.fa_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, w.causal, mask, opt,
                                         stream))
        if not record:
            fa.fa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, N, d, scale, w.causal,
                         mask, opt, stream)
            return
        mark("bwd_preprocess", lambda: fa.fa_bwd_preprocess(o, do, D, B, H, N, d, stream))
        mark("bwd_dkdv", lambda: fa.fa_bwd_dkdv_ex(q, k, v, do, lse, D, dk, dv, B, H, N, d, scale,
                                                   w.causal, mask, opt, stream))
        mark("bwd_dq", lambda: fa.fa_bwd_dq_ex(q, k, v, do, lse, D, dq, B, H, N, d, scale,
                                               w.causal, mask, opt, stream))
        mark("bwd", lambda: fa.fa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, N,
                                         d, scale, w.causal, mask, opt, stream))

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(False)
    barrier()
    code, site = fa.fa_get_device_status(stream)
    if code != 0:
        raise RuntimeError("device status %d at site %d during warm-up" % (code, site))

    sampler = NvmlSampler(device_uuid(dev), local_rank, load_nvml())
    fallback = None
    if not sampler.start():
        fallback = ClockSampler(local_rank)
        fallback.start()
        time.sleep(0.3)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    host_t0 = time.perf_counter()
    t0.record(stream)
    for _ in range(args.steps):
        step(False)
    t1.record(stream)
    barrier()
    host_t1 = time.perf_counter()
    elapsed_ms = t0.elapsed_time(t1)
    # per-kernel pass: CUDA events on the launching stream around each launch
    for _ in range(args.steps):
        step(True)
    barrier()
    clocks = fallback.stop() if fallback is not None else sampler.stop(host_t0, host_t1)
    code, site = fa.fa_get_device_status(stream)
    if code != 0:
        raise RuntimeError("device status %d at site %d in the timed region" % (code, site))
    per_kernel = {n: statistics.mean(a.elapsed_time(b) for a, b in ev[n]) for n in kernels}
    per_kernel["bwd_combined"] = max(per_kernel["bwd"] - per_kernel["bwd_preprocess"], 1e-6)

    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(step_flops, args.steps, elapsed_ms, world)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    peak = peaks["bf16_tflops"]
    # per kernel, the GEMM work it does (each GEMM of the backward = fwd_flops / 2):
    # dK/dV kernel S^T, dP^T, dV, dK (all of them part of the 2.5x algorithmic
    # count); dQ kernel S, dP, dQ (only dQ algorithmic, S and dP recomputed again)
    dkdv_flops = 2.0 * fwd_flops
    dq_flops = 1.5 * fwd_flops
    # the combined kernel does the backward's algorithmic work (2.5 x fwd) and
    # executes dK/dV's and dQ's GEMMs (3.5 x fwd)
    bwd_flops = 2.5 * fwd_flops
    bwd_executed = dkdv_flops + dq_flops
    bwd_achieved = bwd_flops / (per_kernel["bwd_combined"] * 1e-3) / 1e12
    bwd_exec_achieved = bwd_executed / (per_kernel["bwd_combined"] * 1e-3) / 1e12
    dram = DRAM_BYTES.get(w.name, {})
    achieved = dkdv_flops / (per_kernel["bwd_dkdv"] * 1e-3) / 1e12
    dq_achieved = dq_flops / (per_kernel["bwd_dq"] * 1e-3) / 1e12
    fwd_achieved = fwd_flops / (per_kernel["fwd"] * 1e-3) / 1e12
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) x %g, bf16)" % w.value_scale,
        "config": {
            "workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
            "mask": w.mask, "kept_tile_fraction": kept, "dropout": args.dropout,
            "global_batch": B * world,
            "seq_len": N, "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs (Q,K,V,dO = %d MiB) larger than the 129 MB L2; no flush" %
                  (4 * q.numel() * 2 >> 20),
        },
        "pct_of_peak": round(100.0 * (value / world) / peak, 2),
        "inputs_sha256": inputs_sha256,
        "kernels_ms": {n: round(t, 4) for n, t in per_kernel.items()},
        # the step's dominant kernel: fa_bwd's combined dK/dV + dQ launch
        "roofline": {
            "kernel": "fa_bwd combined kernel (dK/dV CTAs, then dQ CTAs, on tcgen05)",
            "bound": "tensor",
            "achieved": round(bwd_achieved, 2),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(bwd_achieved / peak, 4),
            "peak_source": "bf16 burst, %s (MEASURED_PEAKS.json)" % peak_kind,
            "traffic": dram.get("bwd_combined"),
            "traffic_unit": "bytes per launch (ncu capture)",
            "flops_per_launch": bwd_flops,
            "duration_ms": round(per_kernel["bwd_combined"], 4),
            "duration_source": "CUDA events around fa_bwd_ex (preprocess + combined kernel) "
                               "less those around the preprocess launch alone",
            "executed_flops_per_launch": bwd_executed,
            "executed_achieved": round(bwd_exec_achieved, 2),
            "executed_frac": round(bwd_exec_achieved / peak, 4),
        },
        "dkdv_roofline": {
            "kernel": "fa_bwd_dkdv (S^T, dP^T, dV, dK on tcgen05; the standalone call)",
            "achieved": round(achieved, 2),
            "frac": round(achieved / peak, 4),
            "traffic": dram.get("bwd_dkdv"),
            "flops_per_launch": dkdv_flops,
        },
        "fwd_roofline": {"kernel": "fa_fwd", "achieved": round(fwd_achieved, 2),
                         "frac": round(fwd_achieved / peak, 4), "flops_per_launch": fwd_flops},
        "dq_roofline": {"kernel": "fa_bwd_dq (S, dP, dQ on tcgen05; S and dP recomputed)",
                        "achieved": round(dq_achieved, 2), "frac": round(dq_achieved / peak, 4),
                        "flops_per_launch": dq_flops},
        # fa_fwd_ex (1), fa_bwd_ex (the preprocess and the combined dK/dV + dQ
        # kernel: 2), and the work-order kernel when block-sparse (1)
        "gpu_launches": (3 + (1 if order is not None else 0)) * args.steps,
        "tensor_pipe": tensor_pipe_share(w.name, per_kernel, step_flops, fwd_flops),
        "peak_clocks": peak_clock_note(peaks, clocks),
        "clocks": clocks,
        "device": device_info(dev, sampler.driver),
    }
    if kept is not None:
        result["dense_equivalent"] = {
            "value": round(world * dense_step_flops * args.steps / (elapsed_ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "note": "every 128x128 tile counted, skipped ones included"}
    if eff_step_flops is not None:
        result["effective"] = {
            "value": round(world * eff_step_flops * args.steps / (elapsed_ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "note": "sum_b N * kv_len[b] in place of B * N^2"}
    if not args.no_extras:
        result["e2e"] = run_e2e(fa, torch, dev, case, w, mask, step_flops, args, opt,
                                bmask, order)
    return result


def tensor_pipe_share(workload, per_kernel_ms, step_flops, fwd_flops):
    """The step's tensor-pipe activity from the ncu captures of each kernel,
    weighted by this run's kernel times, and the share of it that is
    algorithmic work: the kernels execute fwd (2 GEMMs), dK/dV (4) and dQ (3,
    of which S and dP are a second recomputation) = 4.5 x fwd_flops, while the
    metric counts 3.5 x fwd_flops."""
    act = TENSOR_PIPE_ACTIVE.get(workload)
    if not act or any(act.get(k) is None for k in STEP_KERNELS):
        return None
    total = sum(per_kernel_ms[k] for k in STEP_KERNELS)
    busy = sum(act[k] * per_kernel_ms[k] for k in STEP_KERNELS) / total
    executed = fwd_flops + 2.0 * fwd_flops + 1.5 * fwd_flops
    return {"active_time_weighted": round(busy, 4),
            "executed_tflop": round(executed / 1e12, 4),
            "algorithmic_tflop": round(step_flops / 1e12, 4),
            "algorithmic_active": round(busy * step_flops / executed, 4),
            "per_kernel_active": {k: act[k] for k in STEP_KERNELS},
            "source": "one-kernel ncu --set full captures (sm__pipe_tensor_cycles_active, "
                      "% of elapsed cycles), weighted by this run's per-kernel times"}


def peak_clock_note(peaks, clocks):
    """The SM clock the measured GEMM peak was taken at beside this run's."""
    under = peaks.get("clocks_under_load") or {}
    return {"peak_gemm_sm_mhz_median": under.get("sm_mhz_median"),
            "this_run_sm_mhz_median": (clocks or {}).get("sm_mhz"),
            "note": "the measured bf16 peak comes from cuBLAS GEMMs whose SM clock under the "
                    "power cap had the median above; the attention kernels run at the clock "
                    "of this run"}


def run_e2e(fa, torch, dev, case, w, mask, step_flops, args, opt=None, bmask=None,
            order=None):
    """Same metric through the public API with host buffers: every step copies
    its inputs in from pinned host memory, runs fa_fwd_ex and fa_bwd_ex (as in
    the device-resident steps) and copies its results (O, lse, dQ, dK, dV) out,
    all inside the timed region.  Steps
    are pipelined over two sets of device buffers: step k+1's inputs go in on
    one copy stream and step k-1's results come out on another while step k
    computes."""
    B, H, N, d = w.B, w.H, w.N, w.d
    shape = (B, H, N, d)
    host_in = {n: torch.from_numpy(case[n + "_bits"].view(np.int16)).view(torch.bfloat16)
               .pin_memory() for n in ("q", "k", "v", "do")}
    host_out = [{n: torch.empty(shape, dtype=torch.bfloat16).pin_memory()
                 for n in ("o", "dq", "dk", "dv")} for _ in range(2)]
    for h in host_out:
        h["lse"] = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    dev_in = [{n: torch.empty(shape, dtype=torch.bfloat16, device=dev) for n in host_in}
              for _ in range(2)]
    dev_out = [{n: torch.empty(shape, dtype=torch.bfloat16, device=dev)
                for n in ("o", "dq", "dk", "dv")} for _ in range(2)]
    for o in dev_out:
        o["lse"] = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    s_comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def copy_in(k):
        x = dev_in[k % 2]
        if k >= 2:
            s_in.wait_event(comp_done[k % 2])  # step k-2 has read this set
        with torch.cuda.stream(s_in):
            for n in host_in:
                x[n].copy_(host_in[n], non_blocking=True)
        in_ready[k % 2].record(s_in)

    def compute(k):
        x, y = dev_in[k % 2], dev_out[k % 2]
        s_comp.wait_event(in_ready[k % 2])
        if k >= 2:
            s_comp.wait_event(out_done[k % 2])  # step k-2's results have left this set
        if order is not None:
            fa.fa_block_mask_order(bmask, bmask.shape[0], w.causal, order, s_comp)
        fa.fa_fwd_ex(x["q"], x["k"], x["v"], y["o"], y["lse"], B, H, N, d, w.scale, w.causal, mask,
                     opt, s_comp)
        fa.fa_bwd_ex(x["q"], x["k"], x["v"], y["o"], x["do"], y["lse"], y["dq"], y["dk"], y["dv"],
                     ws, ws_bytes, B, H, N, d, w.scale, w.causal, mask, opt, s_comp)
        comp_done[k % 2].record(s_comp)

    def copy_out(k):
        y, h = dev_out[k % 2], host_out[k % 2]
        s_out.wait_event(comp_done[k % 2])
        with torch.cuda.stream(s_out):
            for n in h:
                h[n].copy_(y[n], non_blocking=True)
        out_done[k % 2].record(s_out)

    def run(n_steps):
        copy_in(0)
        for k in range(n_steps):
            if k + 1 < n_steps:
                copy_in(k + 1)
            compute(k)
            copy_out(k)

    run(args.warmup)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    run(args.steps)
    s_out.wait_event(comp_done[(args.steps - 1) % 2])
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / args.steps
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    return {"value": round(step_flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "step k+1 copied in and step k-1 copied out while step k computes"}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores (CPU baseline / reference arm)
# ---------------------------------------------------------------------------

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(w, case, n_rows, heads=1):
    """Time the oracle on the last n_rows query rows (the rows that see the
    most keys under a causal mask; all N rows when the sequence is shorter) of
    the first `heads` (batch, head) slices: O, lse, dQ of those rows and their
    dK, dV contributions.  Returns (seconds, algorithmic FLOPs of the sample
    under the benchmark's convention, rows timed per slice, slices timed)."""
    import oracle
    n_rows = max(1, min(n_rows, w.N))
    slices = [(b, h) for b in range(w.B) for h in range(w.H)][:max(1, heads)]
    rows = np.arange(w.N - n_rows, w.N)
    kw = dict(causal=w.causal, kv_len=case["kv_len"], block_mask=case["block_mask"])
    sec, fwd = 0.0, 0.0
    for b, h in slices:
        t0 = time.perf_counter()
        oracle.row_block_forward_backward(case["q"], case["k"], case["v"], case["do"], w.scale,
                                          b, h, rows, **kw)
        sec += time.perf_counter() - t0
        vis = oracle.visible(rows, w.N, w.causal,
                             None if case["kv_len"] is None else int(case["kv_len"][b]),
                             case["block_mask"], w.block)
        fwd += 4.0 * w.d * float(vis.sum())   # Q K^T and P V over the visible pairs
    return sec, 3.5 * fwd, n_rows, len(slices)


def cpu_baseline(w, case, n_rows, heads):
    sec, fl, n_rows, n_slices = oracle_sample(w, case, n_rows, heads)
    return {"value": round(fl / sec / 1e12, 6), "unit": "TFLOP/s", "cores": host_cores(),
            "kind": "oracle",
            "sample": "fp64 numpy oracle, fwd+bwd of the last %d query rows of each of the first "
                      "%d (batch, head) slices of %s against all %d keys (O, lse, dQ and the "
                      "rows' dK/dV contributions) in %.1f s; BLAS matmuls threaded over the host "
                      "cores, elementwise steps single-threaded"
                      % (n_rows, n_slices, w.name, w.N, sec)}


def cpu_model():
    """The host CPU's model name (x86: /proc/cpuinfo "model name"; Arm: lscpu's
    "Model name", which names the core, e.g. Neoverse-V2)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# the five workloads the metric's configurations name, in their order
ORACLE_TIME_WORKLOADS = ["tiny_fp32", "tiny_fp32_causal", "gpt2_causal", "bert_padding",
                         "long_causal_d128", "block_sparse"]


def oracle_times(rows_per_block=2048):
    """Host time of the fp64 oracle on every configuration: the whole forward +
    backward where it fits (the short workloads), else one whole (batch, head)
    slice -- every query row, in blocks of rows, forward and backward -- scaled
    by B*H and labelled "extrapolated", plus the wall time of the sampled-row
    check the parity tests make (O, lse, dQ of 256 query rows per head).  One
    JSON line per workload."""
    import oracle
    out = []
    for name in ORACLE_TIME_WORKLOADS:
        w = WORKLOADS[name]
        case = generate(w, seed=0, samples=256)
        kept = kept_fraction(case["block_mask"])
        fwd_fl, step_fl = flops(w, kept)
        kw = dict(causal=w.causal, kv_len=case["kv_len"], block_mask=case["block_mask"])
        rec = {"workload": name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
               "mask": w.mask, "cores": host_cores(), "cpu": cpu_model(),
               "algorithmic_gflop_fwd_bwd": round(step_fl / 1e9, 3)}
        if not w.sampled:
            t0 = time.perf_counter()
            oracle.forward(case["q"], case["k"], case["v"], w.scale, **kw)
            oracle.backward(case["q"], case["k"], case["v"], case["do"], w.scale, **kw)
            sec = time.perf_counter() - t0
            rec.update(kind="whole workload, forward + backward", seconds=round(sec, 3),
                       tflops=round(step_fl / sec / 1e12, 6))
        else:
            t0 = time.perf_counter()
            for r0 in range(0, w.N, rows_per_block):
                oracle.row_block_forward_backward(case["q"], case["k"], case["v"], case["do"],
                                                  w.scale, 0, 0,
                                                  np.arange(r0, min(w.N, r0 + rows_per_block)),
                                                  **kw)
            sec = time.perf_counter() - t0
            slices = w.B * w.H
            rec.update(kind="one (batch, head) slice, forward + backward of every row, x B*H: "
                            "extrapolated",
                       seconds_one_slice=round(sec, 3),
                       seconds=round(sec * slices, 1),
                       tflops=round(step_fl / (sec * slices) / 1e12, 6))
            t0 = time.perf_counter()
            oracle.forward_rows(case["q"], case["k"], case["v"], w.scale, case["rows"], **kw)
            oracle.backward_query_rows(case["q"], case["k"], case["v"], case["do"], w.scale,
                                       case["rows"], **kw)
            rec["sampled_query_rows_check_seconds"] = round(time.perf_counter() - t0, 3)
        out.append(rec)
        print(json.dumps(rec), flush=True)
    return out


def run_reference(args, rank):
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    case = generate(w, seed=0, samples=1)
    n_rows = min(args.reference_rows, w.N)
    for _ in range(args.warmup):
        oracle_sample(w, case, n_rows)
    secs, fl = 0.0, 0.0
    for _ in range(args.steps):
        s, f, _, _ = oracle_sample(w, case, n_rows)
        secs += s
        fl += f
    value = fl / secs / 1e12
    cpu = {"value": round(value, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
           "sample": "per step: fp64 numpy oracle fwd+bwd of the last %d query rows of head "
                     "(0,0) of %s against all %d keys" % (n_rows, w.name, w.N)}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "mask": w.mask},
            "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-extras", action="store_true",
                    help="skip e2e and the CPU baseline (for profiler runs)")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="fused dropout probability on the attention probabilities (0: none)")
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--cpu-heads", type=int, default=5,
                    help="(batch, head) slices in the CPU baseline's sample (about 2 s each "
                         "on the long causal workload)")
    ap.add_argument("--reference-rows", type=int, default=2048)
    ap.add_argument("--oracle-times", action="store_true",
                    help="time the fp64 oracle on the host for every configuration (no GPU) "
                         "and print one JSON line per workload")
    args = ap.parse_args()

    if args.oracle_times:
        oracle_times()
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_extras and world == 1:
            w = WORKLOADS[args.workload]
            case = generate(w, seed=0, samples=1)
            res["cpu_baseline"] = cpu_baseline(w, case, args.cpu_rows, args.cpu_heads)
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
