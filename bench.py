"""Benchmark of fused SDPA training (forward + backward) on GB300.

One step = sdpa_fwd + sdpa_bwd (the whole hot path) on the long-context
decoder workload B8 H16 S4096 D128, causal, bf16, dropout 0 (seeded
synthetic inputs, BHSE). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

value       whole-job TFLOP/s of the step (algorithmic flops: forward 4*D*pairs,
            backward 10*D*pairs per head, pairs = unmasked (query, key) pairs)
            with inputs resident in HBM; the bf16 fraction of the measured
            tensor peak is reported beside it.
clocks      SM clock, power and clock-event reasons sampled (NVML, every 2 ms)
            inside the timed region only.
sustained   the same step back to back for a few seconds after the timed
            region, against the sustained bf16 peak, with the clock samples
            of that window.
e2e         the same metric through the public API with host buffers: each
            step copies q, k, v, dout from pinned host memory and copies out,
            lse, dq, dk, dv back; steps are pipelined over an upload, a
            compute and a download stream.
roofline    the backward (dominant) and forward kernels against the measured
            dense bf16 peak.
extended    the options entry points on the same workload (the step recorded
            once as a CUDA graph, the deterministic backward, dropout 0.1,
            head dims 96 and 256, a relative-position bias, a packed batch of
            mixed lengths) and the other named workloads.
cpu_baseline / --impl reference: the fp64 CPU oracle on a bounded sample of
            the same workload (whole heads), on this host's cores.
"""

import argparse
import ctypes
import hashlib
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "decoder_long"
METRIC = "fwd/bwd TFLOP/s bf16 (B8 H16 S4096 D128 causal); % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def pairs(w):
    """Unmasked (query, key) pairs per head; causal is top-left aligned."""
    if not w.is_causal:
        return w.Sq * w.Sk
    n = min(w.Sq, w.Sk)
    full = w.Sq - n  # rows that see every key
    return n * (n + 1) // 2 + full * w.Sk


def flops(w):
    p = pairs(w) * w.B * w.H * w.D
    return 4 * p, 10 * p


def bwd_small_kernel_bytes(w):
    """Algorithmic HBM bytes of the backward's two small kernels per call.

    bwd_preprocess_kernel reads out and dout (bf16) and lse (fp32), and writes
    the padded lse*log2(e) and Delta rows and the zeroed fp32 dQ accumulator
    (rows of 128 columns, Sq padded to 128); bwd_dq_convert_kernel reads the
    caller's D columns of the accumulator's real rows and writes dq (bf16).
    """
    bh = w.B * w.H
    sq_pad = (w.Sq + 127) // 128 * 128
    pre = bh * (2 * w.Sq * w.D * 2 + 4 * w.Sq + sq_pad * (128 + 2) * 4)
    conv = bh * (w.Sq * w.D * 4 + w.Sq * w.D * 2)
    return pre + conv


# Integer work of one Philox4x32-10 group (four keep decisions) as the
# kernels draw it: ten rounds of two 32x32->64-bit products (the FMA pipe's
# wide multiply) and two three-input XORs, then four threshold compares and
# four selects. The forward takes each round's key from the kernel
# parameters; the backward forms it at run time (two additions per round)
# and assembles the quad's keep nibbles (about eight more operations).
PHILOX_OPS = {"fwd": {"mul_wide": 20, "alu": 28}, "bwd": {"mul_wide": 20, "alu": 56}}
# Per-SM rates of the two pipes, in lane-operations per clock: the ALU pipe
# retires 64 (16 lanes on each of the four schedulers); a 32x32->64-bit
# multiply takes two issue slots of the 16-lane FMA-heavy pipe, so 32. (The
# profiled dropout forward's FMA-heavy active cycles match four cycles per
# warp-wide multiply, and a loop of Philox draws alone saturates at about
# three quarters of this bound.) The two pipes run in parallel, so the
# bound is the busier one.
PIPE_LANE_OPS_PER_CLK_PER_SM = {"mul_wide": 32, "alu": 64}
SM_COUNT = 152


def philox_alu_bound(w, direction, clock_mhz, pass_ms, base_ms, peak_tflops):
    """Roofline of one pass with dropout, which has two bounds: its tensor
    work (the pass's algorithmic flops at the dense bf16 peak) and the integer
    work of its dropout draws -- one Philox group per four visible (query,
    key) pairs (keys past the causal diagonal are not drawn), timed on the
    busier of the ALU and FMA-heavy pipes at the sampled clock. The two run on
    different units and overlap, so the pass can be no faster than the larger
    bound; frac = that bound / the measured pass. dropout_extra_ms, the pass
    less the same pass at p = 0, is the time the draws did not hide."""
    groups = pairs(w) * w.B * w.H / 4
    ops = PHILOX_OPS[direction]
    clk = (clock_mhz or 2070.0) * 1e6
    per_pipe = {k: groups * n / (PIPE_LANE_OPS_PER_CLK_PER_SM[k] * SM_COUNT * clk) * 1e3
                for k, n in ops.items()}
    alu_ms = max(per_pipe.values())
    f_fwd, f_bwd = flops(w)
    tensor_ms = (f_fwd if direction == "fwd" else f_bwd) / (peak_tflops * 1e12) * 1e3
    bound = max(alu_ms, tensor_ms)
    return {"bound": "alu" if alu_ms >= tensor_ms else "tensor", "groups": groups,
            "ops_per_group": ops, "lane_ops_per_clk_per_sm": PIPE_LANE_OPS_PER_CLK_PER_SM,
            "sm_count": SM_COUNT, "clock_mhz": clock_mhz, "pipe_ms": per_pipe,
            "alu_bound_ms": alu_ms, "tensor_bound_ms": tensor_ms, "pass_ms": pass_ms,
            "frac": bound / pass_ms if pass_ms > 0 else None,
            "dropout_extra_ms": pass_ms - base_ms}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def _tensor_mb(w):
    return w.B * w.H * w.Sq * w.D * 2 / 1e6, w.B * w.H * w.Sk * w.D * 2 / 1e6


def small_l2(w):
    q_mb, kv_mb = _tensor_mb(w)
    return 3 * q_mb + 2 * kv_mb <= 129  # q, out, dout, k, v against the 129 MB L2


def l2_note(w):
    q_mb, kv_mb = _tensor_mb(w)
    if small_l2(w):
        return (f"inputs smaller than L2 (q, out, dout {q_mb:.0f} MB each; k, v {kv_mb:.0f} MB "
                f"each): L2 flushed (256 MB write) before each step, outside the fwd/bwd events")
    return (f"inputs larger than L2 (q, out, dout {q_mb:.0f} MB each; k, v {kv_mb:.0f} MB each), "
            f"no flush")


def workload_config(w, extra=None):
    cfg = {"workload": f"{w.name} B{w.B} H{w.H} Sq{w.Sq} Sk{w.Sk} D{w.D} "
                       f"{'causal' if w.is_causal else 'full'} p{w.dropout_p} bf16 BHSE",
           "B": w.B, "H": w.H, "Sq": w.Sq, "Sk": w.Sk, "D": w.D, "causal": w.is_causal,
           "dropout_p": w.dropout_p, "layout": "BHSE",
           "l2": l2_note(w)}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# clock sampling

# clock-event reason bits of NVML's public API (nvmlClocksEventReason*)
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                     "hw_power_brake_slowdown")


class _Nvml:
    """The few read-only NVML queries the sampler needs, through ctypes."""

    def __init__(self, uuid, index):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        h = ctypes.c_void_p()
        ok = False
        if uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid.encode()), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle for the device")
        self.h = h
        try:
            self._reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._clock(lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn):
        v = ctypes.c_uint()
        return float(v.value) if fn(self.h, ctypes.c_int(1), ctypes.byref(v)) == 0 else None

    def sample(self):
        mw = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        power = mw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw)) == 0 \
            else None
        reasons = r.value if self._reasons(self.h, ctypes.byref(r)) == 0 else 0
        return self._clock(self.lib.nvmlDeviceGetClockInfo), power, reasons


class ClockSampler:
    """SM clock, power and clock-event reasons sampled on a host thread, each
    sample stamped with time.perf_counter(), so that the samples of one timed
    window can be cut out afterwards (window()). NVML every 2 ms; nvidia-smi
    every 50 ms where NVML cannot be loaded."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, uuid=None, period_s=0.002):
        self.index, self.uuid, self.period = index, uuid, period_s
        self.samples = []  # (t, sm_mhz, max_mhz, power_w, reasons set)
        self.source = None
        self._stop = threading.Event()
        self.proc = None
        self.thread = None

    def start(self):
        try:
            nv = _Nvml(self.uuid, self.index)
            self.source = "nvml"
            self.thread = threading.Thread(target=self._nvml_loop, args=(nv,), daemon=True)
        except (OSError, AttributeError):
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                self.thread = threading.Thread(target=self._smi_loop, daemon=True)
            except OSError:
                return
        self.thread.start()

    def _nvml_loop(self, nv):
        while not self._stop.is_set():
            sm, power, bits = nv.sample()
            reasons = {name for bit, name in _REASON_BITS.items() if bits & bit}
            self.samples.append((time.perf_counter(), sm, nv.max_mhz, power, reasons))
            time.sleep(self.period)

    def _smi_loop(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.proc.stdout:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax, power = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {n for n, val in zip(names, parts[5:9]) if val.lower() == "active"}
            self.samples.append((time.perf_counter(), sm, smax, power, reasons))

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def window(self, t0, t1):
        return summarize_clocks([s for s in self.samples if t0 <= s[0] <= t1], self.source)


def summarize_clocks(samples, source):
    """Summary of the clock samples taken inside one window (the GPU busy
    throughout it): median and minimum SM clock, maximum power, and every
    clock-event reason seen active."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "samples_under_load": 0,
                "reasons": [] if source else ["no clock source"], "source": source}
    sm = [s[1] for s in samples if s[1] is not None]
    smax = [s[2] for s in samples if s[2] is not None]
    power = [s[3] for s in samples if s[3] is not None]
    reasons = set().union(*(s[4] for s in samples))
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_min_mhz": min(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None, "samples_under_load": len(samples),
            "reasons": sorted(reasons), "source": source,
            "rejected": any(r in reasons for r in REJECTING_REASONS)}


def kernel_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    ent = traffic_entry(kernel)
    return ent["bytes_per_launch"] if ent else None


def traffic_entry(kernel):
    """The committed ncu figures of one kernel, if the source they were taken
    from is the source here (its sha256 prefix matches)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "scaled_dot_product_07_gb300", "csrc", ent["source"])
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return ent if digest == ent.get("source_sha256_16") else None


# ---------------------------------------------------------------------------
# ranks

def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier_max(value, world):
    """Max over ranks (host float) after a barrier."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the oracle (CPU baseline and the reference arm)

_INPUT_CACHE = {}


def cached_inputs(w):
    from scaled_dot_product_07_gb300 import workloads as W
    if w.name not in _INPUT_CACHE:
        _INPUT_CACHE[w.name] = W.draw_inputs(w)
    return _INPUT_CACHE[w.name]


def run_oracle_sample(w, budget_s, min_heads=1, start=0):
    """Oracle forward + backward on whole heads until `budget_s` of CPU time."""
    import numpy as np

    import oracle
    q, k, v, do = cached_inputs(w)
    f64 = lambda t: t.float().numpy().astype(np.float64)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    heads = heads[start % len(heads):] + heads[:start % len(heads)]
    done, t0 = 0, time.perf_counter()
    for b, h in heads:
        qh, kh, vh, doh = f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(do[b, h])
        scale = oracle.default_scale(w.D)
        out, lse = oracle.head_forward(qh, kh, vh, b, h, w.H, w.dropout_p, w.is_causal, scale,
                                       w.seed, w.offset)
        oracle.head_backward(doh, qh, kh, vh, out, lse, b, h, w.H, w.dropout_p, w.is_causal,
                             scale, w.seed, w.offset, check_delta=False)
        done += 1
        if done >= min_heads and time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    f = sum(flops(w)) / (w.B * w.H) * done
    return f / el / 1e12, done, el


def cpu_threads():
    return os.cpu_count() or 1


def bench_reference(args, w):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    # each step: the oracle's fwd+bwd of one whole head of the workload
    cached_inputs(w)
    for i in range(args.warmup):
        run_oracle_sample(w, 0.0, 1, start=i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        run_oracle_sample(w, 0.0, 1, start=args.warmup + i)
    el = time.perf_counter() - t0
    val = sum(flops(w)) / (w.B * w.H) * args.steps / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, {"sample": "one whole head per step"}),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"{args.steps} heads (fwd+bwd, fp64 numpy) of {w.B * w.H}"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# the JSON line

def assemble_line(w, world, steps, warmup, t, peak_table, peak_src, clocks, sustained=None,
                  extras=None, e2e=None, cpu=None, launches_per_step=4):
    """The bench's JSON line from its measurements (no GPU work here).

    t: the timed region's figures in ms -- total_ms (all steps, max over
    ranks), fwd_ms and bwd_ms (mean per call), fwd_kernel_ms and bwd_main_ms
    (mean per launch of the forward kernel and the backward's main kernel).
    """
    f_fwd, f_bwd = flops(w)
    peak = peak_table.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peak_table.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tf = lambda f, ms: f / (ms * 1e-3) / 1e12
    step_ms = t["total_ms"] / steps
    value = world * (f_fwd + f_bwd) / (step_ms * 1e-3) / 1e12
    fwd_tf, bwd_tf = tf(f_fwd, t["fwd_ms"]), tf(f_bwd, t["bwd_ms"])
    # every flop of each pass is in its main kernel
    fwd_kernel_tf, bwd_main_tf = tf(f_fwd, t["fwd_kernel_ms"]), tf(f_bwd, t["bwd_main_ms"])
    # the backward call's small HBM-bound kernels: the call's time less its
    # main kernel's (launch gaps included, so a lower bound on their rate);
    # no figure when the difference is not positive
    small_ms = t["bwd_ms"] - t["bwd_main_ms"]
    small_bytes = bwd_small_kernel_bytes(w)
    small_gbs = small_bytes / (small_ms * 1e-3) / 1e9 if small_ms > 0 else None
    ncu_small = {k: traffic_entry(k) for k in ("bwd_preprocess_kernel", "bwd_dq_convert_kernel")}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w),
        "fwd": {"ms": t["fwd_ms"], "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak},
        "bwd": {"ms": t["bwd_ms"], "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak,
                "note": "the whole backward call: preprocess + main + dQ-convert kernels"},
        "pct_of_bf16_peak": 100.0 * (value / world) / peak,
        "roofline": {"kernel": "bwd_main_kernel_d128", "bound": "tensor", "achieved": bwd_main_tf,
                     "peak": peak, "unit": "TFLOP/s", "frac": bwd_main_tf / peak,
                     "traffic": kernel_traffic("bwd_main_kernel"),
                     "ms_per_launch": t["bwd_main_ms"],
                     "timing": "CUDA events recorded by the library around each launch "
                               "(kernel_events), mean over the timed steps",
                     "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "roofline_fwd": {"kernel": "fwd_kernel", "bound": "tensor", "achieved": fwd_kernel_tf,
                         "peak": peak, "unit": "TFLOP/s", "frac": fwd_kernel_tf / peak,
                         "traffic": kernel_traffic("fwd_kernel"),
                         "ms_per_launch": t["fwd_kernel_ms"],
                         "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "roofline_bwd_hbm": {"kernel": "bwd_preprocess_kernel + bwd_dq_convert_kernel",
                             "bound": "hbm", "achieved": small_gbs, "peak": hbm, "unit": "GB/s",
                             "frac": small_gbs / hbm if small_gbs is not None else None,
                             "bytes": small_bytes, "ms_per_call": small_ms,
                             "timing": "backward call events less the main kernel's events "
                                       "(launch gaps included)",
                             "ncu": {k: ({"gbs": e.get("gbs"), "dram_bytes": e["bytes_per_launch"],
                                          "us": e.get("us_per_launch")} if e else None)
                                     for k, e in ncu_small.items()},
                             "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": e2e,
        "sustained": sustained,
        "extended": extras,
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if sustained is not None:
        sp = peak_table.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
        sustained["peak"] = sp
        sustained["frac"] = sustained["tflops"] / sp
        sustained["peak_source"] = f"{peak_src} bf16_tflops_sustained"
    return line


# ---------------------------------------------------------------------------
# GPU measurements

def _timed(torch, stream, fn, n):
    """Mean ms of fn() over n back-to-back calls, CUDA events on `stream`."""
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def _pass_line(w, fwd_ms, bwd_ms, note, peak):
    f, b = flops(w)
    return {"fwd_ms": fwd_ms, "fwd_tflops": f / (fwd_ms * 1e-3) / 1e12,
            "fwd_frac": f / (fwd_ms * 1e-3) / 1e12 / peak,
            "bwd_ms": bwd_ms, "bwd_tflops": b / (bwd_ms * 1e-3) / 1e12,
            "bwd_frac": b / (bwd_ms * 1e-3) / 1e12 / peak, "note": note}


def measure_sustained(torch, stream, step, seconds, sampler, world):
    """The step back to back for `seconds` (one chunk of steps always queued
    behind the one the host waits on, so the GPU never idles), timed with
    CUDA events, with the clock samples of that window."""
    chunk = 32
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    start.record(stream)
    n = 0
    while True:
        for _ in range(chunk):
            step()
        n += chunk
        e = torch.cuda.Event()
        e.record(stream)
        marks.append(e)
        if len(marks) > 1:
            marks.pop(0).synchronize()
        if time.perf_counter() - h0 >= seconds:
            break
    end.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    ms = start.elapsed_time(end)
    return n, ms, sampler.window(h0, h1)


def bench_ours(args, w):
    import torch

    import scaled_dot_product_07_gb300 as sdpa
    from scaled_dot_product_07_gb300 import workloads as W

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from scaled_dot_product_07_gb300 import _build
    _build.build()
    sdpa.load_library()
    pk_table, pk_src = peaks()
    peak = pk_table.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])

    uuid = None
    try:
        u = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
        uuid = ("GPU-" + str(u)) if u is not None else None
    except Exception:
        uuid = None
    sampler = ClockSampler(local, uuid)
    sampler.start()

    inputs_cpu = cached_inputs(w)
    q, k, v, do = (x.to(dev) for x in inputs_cpu)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(sdpa.sdpa_bwd_workspace_size(w.B, w.H, w.Sq, w.Sk, w.D), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    # profiling the bias path: a relative-position bias shared by the batch
    bias = (W.padded_rows(W.draw_bias((1, w.H, w.Sq, w.Sk), w.input_seed + 17, "relpos").to(dev))
            if args.bias else None)
    # profiling the dropout path with the keep bits carried forward to backward
    bits = (torch.empty(sdpa.sdpa_dropout_bits_size(w.B, w.H, w.Sq, w.Sk) // 4, dtype=torch.int32,
                        device=dev) if args.stored_bits else None)

    def step():
        sdpa.sdpa_fwd_ex(q, k, v, w.dropout_p, w.is_causal, None, w.seed, w.offset,
                         attn_bias=bias, out=out, lse=lse, dropout_bits=bits)
        sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed, w.offset, None,
                         attn_bias=bias, dq=dq, dk=dk, dv=dv, workspace=ws, dropout_bits=bits)

    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if sdpa.sdpa_check_device() != 0:
        raise RuntimeError("kernel wait timed out during warm-up")

    # ---- timed region: K whole steps, per-phase events on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # per step, the library records these around the forward kernel and
    # around the backward's main kernel (the roofline's per-launch times);
    # torch creates a CUDA event on its first record
    km = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    for e4 in km:
        for e in e4:
            e.record(stream)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # a workload whose inputs fit in L2 gets the cache flushed before each
    # step (a 256 MB write, outside the fwd/bwd events); its step time is then
    # the sum of the fwd and bwd events
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev) if small_l2(w) else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(stream)
        sdpa.sdpa_fwd_ex(q, k, v, w.dropout_p, w.is_causal, None, w.seed, w.offset, out=out,
                         lse=lse, attn_bias=bias, kernel_events=km[i][0:2], dropout_bits=bits)
        ev[i][1].record(stream)
        sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed, w.offset, None,
                         attn_bias=bias, dq=dq, dk=dk, dv=dv, workspace=ws,
                         kernel_events=km[i][2:4], dropout_bits=bits)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    h1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.window(h0, h1)
    if sdpa.sdpa_check_device() != 0:
        raise RuntimeError("kernel wait timed out in the timed region")
    t = {"fwd_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
         "bwd_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in ev),
         "fwd_kernel_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in km),
         "bwd_main_ms": statistics.mean(e[2].elapsed_time(e[3]) for e in km)}
    if flush is None:
        t["total_ms"] = barrier_max(t_start.elapsed_time(t_end), world)
    else:
        t["total_ms"] = barrier_max(sum(e[0].elapsed_time(e[2]) for e in ev), world)
    del flush
    f_fwd, f_bwd = flops(w)

    # ---- the end-to-end pass, right after the timed steps: after the
    # extended timings (graph capture, large workspaces) its copies-alone loop
    # ran several times slower than the same copies in a fresh process, while
    # the pipelined step did not change
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(torch, sdpa, w, dev, stream, inputs_cpu, q, k, v, lse, ws, world)
    # ---- the same step back to back for a few seconds: sustained rate and
    # the clocks under a long load
    sustained = None
    if args.sustain_seconds > 0:
        n, ms, sclocks = measure_sustained(torch, stream, step, args.sustain_seconds, sampler,
                                           world)
        if sdpa.sdpa_check_device() != 0:
            raise RuntimeError("kernel wait timed out in the sustained loop")
        s_ms = barrier_max(ms, world) / n
        sustained = {"steps": n, "ms_per_step": s_ms,
                     "tflops": world * (f_fwd + f_bwd) / (s_ms * 1e-3) / 1e12, "clocks": sclocks,
                     "timing": "CUDA events around the whole back-to-back loop"}

    extras = None
    if not args.no_extras:
        extras = measure_extras(torch, sdpa, W, w, dev, stream, q, k, v, do, out, lse, dq, dk, dv,
                                ws, peak, t["fwd_ms"], t["bwd_ms"], clocks.get("sm_mhz"))
    sampler.stop()

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        val, heads, el = run_oracle_sample(w, args.cpu_seconds)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{heads} whole heads of {w.B * w.H} (fwd+bwd, fp64 numpy, {el:.1f} s)"}
    line = assemble_line(w, world, args.steps, warmup, t, pk_table, pk_src, clocks, sustained,
                         extras, e2e, cpu)
    if bias is not None:
        line["config"]["bias"] = "relative-position [1, H, Sq, Sk] bf16 (profiling case)"
    if bits is not None:
        line["config"]["stored_bits"] = "keep bits carried forward to backward (profiling case)"
    print(json.dumps(line))
    return 0


def measure_extras(torch, sdpa, W, w, dev, stream, q, k, v, do, out, lse, dq, dk, dv, ws, peak,
                   base_fwd_ms, base_bwd_ms, clock_mhz):
    """The options entry points on the same workload, and the other named
    workloads' passes (each timed alone, CUDA events, mean of a few calls)."""
    extras = {}
    f_fwd, f_bwd = flops(w)
    timed = lambda fn, n: _timed(torch, stream, fn, n)

    # the step recorded once as a CUDA graph with the rng state read from
    # device memory, then replayed
    rng = torch.tensor([w.seed, w.offset], dtype=torch.int64, device=dev)

    def step_ex():
        sdpa.sdpa_fwd_ex(q, k, v, w.dropout_p, w.is_causal, rng_state=rng, out=out, lse=lse)
        sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal, rng_state=rng,
                         dq=dq, dk=dk, dv=dv, workspace=ws)

    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step_ex()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step_ex()
    g_ms = timed(graph.replay, 20)
    extras["graph_step"] = {"ms": g_ms, "tflops": (f_fwd + f_bwd) / (g_ms * 1e-3) / 1e12,
                            "note": "fwd+bwd captured once (sdpa_fwd_ex/sdpa_bwd_ex, rng "
                                    "state in device memory), replayed"}
    del graph

    # the deterministic (fixed-order dQ) backward
    ws_det = torch.empty(sdpa.sdpa_bwd_workspace_size_ex(w.B, w.H, w.Sq, w.Sk, w.D, True),
                         dtype=torch.uint8, device=dev)
    d_ms = timed(lambda: sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed,
                                          w.offset, deterministic=True, dq=dq, dk=dk, dv=dv,
                                          workspace=ws_det), 5)
    extras["bwd_deterministic"] = {
        "ms": d_ms, "tflops": f_bwd / (d_ms * 1e-3) / 1e12, "workspace_bytes": ws_det.numel(),
        "note": "one fp32 dQ partial per 128-key tile, summed in key-tile order"}
    del ws_det

    # dropout on the same shape: the keep mask is drawn inside the kernels
    # (Philox4x32-10 on the absolute element index), forward and backward
    p_d = 0.1
    fwd_d = timed(lambda: sdpa.sdpa_fwd(q, k, v, p_d, w.is_causal, None, w.seed, w.offset,
                                        out=out, lse=lse), 5)
    bwd_d = timed(lambda: sdpa.sdpa_bwd(do, q, k, v, out, lse, p_d, w.is_causal, w.seed,
                                        w.offset, None, dq=dq, dk=dk, dv=dv, workspace=ws), 5)
    wd = W.make_workload(w.name, dropout_p=p_d)
    extras["dropout_0.1"] = _pass_line(w, fwd_d, bwd_d, "dropout_p 0.1 on the same B, H, S, D; "
                                       "the mask is regenerated in the backward", peak)
    extras["dropout_0.1"]["alu_fwd"] = philox_alu_bound(wd, "fwd", clock_mhz, fwd_d, base_fwd_ms,
                                                        peak)
    extras["dropout_0.1"]["alu_bwd"] = philox_alu_bound(wd, "bwd", clock_mhz, bwd_d, base_bwd_ms,
                                                        peak)
    # the same with the keep bits carried from the forward to the backward
    bits = torch.empty(sdpa.sdpa_dropout_bits_size(w.B, w.H, w.Sq, w.Sk) // 4, dtype=torch.int32,
                       device=dev)
    fwd_s = timed(lambda: sdpa.sdpa_fwd_ex(q, k, v, p_d, w.is_causal, None, w.seed, w.offset,
                                           out=out, lse=lse, dropout_bits=bits), 5)
    bwd_s = timed(lambda: sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, p_d, w.is_causal, w.seed,
                                           w.offset, dq=dq, dk=dk, dv=dv, workspace=ws,
                                           dropout_bits=bits), 5)
    extras["dropout_0.1"]["stored_bits"] = stored_bits_line(wd, fwd_s, bwd_s, fwd_d, bwd_d,
                                                            bits.numel() * 4, peak)
    del bits

    # other head dims on the same B, H, S: 96 (the 128-wide kernels with the
    # last 32 columns zero-filled by TMA) and 256 (the 256-wide kernels)
    for D in (96, 256):
        wd = W.Workload(f"{w.name}_d{D}", w.B, w.H, w.Sq, w.Sk, D, w.is_causal, w.dropout_p,
                        seed=w.seed, offset=w.offset, input_seed=w.input_seed)
        gd = torch.Generator(device="cpu")
        gd.manual_seed(w.input_seed)
        qd, kd, vd, dod = (torch.randn(x.shape[:3] + (D,), generator=gd).to(torch.bfloat16)
                           .to(dev) for x in (q, k, v, do))
        outd, lsed = torch.empty_like(qd), torch.empty_like(lse)
        dqd, dkd, dvd = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        wsd = torch.empty(sdpa.sdpa_bwd_workspace_size(w.B, w.H, w.Sq, w.Sk, D),
                          dtype=torch.uint8, device=dev)
        fwd_x = timed(lambda: sdpa.sdpa_fwd(qd, kd, vd, w.dropout_p, w.is_causal, None, w.seed,
                                            w.offset, out=outd, lse=lsed), 5)
        bwd_x = timed(lambda: sdpa.sdpa_bwd(dod, qd, kd, vd, outd, lsed, w.dropout_p,
                                            w.is_causal, w.seed, w.offset, None, dq=dqd, dk=dkd,
                                            dv=dvd, workspace=wsd), 5)
        extras[f"head_dim_{D}"] = _pass_line(wd, fwd_x, bwd_x, f"algorithmic flops at D={D}",
                                             peak)
        del qd, kd, vd, dod, outd, dqd, dkd, dvd, wsd

    # additive bias: a relative-position bias shared by the batch, [1, H, Sq, Sk];
    # the backward also writes its full [B, H, Sq, Sk] gradient
    bias = W.padded_rows(W.draw_bias((1, w.H, w.Sq, w.Sk), w.input_seed + 17, "relpos").to(dev))
    dbias = torch.empty((w.B, w.H, w.Sq, w.Sk), dtype=torch.bfloat16, device=dev)
    fwd_b = timed(lambda: sdpa.sdpa_fwd_ex(q, k, v, w.dropout_p, w.is_causal, None, w.seed,
                                           w.offset, attn_bias=bias, out=out, lse=lse), 5)
    bwd_b = timed(lambda: sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal,
                                           w.seed, w.offset, attn_bias=bias, dbias=dbias,
                                           dq=dq, dk=dk, dv=dv, workspace=ws), 5)
    extras["attn_bias"] = _pass_line(w, fwd_b, bwd_b, "bf16 relative-position bias [1,H,Sq,Sk] "
                                     "shared by the batch; the backward also writes dbias "
                                     "[B,H,Sq,Sk] bf16", peak)
    del bias, dbias

    # a packed batch of causal sequences of mixed lengths (the decoder's
    # heads and head dim), through the variable-length entry points
    lens = [4096, 2048, 3072, 1024, 4096, 512, 3584, 2560]
    H, D = w.H, w.D
    tot = sum(lens)
    gv = torch.Generator(device="cpu")
    gv.manual_seed(w.input_seed + 29)
    vq, vk, vv, vdo = (torch.randn((tot, H, D), generator=gv).to(torch.bfloat16).to(dev)
                       for _ in range(4))
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device=dev)
    vout = torch.empty_like(vq)
    vlse = torch.empty((H, tot), dtype=torch.float32, device=dev)
    vdq, vdk, vdv = torch.empty_like(vq), torch.empty_like(vk), torch.empty_like(vv)
    vws = torch.empty(sdpa.sdpa_bwd_varlen_workspace_size(cu, cu, max(lens), max(lens), H, D),
                      dtype=torch.uint8, device=dev)
    fwd_v = timed(lambda: sdpa.sdpa_fwd_varlen(vq, vk, vv, cu, cu, max(lens), max(lens), 0.0,
                                               True, None, 0, 0, out=vout, lse=vlse), 5)
    bwd_v = timed(lambda: sdpa.sdpa_bwd_varlen(vdo, vq, vk, vv, vout, vlse, cu, cu, max(lens),
                                               max(lens), 0.0, True, 0, 0, dq=vdq, dk=vdk,
                                               dv=vdv, workspace=vws), 5)
    vpairs = sum(n * (n + 1) // 2 for n in lens) * H
    extras["varlen"] = {
        "fwd_ms": fwd_v, "fwd_tflops": 4 * D * vpairs / (fwd_v * 1e-3) / 1e12,
        "bwd_ms": bwd_v, "bwd_tflops": 10 * D * vpairs / (bwd_v * 1e-3) / 1e12,
        "note": f"packed causal batch, lengths {lens}, H{H} D{D}"}
    del vq, vk, vv, vdo, vout, vlse, vdq, vdk, vdv, vws

    # the other named workloads, each pass timed alone (inputs that fit in L2
    # get a 256 MB flush before every call, outside the events)
    for name in ("pages_test", "encoder_dropout", "cross_attn"):
        wl = W.WORKLOADS[name]
        extras[name] = measure_workload(torch, sdpa, wl, dev, peak, stored_bits=True)
        if wl.dropout_p > 0:
            # the same pass without dropout: the dropout's own time
            base = measure_workload(torch, sdpa, W.make_workload(name, dropout_p=0.0), dev, peak)
            extras[name]["p0_fwd_ms"] = base["fwd_ms"]
            extras[name]["p0_bwd_ms"] = base["bwd_ms"]
            extras[name]["alu_fwd"] = philox_alu_bound(wl, "fwd", clock_mhz, extras[name]["fwd_ms"],
                                                       base["fwd_ms"], peak)
            extras[name]["alu_bwd"] = philox_alu_bound(wl, "bwd", clock_mhz, extras[name]["bwd_ms"],
                                                       base["bwd_ms"], peak)
    if sdpa.sdpa_check_device() != 0:
        raise RuntimeError("kernel wait timed out in the extended-entry-point timings")
    return extras


def stored_bits_line(w, fwd_ms, bwd_ms, fwd_redraw_ms, bwd_redraw_ms, nbytes, peak):
    """A dropout pass pair with the keep bits carried from the forward to the
    backward (dropout_bits): the forward also stores its bits, the backward
    reads them instead of drawing, so its roofline is its tensor work alone."""
    f, b = flops(w)
    return {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "step_ms": fwd_ms + bwd_ms,
            "step_ms_redrawn": fwd_redraw_ms + bwd_redraw_ms, "bits_bytes": nbytes,
            "bwd_tflops": b / (bwd_ms * 1e-3) / 1e12,
            "bwd_frac": b / (bwd_ms * 1e-3) / 1e12 / peak,
            "note": "forward stores the keep bits, backward reads them (same mask, same "
                    "results); step_ms_redrawn is the pair that draws them twice"}


def measure_workload(torch, sdpa, w, dev, peak, reps=10, stored_bits=False):
    """Forward and backward of one named workload (BHSE), each call timed by
    its own CUDA events, mean over `reps` calls; with stored_bits (dropout, D
    up to 128) also the pair that carries the keep bits in a buffer."""
    q, k, v, do = (x.to(dev) for x in cached_inputs(w))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(sdpa.sdpa_bwd_workspace_size(w.B, w.H, w.Sq, w.Sk, w.D), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev) if small_l2(w) else None
    def time_pair(fwd, bwd):
        for _ in range(3):
            fwd()
            bwd()
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(reps)]
        torch.cuda.synchronize()
        for i in range(reps):
            if flush is not None:
                flush.fill_(float(i))
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            if flush is not None:
                flush.fill_(float(i) + 0.5)
            ev[i][2].record(stream)
            bwd()
            ev[i][3].record(stream)
        torch.cuda.synchronize()
        return (statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
                statistics.mean(e[2].elapsed_time(e[3]) for e in ev))

    fwd_ms, bwd_ms = time_pair(
        lambda: sdpa.sdpa_fwd(q, k, v, w.dropout_p, w.is_causal, None, w.seed, w.offset,
                              out=out, lse=lse),
        lambda: sdpa.sdpa_bwd(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed, w.offset,
                              None, dq=dq, dk=dk, dv=dv, workspace=ws))
    flushed = flush is not None
    line = _pass_line(w, fwd_ms, bwd_ms, workload_config(w)["workload"] +
                      ("; L2 flushed before each call" if flushed else ""), peak)
    if stored_bits and w.dropout_p > 0 and w.D <= 128:
        bits = torch.empty(sdpa.sdpa_dropout_bits_size(w.B, w.H, w.Sq, w.Sk) // 4,
                           dtype=torch.int32, device=dev)
        fs, bs = time_pair(
            lambda: sdpa.sdpa_fwd_ex(q, k, v, w.dropout_p, w.is_causal, None, w.seed, w.offset,
                                     out=out, lse=lse, dropout_bits=bits),
            lambda: sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed,
                                     w.offset, dq=dq, dk=dk, dv=dv, workspace=ws,
                                     dropout_bits=bits))
        line["stored_bits"] = stored_bits_line(w, fs, bs, fwd_ms, bwd_ms, bits.numel() * 4, peak)
    return line


def measure_e2e(torch, sdpa, w, dev, stream, inputs_cpu, q, k, v, lse, ws, world):
    """The step through the public API with host buffers (pinned), copies
    inside the timed region."""
    f_fwd, f_bwd = flops(w)
    pin = lambda t: t.pin_memory()
    hq, hk, hv, hdo = (pin(x) for x in inputs_cpu)
    hout, hdq, hdk, hdv = (torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (q, q, k, v))
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo))
    d2h = sum(x.numel() * x.element_size() for x in (hout, hlse, hdq, hdk, hdv))

    # Steps are pipelined over three streams through the public API, with
    # NB sets of device tensors (ordered by events): q, k, v are uploaded
    # before dout so that the forward starts first, out and lse are
    # downloaded while the backward runs, and dq, dk, dv after it. Every
    # step still copies its whole input set in and its whole result out.
    NB = 3
    up, down, comp = torch.cuda.Stream(dev), torch.cuda.Stream(dev), stream
    hres = [tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (q, lse, q, k, v))
            for _ in range(NB)]
    hres[0] = (hout, hlse, hdq, hdk, hdv)
    dins = [tuple(torch.empty_like(x, device=dev) for x in (hq, hk, hv, hdo)) for _ in range(NB)]
    douts = [(torch.empty_like(q), torch.empty_like(lse), torch.empty_like(q), torch.empty_like(k),
              torch.empty_like(v)) for _ in range(NB)]
    ev = {n: [torch.cuda.Event() for _ in range(NB)]
          for n in ("qkv", "in", "fwd", "done", "out1", "out2")}
    started = [False] * NB

    def e2e_step(t):
        bsel = t % NB
        di, do_, ho = dins[bsel], douts[bsel], hres[bsel]
        with torch.cuda.stream(up):
            if started[bsel]:
                up.wait_event(ev["done"][bsel])  # step t-NB has finished reading di
            for src, dst in zip((hq, hk, hv), di[:3]):
                dst.copy_(src, non_blocking=True)
            ev["qkv"][bsel].record(up)
            di[3].copy_(hdo, non_blocking=True)
            ev["in"][bsel].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(ev["qkv"][bsel])
            if started[bsel]:
                comp.wait_event(ev["out1"][bsel])  # step t-NB's out, lse are downloaded
            gq, gk, gv, gdo = di
            o, l, dq_, dk_, dv_ = do_
            _, _, s_, off_ = sdpa.sdpa_fwd(gq, gk, gv, w.dropout_p, w.is_causal, None, w.seed,
                                           w.offset, out=o, lse=l)
            ev["fwd"][bsel].record(comp)
            comp.wait_event(ev["in"][bsel])
            if started[bsel]:
                comp.wait_event(ev["out2"][bsel])  # step t-NB's dq, dk, dv are downloaded
            sdpa.sdpa_bwd(gdo, gq, gk, gv, o, l, w.dropout_p, w.is_causal, s_, off_, None,
                          dq=dq_, dk=dk_, dv=dv_, workspace=ws)
            ev["done"][bsel].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev["fwd"][bsel])
            for src, dst in zip(do_[:2], ho[:2]):
                dst.copy_(src, non_blocking=True)
            ev["out1"][bsel].record(down)
            down.wait_event(ev["done"][bsel])
            for src, dst in zip(do_[2:], ho[2:]):
                dst.copy_(src, non_blocking=True)
            ev["out2"][bsel].record(down)
        started[bsel] = True

    e2e_steps = 40
    for t in range(NB):
        e2e_step(t)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for t in range(e2e_steps):
        e2e_step(t)
    torch.cuda.synchronize()
    e2e_ms = barrier_max((time.perf_counter() - t0) * 1e3, world) / e2e_steps

    # the same copies alone (uploads and downloads concurrently, no kernels):
    # the host link's bound on the step
    def copies_only(t):
        bsel = t % NB
        di, do_, ho = dins[bsel], douts[bsel], hres[bsel]
        with torch.cuda.stream(up):
            for src, dst in zip((hq, hk, hv, hdo), di):
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(down):
            for src, dst in zip(do_, ho):
                dst.copy_(src, non_blocking=True)

    for t in range(NB):
        copies_only(t)
    torch.cuda.synchronize()
    # the fastest of three loops: inside this process the copies-alone loop
    # now and then ran far slower than the same copies in a fresh process
    # (3.2 ms per step there), while the pipelined step above did not
    runs = []
    for _ in range(3):
        t0 = time.perf_counter()
        for t in range(e2e_steps // 3):
            copies_only(t)
        torch.cuda.synchronize()
        runs.append((time.perf_counter() - t0) * 1e3 / (e2e_steps // 3))
    copy_ms = barrier_max(min(runs), world)
    return {"value": world * (f_fwd + f_bwd) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "copies_declared": True,
            "copy_bound": {"ms_per_step": copy_ms, "frac": copy_ms / e2e_ms,
                           "runs_ms": runs,
                           "note": "the step's uploads and downloads alone, concurrently on "
                                   "two streams (no kernels), the fastest of three loops: the "
                                   "host link's bound"},
            "timing": "host wall clock around 40 pipelined steps, synchronised on both sides"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sustain-seconds", type=float, default=3.0,
                    help="length of the back-to-back sustained loop after the timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the extended entry points and the other workloads")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (small cases for profiling; not a bench line)")
    ap.add_argument("--dropout", type=float, default=None,
                    help="override dropout_p (profiling the dropout path; not a bench line)")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="override D (profiling other head dims; not a bench line)")
    ap.add_argument("--bias", choices=["relpos"], default=None,
                    help="add a relative-position bias [1, H, Sq, Sk] to every call (profiling "
                         "the bias path; not a bench line)")
    ap.add_argument("--stored-bits", action="store_true",
                    help="carry the dropout keep bits from forward to backward in a buffer "
                         "(profiling that path; not a bench line)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="another named workload of the package's workloads module (its own "
                         "shape; the bench line is the default one)")
    args = ap.parse_args(argv)
    from scaled_dot_product_07_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    over = {}
    if args.batch is not None:
        over["B"] = args.batch
    if args.dropout is not None:
        over["dropout_p"] = args.dropout
    if args.head_dim is not None:
        over["D"] = args.head_dim
    if over:
        w = W.make_workload(args.workload, **over)
    if args.impl == "reference":
        return bench_reference(args, w)
    return bench_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
