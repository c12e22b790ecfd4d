"""Benchmark of the exact tiled attention path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2|3|4|5]
                    [--impl ours|reference]

Default workload 3, long-context causal prefill B=1 H=16 T=S=32768 D=128
bf16 with Q x 2: one step is one prefill forward (O and LSE) over that
sequence.  The line also carries a ``decode`` block for workload 4, the GQA
KV-cache decode step (B=64, Hq=32, Hkv=8, D=128, cache lengths U[1024,8192]:
append the new token's K/V, then decode), with its own roofline, end-to-end
figure and CPU baseline: the metric names both halves.  ``--workload 2``
times the short causal prefill plus the next-token append and decode of the
same batch; ``--workload 5`` the padded batch prefill; ``--workload 4`` the
decode step alone.  Inputs are seeded synthetic tensors already resident in
HBM; L2 is flushed (256 MiB write) between timed prefill steps, outside the
timed events; the decode steps, which each read a 1.3 GB cache (ten times
L2), are timed back to back in one CUDA graph, and the flushed per-step
figure is reported beside them.

Printed: ONE JSON line (rank 0) with the metric, whole-job throughput, the
roofline of the dominant kernel (its own CUDA-event time), an end-to-end
figure through the public API with host buffers (the prefill through
attn_fwd_host, whose copies overlap the compute; the serial copy / call
breakdown beside it), the float64 CPU oracle timed on the host cores, SM
clocks sampled during the timed region and the number of library kernels
launched.

``--impl reference`` times the float64 CPU oracle (the reference arm; there
is no installable reference implementation) on bounded samples of the same
workload and prints the same metric with ``"impl": "reference"``.
N > 1 (torchrun) runs one independent replica per GPU: no collective on the
data path, a barrier and a max-over-ranks reduction of the timed region only.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOPS vs tensor peak; decode KV-read GB/s vs HBM peak"
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "source": "fallback"}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# each workload's dominant kernel, from the ncu captures summarised under
# profiles/, keyed by workload id.  Each entry records the sha256 prefix of
# the kernel source it was measured on; when the source has changed since,
# the figure no longer describes the kernel and the bench reports null.
# "scale" converts the captured launch to a full launch of the bench
# workload by the units it processes (1.0 when captured at full size).
PROFILED_TRAFFIC = {
    2: {"source": "exact_tiled_attention_49_b300/csrc/fwd_bf16_tc.cuh", "sha256": "103911b9e59f",
        "bytes": 12.65792e6 + 0.0, "scale": 1.0,
        "capture": "fwd_bf16_tc_kernel<64,0,0>, full workload"},
    3: {"source": "exact_tiled_attention_49_b300/csrc/fwd_bf16_tc.cuh", "sha256": "103911b9e59f",
        "bytes": 2237.750528e6 + 119.620608e6, "scale": 1.0,
        "capture": "fwd_bf16_tc_kernel<128,0,0>, full workload"},
    5: {"source": "exact_tiled_attention_49_b300/csrc/fwd_bf16_tc.cuh", "sha256": "103911b9e59f",
        "bytes": 1082.855168e6 + 90.0608e6, "scale": 1.0,
        "capture": "fwd_bf16_tc_kernel<128,0,0>, full workload"},
    4: {"source": "exact_tiled_attention_49_b300/csrc/decode.cuh", "sha256": "69704c0ae728",
        "bytes": 1339.805952e6 + 4.4928e6 + 3.42272e6, "scale": 1.0,
        "capture": "decode_split_mma_kernel<128,4,0> (append fused) + "
                   "decode_combine_spans_kernel, full workload"},
}


def source_sha(rel):
    import hashlib
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return ""


def profiled_traffic(wid):
    """Measured DRAM bytes per launch of workload `wid`'s dominant kernel, or
    None when there is no capture of the kernel as it stands."""
    e = PROFILED_TRAFFIC.get(wid)
    if e is None or not source_sha(e["source"]).startswith(e["sha256"]):
        return None
    return e["bytes"] * e["scale"]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int, device=None) -> float:
    """Max of a float over ranks (identity for one process)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class _NvmlCtypes:
    """The few NVML calls the clock sampler needs, bound with ctypes to the
    driver's libnvidia-ml.so.1 (for hosts where the pynvml module is not
    importable).  Same method names and results as pynvml's."""

    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._chk(self.lib.nvmlInit_v2())

    def _chk(self, rc):
        if rc != 0:
            raise RuntimeError(f"NVML error {rc}")

    def nvmlInit(self):
        pass

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self.ct.c_void_p()
        self._chk(self.lib.nvmlDeviceGetHandleByPciBusId_v2(self.ct.c_char_p(bus),
                                                            self.ct.byref(h)))
        return h

    def nvmlDeviceGetHandleByIndex(self, i):
        h = self.ct.c_void_p()
        self._chk(self.lib.nvmlDeviceGetHandleByIndex_v2(self.ct.c_uint(i), self.ct.byref(h)))
        return h

    def nvmlDeviceGetIndex(self, h):
        v = self.ct.c_uint()
        self._chk(self.lib.nvmlDeviceGetIndex(h, self.ct.byref(v)))
        return v.value

    def _clock(self, fn, h, typ):
        v = self.ct.c_uint()
        self._chk(fn(h, self.ct.c_int(typ), self.ct.byref(v)))
        return v.value

    def nvmlDeviceGetMaxClockInfo(self, h, typ):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo, h, typ)

    def nvmlDeviceGetClockInfo(self, h, typ):
        return self._clock(self.lib.nvmlDeviceGetClockInfo, h, typ)

    def _uint(self, fn, h):
        v = self.ct.c_uint()
        self._chk(fn(h, self.ct.byref(v)))
        return v.value

    def nvmlDeviceGetPowerUsage(self, h):
        return self._uint(self.lib.nvmlDeviceGetPowerUsage, h)

    def nvmlDeviceGetEnforcedPowerLimit(self, h):
        return self._uint(self.lib.nvmlDeviceGetEnforcedPowerLimit, h)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.ct.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._chk(fn(h, self.ct.byref(v)))
        return v.value


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons of one GPU while
    the timed region runs: NVML every 2 ms (the pynvml module, else the
    driver's NVML library through ctypes), plus one sample at entry and one
    at exit; if NVML is unavailable, nvidia-smi queries instead."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2,
        "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sync_boost": 0x10,
        "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80, "display_clock_setting": 0x100,
    }

    def __init__(self, device, period_s: float = 0.002):
        self.period = period_s
        self.samples, self.reasons = [], set()
        self.power_w = []
        self.limit_w = None
        self.mask = 0
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thr = None
        self.mode = None
        self.smi_index = str(device.index)
        try:
            try:
                import pynvml
                pynvml.nvmlInit()
            except ImportError:
                pynvml = _NvmlCtypes()
            self.nv = pynvml
            self.h = None
            try:
                import torch
                pr = torch.cuda.get_device_properties(device)
                bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
                self.h = pynvml.nvmlDeviceGetHandleByPciBusId(bus.encode())
            except Exception:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(device.index)
            self.smi_index = str(pynvml.nvmlDeviceGetIndex(self.h))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self._reasons_fn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.mode = "nvml" if not isinstance(pynvml, _NvmlCtypes) else "nvml-ctypes"
            try:
                self.limit_w = pynvml.nvmlDeviceGetEnforcedPowerLimit(self.h) / 1000.0
            except Exception:
                self.limit_w = None
        except Exception as e:  # fall back to nvidia-smi
            self.error = f"nvml: {type(e).__name__}: {e}"
            self.mode = "smi"

    def _sample_nvml(self):
        self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
        mask = self._reasons_fn(self.h)
        self.mask |= int(mask)
        for name, bit in self.REASONS.items():
            if mask & bit:
                self.reasons.add(name)
        try:
            self.power_w.append(self.nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0)
        except Exception:
            pass

    def _sample_smi(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown")
        out = subprocess.run(["nvidia-smi", "-i", self.smi_index, f"--query-gpu={q}",
                              "--format=csv,noheader,nounits"], capture_output=True,
                             text=True, timeout=10).stdout.strip().split(",")
        self.samples.append(float(out[0]))
        self.max_mhz = float(out[1])
        for name, flag in zip(["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown",
                               "hw_thermal_slowdown"], out[2:]):
            if flag.strip().lower() == "active":
                self.reasons.add(name)

    def sample(self):
        try:
            (self._sample_smi if self.mode == "smi" else self._sample_nvml)()
        except Exception as e:
            self.error = f"{self.mode}: {type(e).__name__}: {e}"

    def _run(self):
        while not self._stop.wait(0.05 if self.mode == "smi" else self.period):
            self.sample()

    def __enter__(self):
        self.sample()
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._thr.join()
        self.sample()

    def record(self):
        rec = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples), "source": self.mode}
        if self.mode != "smi":
            rec["reasons_mask"] = hex(self.mask)  # union of NVML's clock-event bits
        if self.power_w:
            # NVML's board power is a trailing average (about a second): it
            # lags a short timed region
            rec["power_w_trailing_avg"] = statistics.median(self.power_w)
        if self.limit_w:
            rec["power_limit_w"] = self.limit_w
        if self.error:
            rec["error"] = self.error
        return rec


# -------------------------------------------------------------- workloads

def workloads_kind(wid):
    import workloads
    return workloads.WORKLOADS[wid].kind


def prefill_flops(w, key_lens=None):
    """Algorithmic FLOPs of one prefill forward: 4*B*H*T*S*D for full
    attention, the unmasked half 2*B*H*T*S*D for causal, and 2*H*D*sum(L^2)
    for causal with key padding ("Implementing attention from scratch", Cost
    model: the two products cost about 4*B*H*T*S*D)."""
    if key_lens is not None and w.causal:
        return 2.0 * w.Hq * w.D * float(sum(int(x) ** 2 for x in key_lens))
    f = 4.0 * w.B * w.Hq * w.T * w.S * w.D
    return f / 2 if w.causal else f


def decode_bytes(Hkv, D, kv_lens, elem=2):
    """Algorithmic KV bytes one decode step must read: K and V rows of every
    valid cache position, once per KV head."""
    return float(sum(int(x) for x in kv_lens)) * Hkv * D * 2 * elem


def decode_flops(Hq, D, kv_lens):
    return 4.0 * Hq * D * float(sum(int(x) for x in kv_lens))


def quantize_e4m3(t):
    """Per-tensor E4M3 quantisation (descale = amax / 256): (fp8 tensor, descale)."""
    import torch
    x = t.float()
    d = float(x.abs().max()) / 256.0
    return (x / d).to(torch.float8_e4m3fn), d


def build_case(wid, device, batch=None, backward=False, fp8=False):
    """Device tensors for one step of workload `wid` and its bookkeeping.
    With `backward`, the step is the backward pass of the prefill (its O and
    LSE computed once, outside the timed region); with `fp8`, the prefill on
    the inputs quantised to E4M3 per tensor (quantised once, outside)."""
    import torch
    import workloads
    w = workloads.workload(wid, batch)
    case = {"w": w, "wid": wid}
    if w.kind == "prefill":
        x = workloads.workload_inputs(wid, device=device, batch=batch)
        case.update(x)
        case["o"] = torch.empty_like(x["q"])
        case["lse"] = torch.empty(w.B, w.Hq, w.T, device=device, dtype=torch.float32)
        kl = None if x["key_lens"] is None else x["key_lens"].cpu().numpy()
        case["flops"] = prefill_flops(w, kl)
        if fp8:
            f = {}
            for n in ("q", "k", "v"):
                f[n], f["d" + n] = quantize_e4m3(x[n])
            case["fp8"] = f
            case["o"] = torch.empty(x["q"].shape, dtype=torch.bfloat16, device=device)
            return case
        if backward:
            import exact_tiled_attention_49_b300 as E
            scale = 1.0 / math.sqrt(w.D)
            o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=w.causal,
                                key_lens=x["key_lens"], scale=scale)
            g = torch.Generator(device=device).manual_seed(100 + wid)
            case["bwd"] = {
                "o": o, "lse": lse,
                "do": torch.randn(x["q"].shape, generator=g, device=device).to(x["q"].dtype),
                "ws": torch.empty(E.attn_bwd_workspace_size(w.B, w.Hq, w.T), dtype=torch.uint8,
                                  device=device),
                "dq": torch.empty_like(x["q"]), "dk": torch.empty_like(x["k"]),
                "dv": torch.empty_like(x["v"])}
            case["flops"] = 2.5 * prefill_flops(w, kl)
            return case
        if wid == 2:
            # the next generation step for the same batch: cache = prompt K/V
            s_max = w.S + 1
            kc = torch.zeros(w.B, w.Hkv, s_max, w.D, device=device, dtype=x["k"].dtype)
            vc = torch.zeros_like(kc)
            kc[:, :, :w.S] = x["k"]
            vc[:, :, :w.S] = x["v"]
            g = torch.Generator(device=device).manual_seed(1002)
            case["dec"] = {
                "q": torch.randn(w.B, w.Hq, w.D, generator=g, device=device).to(x["q"].dtype),
                "k_new": torch.randn(w.B, w.Hkv, w.D, generator=g, device=device).to(x["q"].dtype),
                "v_new": torch.randn(w.B, w.Hkv, w.D, generator=g, device=device).to(x["q"].dtype),
                "kcache": kc, "vcache": vc,
                "pos": torch.full((w.B,), w.S, dtype=torch.int32, device=device),
                "kv_len": torch.full((w.B,), w.S + 1, dtype=torch.int32, device=device),
            }
            d = case["dec"]
            d["o"] = torch.empty_like(d["q"])
            d["lse"] = torch.empty(w.B, w.Hq, device=device, dtype=torch.float32)
            from exact_tiled_attention_49_b300 import attn_decode_workspace_size
            d["ws"] = torch.empty(attn_decode_workspace_size(w.B, w.Hq, s_max, w.D),
                                  device=device, dtype=torch.uint8)
            kv = [w.S + 1] * w.B
            case["dec_bytes"] = decode_bytes(w.Hkv, w.D, kv)
            case["flops"] += decode_flops(w.Hq, w.D, kv)
    else:
        d = workloads.workload_inputs(wid, device=device, batch=batch)
        case.update(d)
        case["o"] = torch.empty_like(d["q"])
        case["lse"] = torch.empty(w.B, w.Hq, device=device, dtype=torch.float32)
        from exact_tiled_attention_49_b300 import attn_decode_workspace_size
        case["ws"] = torch.empty(attn_decode_workspace_size(w.B, w.Hq, d["S_max"], w.D),
                                 device=device, dtype=torch.uint8)
        kv = d["kv_len"].cpu().numpy()
        case["dec_bytes"] = decode_bytes(w.Hkv, w.D, kv)
        case["flops"] = decode_flops(w.Hq, w.D, kv)
    return case


def step_groups(c):
    """Kernel groups of one step, in order: (name, callable issuing them)."""
    import exact_tiled_attention_49_b300 as E
    w = c["w"]
    scale = 1.0 / math.sqrt(w.D)
    groups = []
    if "fp8" in c:
        f = c["fp8"]
        groups.append(("prefill", lambda: E.attn_fwd_fp8(
            f["q"], f["k"], f["v"], o=c["o"], lse=c["lse"], causal=w.causal,
            key_lens=c["key_lens"], scale=scale, q_descale=f["dq"], k_descale=f["dk"],
            v_descale=f["dv"])))
        return groups
    if "bwd" in c:
        bw = c["bwd"]
        groups.append(("prefill", lambda: E.attn_bwd(
            c["q"], c["k"], c["v"], bw["o"], bw["do"], bw["lse"], causal=w.causal,
            key_lens=c["key_lens"], scale=scale, dq=bw["dq"], dk=bw["dk"], dv=bw["dv"],
            workspace=bw["ws"])))
        return groups
    if w.kind == "prefill":
        groups.append(("prefill", lambda: E.attn_fwd(
            c["q"], c["k"], c["v"], o=c["o"], lse=c["lse"], causal=w.causal,
            key_lens=c["key_lens"], scale=scale)))
        if "dec" in c:
            d = c["dec"]

            groups.append(("decode", lambda: E.attn_decode_append(
                d["q"], d["kcache"], d["vcache"], d["k_new"], d["v_new"], d["kv_len"], o=d["o"],
                lse=d["lse"], workspace=d["ws"], scale=scale)))
    else:
        # the decode step: append the new token and decode over the cache
        # including it, in one call (split kernel + merge)
        groups.append(("decode", lambda: E.attn_decode_append(
            c["q"], c["kcache"], c["vcache"], c["k_new"], c["v_new"], c["kv_len"], o=c["o"],
            lse=c["lse"], workspace=c["ws"], scale=scale)))
    return groups


def run_step(E, c):
    """One step issued call by call through the public API."""
    for _, fn in step_groups(c):
        fn()


def capture_graphs(E, c):
    """One CUDA graph per kernel group of the step, captured once and replayed
    in the timed region so that microsecond kernels are not separated by
    host-side launch latency.  Returns [(name, graph)] and the number of
    library kernels one step launches."""
    import torch
    graphs = []
    n0 = E.attn_kernel_launches()
    for name, fn in step_groups(c):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append((name, g))
    torch.cuda.synchronize()
    return graphs, E.attn_kernel_launches() - n0


def time_graphs(E, c, steps, flush, clk=None, sync=None):
    """Warm replays, then `steps` timed replays of the captured kernel groups
    with the L2 flushed before each step (outside the events).  `sync` (the
    cross-rank barrier) runs right before and after the timed steps, each
    time next to a device synchronize.  Returns (per-step ms list, mean ms
    per group, library launches per step)."""
    import torch
    graphs, launches_per_step = capture_graphs(E, c)
    # Warm replays of the captured step for at least 50 ms of device time, so
    # that a microsecond-scale step is not timed while the clocks still ramp
    # up after an idle spell (e.g. the CPU baseline before it).
    t_end = time.perf_counter() + 0.05
    n_warm = 0
    while n_warm < 2 or time.perf_counter() < t_end:
        flush.zero_()
        for _, g in graphs:
            g.replay()
        n_warm += 1
        if n_warm % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    # events[s] = [start, end of group 0, end of group 1, ...]
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
              for _ in range(steps)]
    if sync is not None:
        sync()
    torch.cuda.synchronize()
    if clk is not None:
        clk.__enter__()
    try:
        for s in range(steps):
            flush.zero_()                     # L2 flush, outside the timed events
            events[s][0].record()
            for i, (_, g) in enumerate(graphs):
                g.replay()
                events[s][i + 1].record()
        torch.cuda.synchronize()
    finally:
        if clk is not None:
            clk.__exit__(None, None, None)
    if sync is not None:
        sync()
    step_ms = [ev[0].elapsed_time(ev[-1]) for ev in events]
    kern_ms = {name: sum(ev[i].elapsed_time(ev[i + 1]) for ev in events) / steps
               for i, (name, _) in enumerate(graphs)}
    return step_ms, kern_ms, launches_per_step


def time_stream(E, c, steps, clk=None, sync=None):
    """`steps` steps back to back in one CUDA graph, without an L2 flush
    between them: for the decode step, whose input (the KV cache, 1.3 GB)
    is ten times the L2, so every step reads it from DRAM anyway.  A serving
    loop issues its steps back to back, and so does this timing: each call's
    launch overlaps the previous call's tail (PDL) instead of being timed
    alone.  Returns (ms for all the steps, ms per step, library launches
    per step)."""
    import torch
    groups = step_groups(c)
    n0 = E.attn_kernel_launches()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        for _ in range(steps):
            for _, fn in groups:
                fn()
    launches = (E.attn_kernel_launches() - n0) // steps
    for _ in range(2):
        g_step.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if sync is not None:
        sync()
    torch.cuda.synchronize()
    if clk is not None:
        clk.__enter__()
    try:
        ev[0].record()
        g_step.replay()
        ev[1].record()
        torch.cuda.synchronize()
    finally:
        if clk is not None:
            clk.__exit__(None, None, None)
    if sync is not None:
        sync()
    ms = ev[0].elapsed_time(ev[1])
    return ms, ms / steps, launches


def other_workloads(E, skip, device, steps, peaks):
    """The other benchmark workloads, timed the same way (one entry each):
    the short and padded prefills (and the long-context one when it is not
    the headline), the decode step (when it has no block of its own), the
    backward passes and the E4M3 prefills."""
    import torch
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    for wid in (2, 3, 5, 4):
        if wid in skip:
            continue
        c = build_case(wid, device)
        w = c["w"]
        for _ in range(3):
            flush.zero_()
            run_step(E, c)
        torch.cuda.synchronize()
        clk = ClockSampler(device)
        _, kern_ms, _ = time_graphs(E, c, steps, flush, clk)
        if w.kind == "prefill":
            kl = None if c["key_lens"] is None else c["key_lens"].cpu().numpy()
            v = prefill_flops(w, kl) / (kern_ms["prefill"] * 1e-3) / 1e12
            out[str(wid)] = {"workload": w.name, "value": v, "unit": "TFLOPS",
                             "ms": kern_ms["prefill"], "kernel": "fwd_bf16_tc_kernel",
                             "frac": v / peaks["bf16_tflops"],
                             "traffic": profiled_traffic(wid), "clocks": clk.record()}
            if "dec" in c:
                gbs = c["dec_bytes"] / (kern_ms["decode"] * 1e-3) / 1e9
                out[str(wid)]["next_token_decode"] = {
                    "value": gbs, "unit": "GB/s", "ms": kern_ms["decode"],
                    "kernels": "decode_split_mma_kernel (append fused), "
                               "decode_combine_spans_kernel",
                    "frac": gbs / peaks["hbm_gbs"]}
        else:
            v = c["dec_bytes"] / (kern_ms["decode"] * 1e-3) / 1e9
            out[str(wid)] = {"workload": w.name, "value": v, "unit": "GB/s",
                             "ms": kern_ms["decode"],
                             "kernel": "decode_split_mma_kernel (append fused)"
                                       "+decode_combine_spans_kernel",
                             "frac": v / peaks["hbm_gbs"], "traffic": profiled_traffic(wid),
                             "clocks": clk.record()}
        del c
        torch.cuda.empty_cache()
    out.update(backward_workloads(E, device, steps, peaks, flush))
    out.update(fp8_workloads(E, device, steps, peaks, flush))
    out.update(chunked_workloads(E, device, steps, peaks, flush))
    out.update(shard_workloads(E, device, steps, peaks, flush))
    out.update(long_decode_workloads(E, device, steps, peaks))
    if E.attn_device_error(clear=True) != 0:
        raise RuntimeError("device error while timing the other workloads")
    return out


def fp8_workloads(E, device, steps, peaks, flush):
    """The long-context and padded prefills with E4M3 inputs (attn_fwd_fp8):
    the bf16 inputs of the workload quantised per tensor (descale = amax /
    256), one CUDA-graph replay per step with the L2 flushed.  Throughput is
    against the FP8 dense peak taken as the measured bf16 burst times the
    nominal FP8 / bf16 ratio (4.5 / 2.25 PFLOP/s)."""
    import torch
    import workloads
    out = {}
    peak = 2.0 * peaks["bf16_tflops"]
    for wid in (3, 5):
        w = workloads.WORKLOADS[wid]
        x = workloads.workload_inputs(wid, device=device)
        q8, k8, v8, ds = [], [], [], []
        for n, lst in (("q", q8), ("k", k8), ("v", v8)):
            t = x[n].float()
            d = float(t.abs().max()) / 256.0
            lst.append((t / d).to(torch.float8_e4m3fn))
            ds.append(d)
            del t
        q8, k8, v8 = q8[0], k8[0], v8[0]
        kl = x["key_lens"]
        del x
        o = torch.empty(q8.shape, dtype=torch.bfloat16, device=device)
        lse = torch.empty(q8.shape[:3], dtype=torch.float32, device=device)

        def step():
            E.attn_fwd_fp8(q8, k8, v8, o=o, lse=lse, causal=w.causal, key_lens=kl,
                           scale=1.0 / math.sqrt(w.D), q_descale=ds[0], k_descale=ds[1],
                           v_descale=ds[2])
        for _ in range(3):
            step()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        total = 0.0
        for _ in range(steps):
            flush.zero_()
            e0.record()
            graph.replay()
            e1.record()
            e1.synchronize()
            total += e0.elapsed_time(e1)
        ms = total / steps
        lens = None if kl is None else kl.cpu().numpy()
        flops = prefill_flops(w, lens)
        v = flops / (ms * 1e-3) / 1e12
        out[f"fp8_{wid}"] = {"workload": f"E4M3 inputs: {w.name}", "value": v, "unit": "TFLOPS",
                             "ms": ms, "kernel": "fwd_bf16_tc_kernel<128,0,1>",
                             "frac": v / peak, "peak": peak,
                             "peak_source": "measured bf16 burst x 2 (nominal FP8/bf16 ratio)"}
        del q8, k8, v8, o, lse, graph
        torch.cuda.empty_cache()
    return out


def chunked_workloads(E, device, steps, peaks, flush):
    """Chunked prefill against a KV cache (attn_fwd_chunked): the last 4096
    query rows of the long-context sequence (B=1 H=16 D=128, Q x 2) as a new
    chunk at positions 28672..32767 over its 32768 cached keys, causal.  One
    CUDA-graph replay per step, L2 flushed.  FLOPs: 4 D per visible (query,
    key) pair, each row seeing its own position and every key before it."""
    import numpy as np
    import torch
    import workloads
    w = workloads.WORKLOADS[3]
    x = workloads.workload_inputs(3, device=device)
    T = 4096
    q = x["q"][:, :, w.T - T:].contiguous()
    k, v = x["k"], x["v"]
    del x
    q_pos = torch.full((w.B,), w.S - T, dtype=torch.int32, device=device)
    kv_lens = torch.full((w.B,), w.S, dtype=torch.int32, device=device)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=device)

    def step():
        E.attn_fwd_chunked(q, k, v, q_pos, kv_lens, o=o, lse=lse, causal=True,
                           scale=1.0 / math.sqrt(w.D))
    for _ in range(3):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    total = 0.0
    for _ in range(steps):
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
        e1.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / steps
    pos = np.arange(w.S - T, w.S, dtype=np.float64)
    flops = 4.0 * w.D * w.Hq * w.B * float((pos + 1).sum())
    v_ = flops / (ms * 1e-3) / 1e12
    out = {"chunked_3": {"workload": f"chunked prefill: the last {T} rows of {w.name} as a chunk "
                                     f"at position {w.S - T} against the {w.S}-key cache",
                         "value": v_, "unit": "TFLOPS", "ms": ms,
                         "kernel": "fwd_bf16_tc_kernel<128,0,0> (q_pos)",
                         "frac": v_ / peaks["bf16_tflops"]}}
    del q, k, v, o, lse, graph
    torch.cuda.empty_cache()
    return out


def shard_workloads(E, device, steps, peaks, flush):
    """The single-GPU half of sequence parallelism: the long-context prefill
    (B=1 H=16 T=S=32768 D=128, Q x 2) computed as 4 key shards of 8192 keys
    (attn_fwd_kv_shard at global offsets 0, 8192, 16384, 24576, each
    partial normalised over its shard) and their LSE merge (attn_lse_merge).
    One CUDA graph of the five calls per step, L2 flushed; throughput counts
    the prefill's own FLOPs, so the merge and the shards' tails show as
    the difference from the unsharded prefill."""
    import torch
    import workloads
    w = workloads.WORKLOADS[3]
    x = workloads.workload_inputs(3, device=device)
    n = 4
    S1 = w.S // n
    q = x["q"]
    ks = [x["k"][:, :, i * S1:(i + 1) * S1].contiguous() for i in range(n)]
    vs = [x["v"][:, :, i * S1:(i + 1) * S1].contiguous() for i in range(n)]
    del x
    q_pos = torch.zeros((w.B,), dtype=torch.int32, device=device)
    key_lens = torch.full((w.B,), w.S, dtype=torch.int32, device=device)
    o_parts = torch.empty((n,) + tuple(q.shape), dtype=q.dtype, device=device)
    lse_parts = torch.empty((n,) + tuple(q.shape[:3]), dtype=torch.float32, device=device)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=device)
    scale = 1.0 / math.sqrt(w.D)

    def step():
        for i in range(n):
            E.attn_fwd_kv_shard(q, ks[i], vs[i], q_pos, key_lens, i * S1, o=o_parts[i],
                                lse=lse_parts[i], causal=True, scale=scale)
        E.attn_lse_merge(o_parts, lse_parts, o=o, lse=lse)
    for _ in range(3):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    total = 0.0
    for _ in range(steps):
        flush.zero_()
        e0.record()
        graph.replay()
        e1.record()
        e1.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / steps
    v_ = prefill_flops(w, None) / (ms * 1e-3) / 1e12
    out = {"shard4_3": {"workload": f"{w.name} as {n} key shards of {S1} keys + LSE merge",
                        "value": v_, "unit": "TFLOPS", "ms": ms,
                        "kernel": "fwd_bf16_tc_kernel<128,0,0> (key shards) + lse_merge_kernel",
                        "frac": v_ / peaks["bf16_tflops"]}}
    del q, ks, vs, o_parts, lse_parts, o, lse, graph
    torch.cuda.empty_cache()
    return out


def long_decode_workloads(E, device, steps, peaks):
    """One long sequence: the GQA decode step (Hq=32 Hkv=8 D=128 bf16) of a
    single sequence with 131071 cached tokens plus the new one, where the
    balanced spans split one sequence's 8 streams over every SM.  Steps
    (attn_decode_append) back to back in one CUDA graph (the 537 MB cache is
    four times L2)."""
    import torch
    import workloads
    d = workloads.decode_inputs(1, 32, 8, 128, 131071, 131071, "bf16", seed=9, device=device)
    ws = torch.empty(E.attn_decode_workspace_size(1, 32, d["S_max"], 128), dtype=torch.uint8,
                     device=device)
    o = torch.empty_like(d["q"])
    lse = torch.empty((1, 32), dtype=torch.float32, device=device)
    scale = 1.0 / math.sqrt(128)

    def step():
        E.attn_decode_append(d["q"], d["kcache"], d["vcache"], d["k_new"], d["v_new"], d["kv_len"],
                             o=o, lse=lse, workspace=ws, scale=scale)
    for _ in range(3):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            step()
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = float(d["kv_len"].sum().item()) * 8 * 128 * 2 * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    out = {"decode_long": {"workload": "GQA decode, one sequence of 131072 tokens, Hq=32 Hkv=8 "
                                       "D=128 bf16 (attn_decode_append)",
                           "value": gbs, "unit": "GB/s", "ms": ms,
                           "kernel": "decode_split_mma_kernel<128,4,0>+decode_combine_spans_kernel",
                           "frac": gbs / peaks["hbm_gbs"]}}
    del d, ws, o, lse, graph
    torch.cuda.empty_cache()
    return out


def backward_workloads(E, device, steps, peaks, flush):
    """The backward pass (dQ, dK, dV from the saved LSE) of the long-context,
    padded-batch and short prefills, one CUDA-graph replay per step with the
    L2 flushed.  Throughput counts the algorithmic 2.5x the forward's FLOPs
    (five products against two); the kernels compute S and dP twice, so
    they execute 3.5x."""
    import torch
    import workloads
    out = {}
    for wid in (3, 5, 2):
        w = workloads.WORKLOADS[wid]
        x = workloads.workload_inputs(wid, device=device)
        scale = 1.0 / math.sqrt(w.D)
        kl = x["key_lens"]
        o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=w.causal, key_lens=kl, scale=scale)
        g = torch.Generator(device=device).manual_seed(100 + wid)
        do = torch.randn(x["q"].shape, generator=g, device=device).to(x["q"].dtype)
        ws = torch.empty(E.attn_bwd_workspace_size(w.B, w.Hq, w.T), dtype=torch.uint8,
                         device=device)
        dq, dk, dv = (torch.empty_like(x[n]) for n in ("q", "k", "v"))

        def step():
            E.attn_bwd(x["q"], x["k"], x["v"], o, do, lse, causal=w.causal, key_lens=kl,
                       scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)
        for _ in range(3):
            step()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        total = 0.0
        for _ in range(steps):
            flush.zero_()
            e0.record()
            graph.replay()
            e1.record()
            e1.synchronize()
            total += e0.elapsed_time(e1)
        ms = total / steps
        flops = 2.5 * prefill_flops(w, None if kl is None else kl.cpu().numpy())
        v = flops / (ms * 1e-3) / 1e12
        out[f"bwd{wid}"] = {"workload": f"backward (dQ, dK, dV) of: {w.name}", "value": v,
                            "unit": "TFLOPS", "ms": ms,
                            "kernel": "bwd_delta_kernel+bwd_dq_kernel+bwd_dkdv_kernel",
                            "frac": v / peaks["bf16_tflops"],
                            "flops": "2.5x the forward's (algorithmic)"}
        del x, o, lse, do, ws, dq, dk, dv, kl
        torch.cuda.empty_cache()
    return out


def e2e_buffers(c):
    """(device inputs {name: tensor}, device results [tensor]) of one step as
    a user of the public API sees it: what is copied in from the host before
    the calls and read back after them."""
    w = c["w"]
    if "bwd" in c:
        # backward: inputs q, k, v, dO, O, LSE; results dQ, dK, dV
        bw = c["bwd"]
        return ({"q": c["q"], "k": c["k"], "v": c["v"], "do": bw["do"], "o": bw["o"],
                 "lse": bw["lse"]}, [bw[n] for n in ("dq", "dk", "dv")])
    if "fp8" in c:
        # E4M3 prefill: inputs the quantised q, k, v; results O, LSE
        f = c["fp8"]
        return {n: f[n] for n in ("q", "k", "v")}, [c["o"], c["lse"]]
    if w.kind == "prefill":
        dev_in = {n: c[n] for n in ("q", "k", "v")}
        dev_out = [c["o"], c["lse"]]
        if "dec" in c:
            d = c["dec"]
            dev_in.update({"dec_" + n: d[n] for n in ("q", "k_new", "v_new")})
            dev_out += [d["o"], d["lse"]]
        return dev_in, dev_out
    # decode step: the new token's q, k, v in; O and LSE out (the cache stays
    # resident on the device between steps, as in generation)
    return {n: c[n] for n in ("q", "k_new", "v_new")}, [c["o"], c["lse"]]


def run_e2e(E, c, steps, device):
    """Same step through the public API with pinned host buffers: H2D copy of
    the step's inputs, the library calls, D2H copy of its results, all timed
    on the stream with CUDA events between the three phases.  Returns a dict
    with the mean ms per step, the mean ms of each phase and the bytes."""
    import torch
    dev_in, dev_out = e2e_buffers(c)
    host_in = {n: t.cpu().pin_memory() for n, t in dev_in.items()}
    outs = [(torch.empty(t.shape, dtype=t.dtype).pin_memory(), t) for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(h.numel() * h.element_size() for h, _ in outs)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    for _ in range(3):  # untimed: first-use costs of the copies and calls
        for n, t in dev_in.items():
            t.copy_(host_in[n], non_blocking=True)
        run_step(E, c)
        for h, dv in outs:
            h.copy_(dv, non_blocking=True)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for s in range(steps):
        flush.zero_()
        ev[s][0].record()
        for n, t in dev_in.items():
            t.copy_(host_in[n], non_blocking=True)
        ev[s][1].record()
        run_step(E, c)
        ev[s][2].record()
        for h, dv in outs:
            h.copy_(dv, non_blocking=True)
        ev[s][3].record()
        ev[s][3].synchronize()            # the results are on the host

    def mean(a, b):
        return sum(e[a].elapsed_time(e[b]) for e in ev) / steps
    return {"ms": mean(0, 3), "h2d_ms": mean(0, 1), "call_ms": mean(1, 2),
            "d2h_ms": mean(2, 3), "h2d": h2d, "d2h": d2h}


def run_e2e_host(E, c, steps, device):
    """The prefill step through attn_fwd_host: q, k, v (and key_lens) in
    pinned host memory, O and LSE written to pinned host memory; the library
    pipelines copy-in, compute and copy-out in stages over the compute
    stream and two copy streams.  Timed with CUDA events on the compute
    stream from before the call to after its join; returns the mean ms per
    step, the bytes copied and the stage count."""
    import torch
    w = c["w"]
    host = {n: c[n].cpu().pin_memory() for n in ("q", "k", "v")}
    kl = None if c["key_lens"] is None else c["key_lens"].cpu()
    o = torch.empty(c["o"].shape, dtype=c["o"].dtype, pin_memory=True)
    lse = torch.empty(c["lse"].shape, dtype=torch.float32, pin_memory=True)
    need = E.attn_fwd_host_workspace_size(w.B, w.Hq, w.Hkv, w.T, w.S, w.D, c["q"].dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    cin, cout = torch.cuda.Stream(device), torch.cuda.Stream(device)
    scale = 1.0 / math.sqrt(w.D)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def call():
        E.attn_fwd_host(host["q"], host["k"], host["v"], o=o, lse=lse, causal=w.causal,
                        key_lens=kl, scale=scale, workspace=ws, copy_in=cin, copy_out=cout)
    call()
    torch.cuda.synchronize()
    n0 = E.attn_kernel_launches()
    call()
    torch.cuda.synchronize()
    stages = E.attn_kernel_launches() - n0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for s in range(steps):
        flush.zero_()
        ev[s][0].record()
        call()
        ev[s][1].record()
        ev[s][1].synchronize()            # O and LSE are on the host
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + (0 if kl is None else 4 * w.B)
    d2h = o.numel() * o.element_size() + lse.numel() * 4
    return {"ms": ms, "h2d": h2d, "d2h": d2h, "stages": stages}


_CPU_INPUTS = {}


def cpu_baseline(wid, budget_s=12.0, seed=0):
    """Time the float64 oracle on the host cores over a bounded row sample of
    the workload; returns (value in the metric's unit, unit, cores, sample)."""
    import numpy as np
    import torch
    import oracle
    import workloads
    w = workloads.WORKLOADS[wid]
    cores = oracle.default_threads()
    rng = np.random.default_rng(seed)
    if w.kind == "prefill":
        if wid not in _CPU_INPUTS:   # drawn once per process (the reference arm calls again)
            if wid in (2,):
                x = workloads.workload_inputs(wid, device="cpu")
            else:  # same shapes; a smaller batch keeps host memory modest
                x = workloads.prefill_inputs(1, w.Hq, w.Hkv, w.T, w.S, w.D, w.dtype, seed=wid,
                                             q_scale=w.q_scale)
            arr = [workloads.to_numpy_exact(x[n])[0] for n in ("q", "k", "v")]
            lens = x["key_lens"].numpy() if x["key_lens"] is not None else None
            if lens is None and w.lens is not None:
                lens = workloads.lengths(wid, w.lens[0], w.lens[1], arr[0].shape[0])
            _CPU_INPUTS[wid] = (arr, lens)
        arr, lens = _CPU_INPUTS[wid]
        Bx = arr[0].shape[0]
        n_rows_total = Bx * w.Hq * w.T
        done_flops, t_used, rows_done = 0.0, 0.0, 0
        chunk = 256
        while t_used < budget_s:
            rows = rng.integers(0, n_rows_total, size=chunk).astype(np.int64)
            t0 = time.perf_counter()
            oracle.attn_fwd(*arr, causal=w.causal, key_lens=lens, scale=1 / math.sqrt(w.D),
                            bf16=True, rows=rows, nthreads=cores)
            t_used += time.perf_counter() - t0
            rows_done += chunk
            i = rows % w.T
            b = rows // (w.Hq * w.T)
            L = np.full_like(i, w.S) if lens is None else np.asarray(lens)[b]
            vis = np.minimum(L, i + (w.S - w.T) + 1) if w.causal else L
            vis = np.where(i + (w.S - w.T) < L, np.maximum(vis, 0), 0)
            # 4*D FLOPs per visible key (q.k and p*v), the per-row form of
            # the cost model; for causal rows this is the unmasked half.
            done_flops += float((4.0 * w.D * vis).sum())
            chunk = min(chunk * 2, 8192)
        return done_flops / t_used / 1e12, "TFLOPS", cores, \
            f"{rows_done} random query rows of {w.name} (visible-key FLOPs), {t_used:.1f} s"
    if wid not in _CPU_INPUTS:
        d = workloads.decode_inputs(8, w.Hq, w.Hkv, w.D, w.lens[0], w.lens[1], w.dtype, seed=wid)
        _CPU_INPUTS[wid] = ([workloads.to_numpy_exact(d[n])[0] for n in ("q", "kcache", "vcache")],
                            d["kv_len"].numpy())
    arr, kv = _CPU_INPUTS[wid]
    t_used, nbytes, reps = 0.0, 0.0, 0
    while t_used < budget_s:
        t0 = time.perf_counter()
        oracle.attn_decode(*arr, kv, scale=1 / math.sqrt(w.D), bf16=True, nthreads=cores)
        t_used += time.perf_counter() - t0
        nbytes += decode_bytes(w.Hkv, w.D, kv)
        reps += 1
    return nbytes / t_used / 1e9, "GB/s", cores, \
        f"{reps} decode steps of an 8-sequence batch of {w.name}, {t_used:.1f} s"


def cpu_baseline_bwd(wid, budget_s=12.0, seed=0):
    """Time the float64 oracle's backward on the host over a bounded sample:
    whole (b, kv-head group) slices of the prefill workload, one at a time.
    Counts 2.5x the forward's visible-key FLOPs, the GPU line's unit."""
    import numpy as np
    import oracle
    import workloads
    w = workloads.WORKLOADS[wid]
    G = w.Hq // w.Hkv
    # the dense float64 matrices of a 32k x 32k slice would take 8.6 GB each:
    # long sequences are sampled as their first 4096 x 4096 causal block
    T, S = min(w.T, 4096), min(w.S, 4096)
    x = workloads.prefill_inputs(1, G, 1, T, S, w.D, w.dtype, seed=wid, q_scale=w.q_scale)
    q, k, v = (workloads.to_numpy_exact(x[n])[0] for n in ("q", "k", "v"))
    rng = np.random.default_rng(seed)
    do = rng.standard_normal(q.shape)
    lo_hi = None if w.lens is None else (min(w.lens[0], S), min(w.lens[1], S))
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except ImportError:
        cores = 1
    t_used, flops, slices = 0.0, 0.0, 0
    while t_used < budget_s:
        L = S if lo_hi is None else int(rng.integers(lo_hi[0], lo_hi[1] + 1))
        t0 = time.perf_counter()
        oracle.attn_bwd_np(q, k, v, do, causal=w.causal, key_lens=np.array([L]),
                           scale=1 / math.sqrt(w.D), bf16=True)
        t_used += time.perf_counter() - t0
        i = np.arange(T)
        vis = np.minimum(L, i + (S - T) + 1) if w.causal else np.full(T, L)
        vis = np.where(i + (S - T) < L, np.maximum(vis, 0), 0)
        flops += 2.5 * float((4.0 * w.D * vis).sum()) * G
        slices += 1
    return flops / t_used / 1e12, "TFLOPS", cores, \
        (f"{slices} single (b, kv-head group of {G}) backward slices, T={T} S={S}, "
         f"of {w.name}, {t_used:.1f} s")


# ------------------------------------------------------------------- arms

def measure_block(E, args, wid, device, peaks, ws, rank, backward=False, fp8=False,
                  batch=None):
    """One workload measured for the JSON line: warm-up steps, K timed steps
    (CUDA-graph replays, L2 flushed between steps -- for the decode step, whose
    cache is far larger than L2, the K steps back to back in one graph, with
    the flushed per-step timing reported beside it -- clocks sampled, barrier
    and max over ranks), the roofline of its dominant kernel, the end-to-end
    figure through the public API, and (rank 0) the float64 oracle timed on
    the host cores.  Returns the block's dict."""
    import torch
    c = build_case(wid, device, batch, backward=backward, fp8=fp8)
    w = c["w"]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    for _ in range(args.warmup):
        flush.zero_()
        run_step(E, c)
    torch.cuda.synchronize()
    if E.attn_device_error(clear=True) != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    clk = ClockSampler(device)
    isolated = None
    if w.kind == "decode":
        # each step alone after an L2 flush (reported), then the K steps back
        # to back (the value): the cache is far larger than L2
        step_ms, kern_ms, launches_per_step = time_graphs(E, c, K, flush, ClockSampler(device))
        isolated = {"ms_per_step": sum(step_ms) / K,
                    "value": c["dec_bytes"] / (sum(step_ms) / K * 1e-3) / 1e9,
                    "timing": "each step alone: L2 flushed before it, CUDA events around "
                              "its graph replays"}
        tot_ms, dec_ms, launches_per_step = time_stream(E, c, K, clk, sync=lambda: barrier(ws))
        total_ms = reduce_max(tot_ms, ws, device)
        kern_ms = {"decode": dec_ms}
    else:
        step_ms, kern_ms, launches_per_step = time_graphs(E, c, K, flush, clk,
                                                          sync=lambda: barrier(ws))
        total_ms = reduce_max(sum(step_ms), ws, device)
    if E.attn_device_error(clear=True) != 0:
        raise RuntimeError("device error during the timed region")
    ms_per_step = total_ms / K
    out = {"value": None, "unit": None, "ms_per_step": ms_per_step, "dtype": "bf16"}
    if w.kind == "prefill":
        out["value"] = c["flops"] * ws / (ms_per_step * 1e-3) / 1e12
        out["unit"] = "TFLOPS"
        kl = None if c["key_lens"] is None else c["key_lens"].cpu().numpy()
        achieved = (c["flops"] if "bwd" in c else prefill_flops(w, kl)) \
            / (kern_ms["prefill"] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        kernel = ("bwd_delta_kernel+bwd_dq_kernel+bwd_dkdv_kernel" if "bwd" in c else
                  "fwd_bf16_tc_kernel<128,0,1>" if "fp8" in c else
                  f"fwd_bf16_tc_kernel<{w.D},0,0>")
        peak_source = peaks["source"] + " bf16 burst (kernel timed alone)"
        if "fp8" in c:
            # a contraction takes the peak of its own type: the measured bf16
            # burst times the nominal FP8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
            peak *= 2.0
            peak_source += " x 2 (nominal FP8/bf16 ratio)"
            out["dtype"] = "e4m3"
        traffic = profiled_traffic(wid) if batch is None and not backward and not fp8 else None
        out["roofline"] = {"kernel": kernel, "bound": "tensor",
                           "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                           "frac": achieved / peak, "traffic": traffic,
                           "peak_source": peak_source, "kernel_ms": kern_ms["prefill"]}
        if "dec" in c:
            gbs = c["dec_bytes"] / (kern_ms["decode"] * 1e-3) / 1e9
            out["next_token_decode"] = {
                "workload": "next-token append + decode of the same batch (kv_len 1025)",
                "ms": kern_ms["decode"], "value": gbs, "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"]}
    else:
        out["value"] = c["dec_bytes"] * ws / (ms_per_step * 1e-3) / 1e9
        out["unit"] = "GB/s"
        achieved = c["dec_bytes"] / (kern_ms["decode"] * 1e-3) / 1e9
        out["roofline"] = {"kernel": "decode_split_mma_kernel (new token's K/V written in it)"
                                     "+decode_combine_spans_kernel",
                           "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                           "traffic": profiled_traffic(wid) if batch is None else None,
                           "peak_source": peaks["source"] + " HBM copy",
                           "kernel_ms": kern_ms["decode"]}
        out["isolated_step"] = isolated
    cfg = {"workload": ("backward (dQ, dK, dV, 2.5x the forward's FLOPs) of: " + w.name
                        if "bwd" in c else
                        "E4M3 inputs (per-tensor descales): " + w.name if "fp8" in c else w.name),
           "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
           "l2": "flushed between steps (256 MiB write, outside the timed events)",
           "timing": "CUDA events around CUDA-graph replays of each kernel group of the step",
           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
           "algorithmic_work_per_step": c["flops"] if w.kind == "prefill" else c["dec_bytes"]}
    if w.kind == "prefill":
        cfg.update({"T": w.T, "S": w.S, "causal": w.causal,
                    "key_lens": None if w.lens is None else f"U[{w.lens[0]},{w.lens[1]}]"})
        if w.q_scale != 1.0:
            cfg["q_scale"] = w.q_scale
    else:
        cfg.update({"cache_len": f"U[{w.lens[0]},{w.lens[1]}]", "S_max": c["S_max"],
                    "kv_bytes_per_step": c["dec_bytes"],
                    "l2": "not flushed: the K steps run back to back and each reads "
                          f"{c['dec_bytes'] / 1e9:.2f} GB of K/V, ten times the 126 MB L2 "
                          "(isolated_step: flushed)",
                    "timing": "CUDA events around one CUDA graph of the K steps back to back "
                              "(each step one attn_decode_append call: append + decode)"})
    out["config"] = cfg
    out["gpu_launches"] = int(launches_per_step * K)
    out["clocks"] = clk.record()
    if out["roofline"]["bound"] == "tensor":
        # The burst peak was measured at full clocks; a prefill timed over
        # many steps runs into the 1100 W cap (sw_power_cap, ~1.46-1.54 GHz
        # for the long-context kernel), the regime of the sustained peak.
        r = out["roofline"]
        f8 = 2.0 if "fp8" in c else 1.0
        r["peak_sustained"] = peaks["bf16_tflops_sustained"] * f8
        r["frac_sustained"] = r["achieved"] / r["peak_sustained"]

    if not args.no_e2e:
        # End to end through the public API with host buffers.  A plain
        # prefill step goes through attn_fwd_host (copies pipelined with the
        # compute); the serial form (torch copies, then the device-pointer
        # calls, then the copies back) is reported beside it.
        n_e2e = max(3, min(K, 20))
        e = run_e2e(E, c, n_e2e, device)
        work = c["flops"] if w.kind == "prefill" else c["dec_bytes"]
        scale = 1e12 if w.kind == "prefill" else 1e9
        serial = {"ms_per_step": reduce_max(e["ms"], ws, device),
                  "breakdown_ms": {"h2d_copies": e["h2d_ms"], "library_calls": e["call_ms"],
                                   "d2h_copies": e["d2h_ms"]},
                  "copy_gbs": (e["h2d"] + e["d2h"]) / ((e["h2d_ms"] + e["d2h_ms"]) * 1e-3) / 1e9}
        if w.kind == "prefill" and not any(x in c for x in ("dec", "fp8", "bwd")):
            eh = run_e2e_host(E, c, n_e2e, device)
            e2e_ms = reduce_max(eh["ms"], ws, device)
            out["e2e"] = {"value": work * ws / (e2e_ms * 1e-3) / scale, "unit": out["unit"],
                          "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(eh["h2d"]),
                          "d2h_bytes_per_step": int(eh["d2h"]),
                          "api": f"attn_fwd_host: {eh['stages']} stages pipelined over a "
                                 "compute stream and two copy streams",
                          "serial": serial}
        else:
            e2e_ms = serial["ms_per_step"]
            out["e2e"] = {"value": work * ws / (e2e_ms * 1e-3) / scale, "unit": out["unit"],
                          "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(e["h2d"]),
                          "d2h_bytes_per_step": int(e["d2h"]),
                          "api": "torch copies in, device-pointer library calls, copies out",
                          "breakdown_ms": serial["breakdown_ms"], "copy_gbs": serial["copy_gbs"]}
    del c
    torch.cuda.empty_cache()
    return out


def add_cpu_baseline(block, args, wid, rank, backward=False):
    """The float64 oracle timed on the host cores for one block (rank 0).
    Run after every GPU measurement of the line, so that no GPU timing
    follows a long idle spell of the device."""
    if rank == 0 and not args.no_cpu_baseline:
        fn = cpu_baseline_bwd if backward else cpu_baseline
        v, unit, cores, sample = fn(wid, budget_s=args.cpu_budget)
        block["cpu_baseline"] = {"value": v, "unit": unit, "cores": cores, "kind": "oracle",
                                 "sample": sample}


def bench_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    from exact_tiled_attention_49_b300 import build
    if rank == 0 or ws == 1:
        build.build()
    barrier(ws)
    import exact_tiled_attention_49_b300 as E
    E.load()
    peaks = load_peaks()
    if (args.backward or args.fp8) and workloads_kind(args.workload) != "prefill":
        raise SystemExit("--backward and --fp8 need a prefill workload (2, 3 or 5)")
    if args.backward and args.fp8:
        raise SystemExit("--backward and --fp8 are separate modes")

    head = measure_block(E, args, args.workload, device, peaks, ws, rank,
                         backward=args.backward, fp8=args.fp8, batch=args.batch)
    out = {
        "metric": METRIC,
        "value": head.pop("value"), "unit": head.pop("unit"),
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head.pop("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head.pop("dtype"), "data": "synthetic",
    }
    out.update(head)
    plain = not args.backward and not args.fp8 and args.batch is None
    skip = {args.workload}
    if plain and workloads_kind(args.workload) == "prefill" and not args.no_decode_block:
        # the metric's other half: the GQA decode step, with its own block
        out["decode"] = measure_block(E, args, 4, device, peaks, ws, rank)
        skip.add(4)
    if not args.no_other_workloads and args.batch is None:
        out["other_workloads"] = other_workloads(E, skip, device, max(3, min(args.steps, 10)),
                                                 peaks)
    add_cpu_baseline(out, args, args.workload, rank, backward=args.backward)
    if "decode" in out:
        add_cpu_baseline(out["decode"], args, 4, rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import workloads
    w = workloads.WORKLOADS[args.workload]
    per_step = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(args.workload, budget_s=per_step / 4)
    vals, samples, cores, unit = [], [], None, None
    t0 = time.perf_counter()
    for s in range(args.steps):
        v, unit, cores, sample = cpu_baseline(args.workload, budget_s=per_step, seed=s + 1)
        vals.append(v)
        samples.append(sample)
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": dict({"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                           "parallelism": "host cores"},
                          **({"T": w.T, "S": w.S, "causal": w.causal} if w.kind == "prefill"
                             else {"cache_len": f"U[{w.lens[0]},{w.lens[1]}]"})),
           "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                            "sample": samples[0] + f" (per step; {args.steps} steps)"},
           "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=3, choices=[2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (dQ, dK, dV) of the prefill workload instead")
    ap.add_argument("--fp8", action="store_true",
                    help="time the prefill workload on E4M3 inputs (attn_fwd_fp8) instead")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip timing the other benchmark workloads")
    ap.add_argument("--no-decode-block", action="store_true",
                    help="skip the decode block that follows a prefill headline")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end (host buffer) measurement")
    ap.add_argument("--batch", type=int, default=None,
                    help="smaller batch of the same workload (ncu profiling cases only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
