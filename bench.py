#!/usr/bin/env python
"""Benchmark of the selective scan's hot path on B300; prints one JSON line (rank 0).

One step = the whole path on one batch of synthetic input: ssm_scan_fwd over the long-sequence
workload (batch 1, L 131072, D 1536, N 16, fp32, exact ZOH; 2.43 GB of compulsory traffic, far larger
than L2), then one ssm_scan_step continuing from its final state (the prefill -> decode hand-off).
Units per step: batch * (L + 1) * D scan elements. The other prefill workloads (the Mamba-130M and
Mamba-1.4B layers), the fused layer, the backward pass, the SSD layer and the decode workload are timed
after it and reported under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Timing: W untimed steps, then K timed steps bracketed by a barrier and a device synchronise; L2 is
flushed (a 512 MiB write, then a read of the same buffer, so that no dirty line of the flush is left to
write back) before every step, outside the CUDA-event pairs that time the step's kernels on the launching
stream; the job time is the maximum over ranks. Multi-GPU runs (torchrun) are weak
scaling: every rank scans its own independent batch on its own GPU, with no data-path collective.

--impl reference times the CPU oracle (double precision, OpenMP over channels, as it stands) on the
host cores: each step is a bounded sample (whole sequences of a subset of the workload's channels).
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
sys.path.insert(0, ROOT)

import ssm_inputs  # noqa: E402

METRIC = "selective-scan B·L·D elems/s; achieved HBM GB/s as fraction of B300 peak"
FALLBACK_HBM_GBS = 6400.0
FLUSH_BYTES = 512 << 20
FWD_SOURCES = ("scan_fwd_tma.cu", "common.cuh")  # the prefill kernel's device code (host declarations excluded)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long",
                    choices=sorted(k for k in ssm_inputs.WORKLOADS if k != "decode"))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=None,
                    help="CPU oracle seconds per sample (default: 5 for the GPU arm's baseline, "
                         "120 / (steps + warmup) for --impl reference)")
    ap.add_argument("--oracle-threads", type=int, default=None,
                    help="threads of the CPU oracle in --impl reference (default: every host core)")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=VALUE",
                    help="override a size of the workload (batch, L or D), e.g. for a small profiling case")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (reported under 'workloads')")
    ap.add_argument("--profile", action="store_true",
                    help="a lean run for profilers: no L2-flush buffers, no end-to-end leg, no CPU baseline, other "
                         "workloads only if --extra names them (its timings are not benchmark values)")
    ap.add_argument("--extra", default="all", metavar="KIND[,KIND]",
                    help="which other workloads to time: all, or any of prefill, fused, bwd, ssd, decode")
    return ap.parse_args(argv)


def describe(name, cfg):
    return (f"{name}: batch {cfg['batch']}, L {cfg['L']}, D {cfg['D']}, N {cfg['N']}, {cfg['dtype']}, "
            f"{cfg['disc']}; delta = softplus(N({cfg['mu']}, {cfg['sigma']})), A_log = log(1..N); "
            f"+ 1 decode step from the final state")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s (burst) from MEASURED_PEAKS.json, else None."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return None


def fwd_bytes(cfg):
    """Compulsory bytes of one prefill launch: x, delta, B, C, A_log read; y, final state written."""
    es = 2 if cfg["dtype"] == "bf16" else 4
    b, L, D, N = cfg["batch"], cfg["L"], cfg["D"], cfg["N"]
    return 3 * b * L * D * es + 2 * b * L * N * es + D * N * 4 + b * D * N * 4


def bwd_bytes(cfg):
    """Compulsory bytes of one backward launch: x, delta, dy, B, C, A_log read; dx, ddelta (input dtype) and
    dA_log, dB, dC, dh0 (fp32) written. The recomputed states and the workspace's chunk-end states are not
    counted."""
    es = 2 if cfg["dtype"] == "bf16" else 4
    b, L, D, N = cfg["batch"], cfg["L"], cfg["D"], cfg["N"]
    return 5 * b * L * D * es + 2 * b * L * N * es + 2 * b * L * N * 4 + 2 * D * N * 4 + b * D * N * 4


def flush_l2(buf):
    """Evict the L2 before a timed launch: write a buffer larger than the L2 (126 MB), then read it back. The
    read leaves only clean lines in the L2, so the timed kernels do not also pay for writing the flush's own
    data back to DRAM (about 100 MB of dirty lines after the write alone)."""
    buf.zero_()
    buf.sum()


def step_bytes(cfg):
    """Compulsory bytes of one decode step: state read + written, x_t, delta_t, y_t, B_t, C_t, A_log."""
    es = 2 if cfg["dtype"] == "bf16" else 4
    b, D, N = cfg["batch"], cfg["D"], cfg["N"]
    return 2 * b * D * N * 4 + 3 * b * D * es + 2 * b * N * es + D * N * 4


def ncu_traffic(kernel_prefix, workload):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    from selective_state_space_124_b300 import build as lib_build
    entry = rec.get(workload, {})
    if entry.get("source_hash") != lib_build.source_hash(FWD_SOURCES) or not entry.get("kernel", "").startswith(kernel_prefix):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples the SM clock and clock-event reasons during the timed region (reads only): NVML when the
    Python bindings are importable, else `nvidia-smi --query-gpu ... -lms 20` as a subprocess."""

    NVML_NAMES = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                  0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                  0x2: "applications_clocks_setting"}
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.sw_power_cap",
                  "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                  "clocks_event_reasons.sw_thermal_slowdown"]

    def __init__(self, local_rank):
        self.local = local_rank
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.mode, self.error = None, None
        self._stop = threading.Event()
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = self._nvml_handle(pynvml, local_rank)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:  # noqa: BLE001 -- fall back to nvidia-smi
            self.error = f"nvml: {type(e).__name__}: {e}"
            self.mode = "smi"

    @staticmethod
    def _nvml_handle(nv, local_rank):
        try:
            import torch
            pr = torch.cuda.get_device_properties(local_rank)
            return nv.nvmlDeviceGetHandleByPciBusId(
                f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0")
        except Exception:  # noqa: BLE001
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            entry = vis.split(",")[local_rank].strip()
            if entry.startswith(("GPU-", "MIG-")):
                return nv.nvmlDeviceGetHandleByUUID(entry)
            return nv.nvmlDeviceGetHandleByIndex(int(entry))
        return nv.nvmlDeviceGetHandleByIndex(local_rank)

    def _smi_id(self):
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.local)
            return f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        except Exception:  # noqa: BLE001
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            return vis.split(",")[self.local].strip() if vis else str(self.local)

    def _run_nvml(self):
        nv = self.nv
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                bits = int(get_r(self.h))
                self.reasons |= {n for b, n in self.NVML_NAMES.items() if bits & b}
            except Exception:  # noqa: BLE001
                pass
            time.sleep(0.002)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", self._smi_id(), "--query-gpu=" + ",".join(self.SMI_FIELDS),
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.3)
            except Exception as e:  # noqa: BLE001
                self.proc = None
                self.error = (self.error or "") + f"; smi: {type(e).__name__}: {e}"
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self.t.join()
            return
        if getattr(self, "proc", None) is None:
            return
        time.sleep(0.05)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        names = ["sw_power_cap", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
        for line in out.splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) != len(self.SMI_FIELDS):
                continue
            try:
                self.samples.append(float(f[0]))
                self.max_mhz = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[2:]):
                if v.lower() == "active":
                    self.reasons.add(n)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0,
                    "error": self.error}
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.mode}


def _dev_tensor(torch, a, bf16):
    if bf16:
        return torch.from_numpy(ssm_inputs.bf16_round(a).view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def measure_prefill(name, reps, flush, peak, fused=False):
    """Prefill of another workload, timed like the main one (L2 flushed before each launch, CUDA events).
    fused: the layer pieces around the scan as well -- delta = softplus(delta_raw + bias), y = (C h + D x) *
    SiLU(z) -- with raw delta ~ N(mu, sigma) (the workload's law before its softplus), bias ~ U(-0.5, 0.5),
    D ~ N(0, 1), z ~ N(0, 1); the gate input z adds one [batch, L, D] read."""
    import ctypes
    import torch
    import selective_state_space_124_b300 as lib
    from selective_state_space_124_b300 import _ffi
    cfg = dict(ssm_inputs.WORKLOADS[name])
    inp = ssm_inputs.workload_inputs(name)
    bf16 = cfg["dtype"] == "bf16"
    b, L, D, N = cfg["batch"], cfg["L"], cfg["D"], cfg["N"]
    if fused:
        rng = np.random.default_rng(99)
        inp["delta"] = rng.normal(cfg["mu"], cfg["sigma"], (b, L, D)).astype(np.float32)
        inp["z"] = rng.standard_normal((b, L, D)).astype(np.float32)
    d = {k: _dev_tensor(torch, inp[k], bf16) for k in ("x", "delta", "B", "C") + (("z",) if fused else ())}
    A = torch.from_numpy(inp["A_log"].copy()).cuda()
    y = torch.empty((b, L, D), dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")
    fs = torch.empty((b, D, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    if fused:
        bias = torch.from_numpy(np.random.default_rng(98).uniform(-0.5, 0.5, D).astype(np.float32)).cuda()
        dsk = torch.from_numpy(np.random.default_rng(97).standard_normal(D).astype(np.float32)).cuda()
        v = ctypes.c_void_p
        fn = _ffi.load().ssm_scan_fwd_ex
        cargs = (v(d["x"].data_ptr()), v(d["delta"].data_ptr()), v(A.data_ptr()), v(d["B"].data_ptr()),
                 v(d["C"].data_ptr()), None, v(bias.data_ptr()), 1, v(dsk.data_ptr()), v(d["z"].data_ptr()),
                 v(y.data_ptr()), v(fs.data_ptr()), b, L, D, N, _ffi.DTYPE[cfg["dtype"]], _ffi.DISC[cfg["disc"]],
                 v(stream.cuda_stream))
        launch = lambda: _ffi.check("ssm_scan_fwd_ex", fn(*cargs))
    else:
        args = (d["x"].data_ptr(), d["delta"].data_ptr(), A.data_ptr(), d["B"].data_ptr(), d["C"].data_ptr(), 0,
                y.data_ptr(), fs.data_ptr(), b, L, D, N, cfg["dtype"], cfg["disc"], stream.cuda_stream)
        launch = lambda: lib.ssm_scan_fwd_ptr(*args)
    ms = []
    for i in range(3 + reps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ms.append(e0.elapsed_time(e1))
    lib.check_device()
    med = statistics.median(ms) / 1e3
    es = 2 if bf16 else 4
    nbytes = fwd_bytes(cfg) + ((b * L * D * es + 2 * D * 4) if fused else 0)  # + z, bias, D
    gbs = nbytes / med / 1e9
    what = describe(name, cfg).split(";")[0] + ("; fused softplus(delta + bias), + D x, * SiLU(z)" if fused else "")
    out = {"workload": what, "launch_ms_median": med * 1e3, "elems_per_s": b * L * D / med, "gbs": gbs,
           "hbm_frac": gbs / peak, "bytes_per_launch": nbytes, "reps": reps,
           "traffic": None if fused else ncu_traffic("scan_fwd", name)}
    if nbytes < (1 << 20):  # the tiny scan moves kilobytes: its time is launch latency, not a roofline figure
        out["bound"] = "launch latency (no roofline gate)"
    return out


def measure_backward(name, reps, flush, peak):
    """Backward pass of a prefill workload (ssm_scan_bwd through the C ABI, dy ~ N(0, 1), no initial state,
    no final-state gradient), timed like the prefill: L2 flushed before each launch, CUDA events."""
    import ctypes
    import torch
    import selective_state_space_124_b300 as lib
    from selective_state_space_124_b300 import _ffi
    cfg = dict(ssm_inputs.WORKLOADS[name])
    inp = ssm_inputs.workload_inputs(name)
    bf16 = cfg["dtype"] == "bf16"
    b, L, D, N = cfg["batch"], cfg["L"], cfg["D"], cfg["N"]
    inp["dy"] = np.random.default_rng(5).standard_normal((b, L, D)).astype(np.float32)
    d = {k: _dev_tensor(torch, inp[k], bf16) for k in ("x", "delta", "B", "C", "dy")}
    A = torch.from_numpy(inp["A_log"].copy()).cuda()
    tdt = torch.bfloat16 if bf16 else torch.float32
    out = [torch.empty((b, L, D), dtype=tdt, device="cuda"), torch.empty((b, L, D), dtype=tdt, device="cuda"),
           torch.empty((D, N), device="cuda"), torch.empty((b, L, N), device="cuda"),
           torch.empty((b, L, N), device="cuda"), torch.empty((b, D, N), device="cuda")]
    need = lib.bwd_workspace_size(b, L, D, N)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    v = ctypes.c_void_p
    fn = _ffi.load().ssm_scan_bwd
    cargs = (v(d["x"].data_ptr()), v(d["delta"].data_ptr()), v(A.data_ptr()), v(d["B"].data_ptr()),
             v(d["C"].data_ptr()), None, v(d["dy"].data_ptr()), None, *(v(t.data_ptr()) for t in out),
             v(ws.data_ptr()), ws.numel(), b, L, D, N, _ffi.DTYPE[cfg["dtype"]], _ffi.DISC[cfg["disc"]],
             v(stream.cuda_stream))
    ms = []
    for i in range(3 + reps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        _ffi.check("ssm_scan_bwd", fn(*cargs))
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ms.append(e0.elapsed_time(e1))
    lib.check_device()
    med = statistics.median(ms) / 1e3
    nbytes = bwd_bytes(cfg)
    gbs = nbytes / med / 1e9
    return {"workload": describe(name, cfg).split(";")[0] + "; backward (all input gradients)",
            "launch_ms_median": med * 1e3, "elems_per_s": b * L * D / med, "gbs": gbs, "hbm_frac": gbs / peak,
            "bytes_per_launch": nbytes, "workspace_bytes": need, "reps": reps}


def ssd_bytes(cfg):
    """Compulsory bytes of one SSD launch: x, B, C (bf16), delta (fp32), A_log read; y (bf16) and the final
    state (fp32) written."""
    b, L, H, P, N = cfg["batch"], cfg["L"], cfg["H"], cfg["P"], cfg["N"]
    return 2 * b * L * H * P * 2 + 2 * b * L * N * 2 + b * L * H * 4 + H * 4 + b * H * P * N * 4


def ssd_flops(cfg, Q=128):
    """Tensor-core work of the chunked algorithm per launch, full tiles (the causal half of the masked product is
    counted whole, as a dense evaluation does it): per (batch element, chunk) C B^T once (2 Q^2 N; all heads share
    B and C); per (batch element, chunk, head) the masked product with x (2 Q^2 P), the inter-chunk read-out
    C S (2 Q N P) and the chunk's state contribution (B^T (w x), 2 Q N P)."""
    b, L, H, P, N = cfg["batch"], cfg["L"], cfg["H"], cfg["P"], cfg["N"]
    chunks = (L + Q - 1) // Q
    return b * chunks * (2 * Q * Q * N + H * (2 * Q * Q * P + 4 * Q * N * P))


def measure_ssd(name, reps, flush, peak):
    """The Mamba-2 SSD layer (ssm_ssd_fwd), timed like the prefill: L2 flushed before each launch, CUDA events.
    Reports the HBM fraction of the compulsory bytes and the tensor throughput of the chunked algorithm."""
    import torch
    import selective_state_space_124_b300 as lib
    cfg = dict(ssm_inputs.SSD_WORKLOADS[name])
    inp = ssm_inputs.make_ssd_inputs(**cfg)
    b, L, H, P, N = cfg["batch"], cfg["L"], cfg["H"], cfg["P"], cfg["N"]

    def bf(bits, shape):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(shape).cuda()
    x, B, C = bf(inp["x_bits"], (b, L, H, P)), bf(inp["B_bits"], (b, L, N)), bf(inp["C_bits"], (b, L, N))
    dt, A = torch.from_numpy(inp["delta"]).cuda(), torch.from_numpy(inp["A_log"]).cuda()
    y = torch.empty((b, L, H, P), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((b, H, P, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    need = lib.ssd_workspace_size(b, L, H, P, N)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    args = [t.data_ptr() for t in (x, dt, A, B, C)] + [0, y.data_ptr(), fs.data_ptr(), ws.data_ptr()]
    from selective_state_space_124_b300 import _ffi
    fn = _ffi.load().ssm_ssd_fwd
    import ctypes
    cargs = [ctypes.c_void_p(a) if a else None for a in args] + [need, b, L, H, P, N, _ffi.DTYPE["bf16"],
                                                                 _ffi.DISC[cfg["disc"]], ctypes.c_void_p(stream.cuda_stream)]
    ms = []
    for i in range(3 + reps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        _ffi.check("ssm_ssd_fwd", fn(*cargs))
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            ms.append(e0.elapsed_time(e1))
    lib.check_device()
    med = statistics.median(ms) / 1e3
    nbytes, flops = ssd_bytes(cfg), ssd_flops(cfg)
    bf16_peak = measured_tensor_peak()
    return {"workload": f"{name}: Mamba-2 SSD layer, batch {b}, L {L}, {H} heads x {P}, N {N}, bf16, {cfg['disc']}, "
                        f"chunks of 128", "launch_ms_median": med * 1e3, "elems_per_s": b * L * H * P / med,
            "gbs": nbytes / med / 1e9, "hbm_frac": nbytes / med / 1e9 / peak, "bytes_per_launch": nbytes,
            "tflops": flops / med / 1e12, "tensor_frac": flops / med / 1e12 / bf16_peak if bf16_peak else None,
            "flops_per_launch": flops, "workspace_bytes": need, "reps": reps}


def measure_decode(steps, flush, peak):
    """The decode workload (batch 128, D 5120, N 16, fp32 state in HBM): `steps` consecutive ssm_scan_step
    calls over a fixed set of 16 device-resident tokens, (a) back to back as one CUDA graph (the 42 MB
    state stays L2-resident between steps) and (b) one step at a time with the L2 flushed before each."""
    import torch
    import selective_state_space_124_b300 as lib
    cfg = dict(ssm_inputs.WORKLOADS["decode"])
    ds = ssm_inputs.DecodeStream(**cfg)
    batch, D, N = cfg["batch"], cfg["D"], cfg["N"]
    toks = [ds.next_step() for _ in range(16)]
    dt = [{k: _dev_tensor(torch, t[k], False) for k in ("x", "delta", "B", "C")} for t in toks]
    A = torch.from_numpy(ds.A_log.copy()).cuda()
    state = torch.from_numpy(ds.state0.copy()).cuda()
    y = torch.empty((batch, D), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    def step_args(i, s):
        t = dt[i % 16]
        return (state.data_ptr(), t["x"].data_ptr(), t["delta"].data_ptr(), A.data_ptr(), t["B"].data_ptr(),
                t["C"].data_ptr(), y.data_ptr(), batch, D, N, "f32", cfg["disc"], s.cuda_stream)
    per_graph = 100
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(3):
            lib.ssm_scan_step_ptr(*step_args(i, side))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(per_graph):
                lib.ssm_scan_step_ptr(*step_args(i, side))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // per_graph)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    resident = e0.elapsed_time(e1) / 1e3 / (reps * per_graph)
    stream = torch.cuda.current_stream()
    ms = []
    for i in range(3 + 50):
        flush_l2(flush)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        lib.ssm_scan_step_ptr(*step_args(i, stream))
        a1.record(stream)
        if i >= 3:
            ms.append((a0, a1))
    torch.cuda.synchronize()
    lib.check_device()
    cold = statistics.median(a.elapsed_time(b_) for a, b_ in ms) / 1e3
    nb = step_bytes(cfg)
    return {"workload": f"decode: batch {batch}, D {D}, N {N}, fp32 state, {cfg['disc']}",
            "steps_timed": reps * per_graph, "us_per_step_l2_resident": resident * 1e6,
            "state_entries_per_s_l2_resident": batch * D * N / resident,
            "us_per_step_l2_flushed": cold * 1e6, "gbs_l2_flushed": nb / cold / 1e9,
            "hbm_frac_l2_flushed": nb / cold / 1e9 / peak, "bytes_per_step": nb}


def dist_setup():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank: int) -> int:
    """Each rank scans its own independent batch (weak scaling): same shapes and laws, seed = rank."""
    return rank


def job_seconds(local_seconds: float, world: int, device=None) -> float:
    """Job time = the slowest rank's time (max over ranks; the local value when running alone)."""
    if world <= 1:
        return local_seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput: the units every rank processed, over the job time."""
    return world * units_per_step * steps / seconds


def oracle_threads() -> int:
    """Threads the CPU oracle runs on: every host core this process may use."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def pin_oracle_threads(n=None) -> None:
    """Fix the oracle's OpenMP thread count (default: every host core) before its library (and so libgomp) is
    loaded, so that both bench arms time it on the same number of threads."""
    os.environ["OMP_NUM_THREADS"] = str(n if n else oracle_threads())


def oracle_sample(inp, cfg, budget_s):
    """Pick a channel subset whose whole sequences take about budget_s seconds in the oracle."""
    import oracle
    orc = oracle.default()
    total = cfg["batch"] * cfg["D"]
    n = min(total, max(16, 2 * orc.num_threads()))
    t0 = time.perf_counter()
    orc.scan_fwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], disc=cfg["disc"],
                 channels=list(range(n)))
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(min(total, max(1, n * budget_s / dt)))
    return list(np.linspace(0, total - 1, n).astype(np.int64))


def cpu_oracle_rate(inp, cfg, chans):
    """Time the oracle on whole sequences of the given channels; returns (elems/s, threads, sample)."""
    import oracle
    orc = oracle.default()
    L, total = cfg["L"], cfg["batch"] * cfg["D"]
    t0 = time.perf_counter()
    orc.scan_fwd(inp["x"], inp["delta"], inp["A_log"], inp["B"], inp["C"], disc=cfg["disc"], channels=chans)
    dt = time.perf_counter() - t0
    n = len(chans)
    return n * L / dt, orc.num_threads(), f"{n} of {total} channels, full L = {L} each ({n * L} elems)"


def workload_config(args, world):
    """Size overrides and the JSON `config` of a run; both arms report the same config."""
    overrides = {}
    for kv in args.set:
        k, v = kv.split("=", 1)
        if k not in ("batch", "L", "D"):
            raise SystemExit(f"--set: unknown size {k!r} (batch, L or D)")
        overrides[k] = int(v)
    cfg = dict(ssm_inputs.WORKLOADS[args.workload], **overrides)
    es = 2 if cfg["dtype"] == "bf16" else 4
    in_bytes = cfg["batch"] * cfg["L"] * (2 * cfg["D"] + 2 * cfg["N"]) * es
    config = {"workload": describe(args.workload, cfg),
              "l2": f"L2 flushed (512 MiB write, then read back) before every step; prefill inputs {in_bytes / 1e9:.3g} GB "
                    f"({'larger' if in_bytes > 126e6 else 'smaller'} than the 126 MB L2)",
              "parallelism": f"weak x{world}: one independent batch per GPU (seed = rank), no collective"}
    return overrides, cfg, config


def run_reference(args, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores, one bounded sample per step."""
    if rank != 0:
        return
    pin_oracle_threads(args.oracle_threads)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    overrides, cfg, config = workload_config(args, world)
    inp = ssm_inputs.workload_inputs(args.workload, **overrides)
    budget = args.cpu_seconds if args.cpu_seconds is not None else 120.0 / max(1, args.steps + args.warmup)
    chans = oracle_sample(inp, cfg, max(0.02, budget))
    rates, cores, sample = [], None, None
    for i in range(args.warmup + args.steps):
        r, cores, sample = cpu_oracle_rate(inp, cfg, chans)
        if i >= args.warmup:
            rates.append(r)
    value = float(statistics.median(rates))
    units = cfg["batch"] * (cfg["L"] + 1) * cfg["D"]
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elems/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": units / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": "elems/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: " + sample},
        "e2e": {"value": value, "unit": "elems/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def cpu_baseline_subprocess(args):
    """The oracle timed in a fresh process (no torch, no CUDA context, OpenMP pinned to the host cores),
    exactly as the reference arm times it: 1 untimed and 2 timed samples of the same workload. A second,
    shorter run on one thread gives the per-core rate."""
    def run(threads, seconds):
        cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", args.workload,
               "--steps", "2", "--warmup", "1", "--cpu-seconds", str(seconds), "--oracle-threads", str(threads)]
        for kv in args.set:
            cmd += ["--set", kv]
        env = {k: v for k, v in os.environ.items()
               if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "LOCAL_WORLD_SIZE", "GROUP_RANK", "ROLE_RANK",
                            "TORCHELASTIC_RUN_ID", "MASTER_ADDR", "MASTER_PORT")}
        env["OMP_NUM_THREADS"] = str(threads)
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900, check=True).stdout
        rec = json.loads(out.strip().splitlines()[-1])["cpu_baseline"]
        rec["sample"] = rec["sample"].replace("each step: ", "median of 2 timed samples, each ")
        return rec

    try:
        rec = run(oracle_threads(), args.cpu_seconds or 5.0)
    except (subprocess.SubprocessError, ValueError, KeyError, IndexError) as e:
        return {"value": None, "unit": "elems/s", "cores": None, "kind": "oracle",
                "sample": f"unavailable: {type(e).__name__}: {str(e)[:200]}"}
    rec["process"] = "separate process, OMP_NUM_THREADS = host cores (as the reference arm)"
    try:
        one = run(1, 1.0)
        rec["single_thread"] = {"value": one["value"], "unit": "elems/s", "cores": one["cores"],
                                "sample": one["sample"]}
    except (subprocess.SubprocessError, ValueError, KeyError, IndexError) as e:
        rec["single_thread"] = {"value": None, "sample": f"unavailable: {type(e).__name__}: {str(e)[:200]}"}
    return rec


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, rank)

    import torch
    import torch.distributed as dist

    import selective_state_space_124_b300 as lib

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))

    overrides, cfg, config = workload_config(args, world)
    inp = ssm_inputs.workload_inputs(args.workload, seed=rank_seed(rank), **overrides)
    tok = ssm_inputs.token_inputs(cfg["batch"], cfg["D"], cfg["N"], seed=1000 + rank_seed(rank),
                                  mu=cfg["mu"], sigma=cfg["sigma"])
    bf16 = cfg["dtype"] == "bf16"
    tdt = torch.bfloat16 if bf16 else torch.float32

    def host_tensor(a):
        if bf16:
            return torch.from_numpy(ssm_inputs.bf16_round(a).view(np.int16).copy()).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a, np.float32))

    hx = {k: host_tensor(inp[k]).pin_memory() for k in ("x", "delta", "B", "C")}
    hx["A_log"] = torch.from_numpy(inp["A_log"].copy()).pin_memory()
    ht = {k: host_tensor(tok[k]).pin_memory() for k in ("x", "delta", "B", "C")}
    dev = {k: v.cuda() for k, v in hx.items()}
    dtok = {k: v.cuda() for k, v in ht.items()}
    b, L, D, N = cfg["batch"], cfg["L"], cfg["D"], cfg["N"]
    y = torch.empty((b, L, D), dtype=tdt, device="cuda")
    state = torch.empty((b, D, N), dtype=torch.float32, device="cuda")
    y_t = torch.empty((b, D), dtype=tdt, device="cuda")
    if args.profile:  # other workloads only when --extra names them
        args.no_e2e = args.no_cpu_baseline = True
        args.no_extra = args.no_extra or args.extra == "all"
    flush = torch.empty(FLUSH_BYTES // 4 if not args.profile else 256, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    # The timed loop calls the C ABI on precomputed device addresses: launching costs a few microseconds of
    # host time, well under the L2 flush that precedes every step, so the host stays ahead of the device and
    # the event pairs measure kernel time only (the e2e leg below goes through the tensor-level binding).
    sh = stream.cuda_stream
    fwd_args = (dev["x"].data_ptr(), dev["delta"].data_ptr(), dev["A_log"].data_ptr(), dev["B"].data_ptr(),
                dev["C"].data_ptr(), 0, y.data_ptr(), state.data_ptr(), b, L, D, N, cfg["dtype"], cfg["disc"], sh)
    step_args = (state.data_ptr(), dtok["x"].data_ptr(), dtok["delta"].data_ptr(), dev["A_log"].data_ptr(),
                 dtok["B"].data_ptr(), dtok["C"].data_ptr(), y_t.data_ptr(), b, D, N, cfg["dtype"], cfg["disc"], sh)

    def fwd():
        lib.ssm_scan_fwd_ptr(*fwd_args)

    def step():
        lib.ssm_scan_step_ptr(*step_args)

    for _ in range(max(3, args.warmup)):
        flush_l2(flush)
        fwd()
        step()
    lib.check_device()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    head = torch.empty(4 * FLUSH_BYTES // 4 if not args.profile else 256, dtype=torch.float32, device="cuda")
    with sampler:
        wall0 = time.perf_counter()
        head.zero_()  # a long first write: the host enqueues ahead of the device from the start
        for i in range(K):
            flush_l2(flush)
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            step()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    lib.check_device()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    stp_ms = [e[1].elapsed_time(e[2]) for e in ev]
    total_s = job_seconds((sum(fwd_ms) + sum(stp_ms)) / 1e3, world, device="cuda")
    units_step = b * (L + 1) * D
    value = job_value(units_step, K, world, total_s)

    # ---- end to end through the public API: pinned host inputs in, results back to the host ------------
    # The prefill goes through ssm_scan_fwd_host (host arrays, streamed through the device in segments whose
    # uploads, scan and downloads overlap); the decode step then copies the final state and the token in,
    # steps on the device and copies y_t out.
    e2e = None
    if not args.no_e2e:
        hy = torch.empty((b, L, D), dtype=tdt).pin_memory()
        hs = torch.empty((b, D, N), dtype=torch.float32).pin_memory()
        hyt = torch.empty((b, D), dtype=tdt).pin_memory()
        seg = min(lib.HOST_SEGMENT_STEPS, L)
        hws = torch.empty(lib.host_workspace_size(b, D, N, cfg["dtype"], seg), dtype=torch.uint8, device="cuda")
        KE = max(3, min(K, 200))
        eve = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(KE)]
        h2d = sum(t.numel() * t.element_size() for t in list(hx.values()) + list(ht.values())) + \
            hs.numel() * hs.element_size()
        d2h = sum(t.numel() * t.element_size() for t in (hy, hs, hyt))
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(KE):
            flush_l2(flush)
            eve[i][0].record(stream)
            lib.ssm_scan_fwd_host(hx["x"], hx["delta"], hx["A_log"], hx["B"], hx["C"], disc=cfg["disc"], y=hy,
                                  final_state=hs, workspace=hws, stream=stream, seg_L=seg)
            state.copy_(hs, non_blocking=True)
            for k in ht:
                dtok[k].copy_(ht[k], non_blocking=True)
            step()
            hyt.copy_(y_t, non_blocking=True)
            eve[i][1].record(stream)
        torch.cuda.synchronize()
        lib.check_device()
        e2e_s = job_seconds(sum(e[0].elapsed_time(e[1]) for e in eve) / 1e3, world, device="cuda")
        e2e = {"value": job_value(units_step, KE, world, e2e_s), "unit": "elems/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": KE, "segment_steps": seg,
               "path": "ssm_scan_fwd_host (segments streamed from pinned host memory) + ssm_scan_step"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    fwd_avg_s = statistics.mean(fwd_ms) / 1e3
    achieved = fwd_bytes(cfg) / fwd_avg_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "elems/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_s / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg["dtype"], "data": "synthetic",
        "config": config,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": None if overrides else ncu_traffic("scan_fwd", args.workload),
                     "peak_kind": peak_kind, "kernel": "ssm_scan_fwd",
                     "algorithmic_bytes_per_launch": fwd_bytes(cfg), "avg_launch_ms": fwd_avg_s * 1e3},
        "fwd_ms_median": statistics.median(fwd_ms), "step_ms_median": statistics.median(stp_ms),
        "step_kernel_gbs": step_bytes(cfg) / (statistics.mean(stp_ms) / 1e3) / 1e9,
        "wall_s_timed_region": wall,
        "clocks": sampler.summary(),
        "e2e": e2e,
        "gpu_launches": 2 * K,
    }
    if not args.no_extra and world == 1:
        kinds = set(args.extra.split(",")) if args.extra != "all" else {"prefill", "fused", "bwd", "ssd", "decode"}
        extra = {}
        if "prefill" in kinds:
            for name in ("long", "mamba130m", "mamba1p4b", "tiny"):
                if name != args.workload:
                    extra[name] = measure_prefill(name, 20, flush, peak)
        if "fused" in kinds:  # the layer pieces on the Mamba-130M (fp32) and Mamba-1.4B (bf16) layers
            extra["mamba130m_fused"] = measure_prefill("mamba130m", 20, flush, peak, fused=True)
            extra["mamba1p4b_fused"] = measure_prefill("mamba1p4b", 20, flush, peak, fused=True)
        if "bwd" in kinds:
            extra["mamba130m_bwd"] = measure_backward("mamba130m", 20, flush, peak)
        if "ssd" in kinds:
            extra["mamba2_130m_ssd"] = measure_ssd("mamba2_130m", 20, flush, peak)
            extra["mamba2_2p7b_ssd"] = measure_ssd("mamba2_2p7b", 20, flush, peak)
        if "decode" in kinds:
            extra["decode"] = measure_decode(1000, flush, peak)
        line["workloads"] = extra
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline is timed at N = 1 only
        line["cpu_baseline"] = cpu_baseline_subprocess(args)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
