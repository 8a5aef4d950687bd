#!/usr/bin/env python3
"""Benchmark of the fused GEMM + bias + activation / chained-MLP hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras] [--no-cpu-baseline]

One step = one call of the library's C ABI over one batch of synthetic input
(the headline workload is the bf16 FFN up-projection X[16384,4096] @
W[4096,16384] + bias, GELU_erf).  Before every timed step a 512 MiB buffer is
written to flush the 129 MB L2 (the inputs are larger than L2 as well); each
step is bracketed by CUDA events on the launching stream; the line reports the
mean (and median) per-step kernel time.  Under torchrun (N > 1) every rank
runs its own replica on its own GPU (the path needs no exchange between
GPUs); rank 0 prints one JSON line with the max time over ranks.

``e2e`` is the same metric through the C ABI with pinned host buffers: the
inputs' host-to-device copies, the calls and the output's device-to-host copy
are all inside the timed region, pipelined over row chunks on separate copy
streams the way a user with host data would call the library.

``sustained`` runs the headline back to back for about three seconds (its own
clock record; the GPU reaches its power cap) and reports that rate against
the measured sustained bf16 peak, beside the per-step burst ``value``.  The
FP32 roofline is taken against the FMA rate measured in the same run by the
library's FMA-chain kernel (coalesce_measure_ffma).

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (rank 0 only) and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import hashlib
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

HEADLINE = "bf16_ffn_up_bias_gelu_16384x16384x4096"
METRIC = "fused GEMM+bias+GELU TFLOP/s and % of roofline; fused MLP rows/s and HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# workload's kernel at full size (for the training step, the sum over its two
# kernels, per step), from one single-pass ncu capture of this script's own
# full-size run of that workload (`ncu --metrics dram__bytes_read.sum,
# dram__bytes_write.sum --clock-control none -k regex:<kernel> -c 1`), with
# the fingerprint of the kernel sources it was taken on: first 16 hex digits
# of SHA-256 over the listed files, concatenated.  Reported only while those
# sources are unchanged.
CSRC = os.path.join(ROOT, "gemm_bias_activation_gb300", "csrc")
MEASURED_TRAFFIC = {
    "bf16_ffn_up_bias_gelu_16384x16384x4096":
        (('gemm_tc.cu', 'gemm_tc_pair.cu', 'gemm_tc.cuh', 'sm100_ptx.cuh', 'sm100_pair.cuh', 'epilogue.cuh'), "4697657c3bd78e44", 1385149952),
    "fp32_gemm_bias_gelu_4096":
        (('gemm_f32.cu', 'epilogue.cuh'), "c290b2b51d80ea8f", 302168832),
    "fp16_mlp3_softplus_128w_2p20rows":
        (('mlp_fused.cu', 'sm100_ptx.cuh', 'epilogue.cuh'), "677194fcde93effa", 486226944),
    "fp16_mlp5_softplus_64w_2p22rows":
        (('mlp_fused.cu', 'sm100_ptx.cuh', 'epilogue.cuh'), "677194fcde93effa", 1019516160),
    "fp16_mlp3_softplus_128w_2p20rows_train":
        (('mlp_fused.cu', 'mlp_backward.cu', 'mlp_train.cu', 'sm100_ptx.cuh', 'epilogue.cuh'), "091958fda30b68eb", 2333971456),
}


def measured_traffic(case):
    """The stored per-launch DRAM traffic of this case's kernel, or None if the
    case is not the full-size workload or the kernel changed since the capture."""
    from gemm_bias_activation_gb300 import inputs

    ent = MEASURED_TRAFFIC.get(case.w.name)
    if ent is None or case.w != inputs.WORKLOADS.get(case.w.name):
        return None
    files, fp, nbytes = ent
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest()[:16] == fp else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    except Exception:
        return dict(FALLBACK_PEAKS)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons, sampled every 20 ms
    during the timed region through NVML (read-only queries), or through
    nvidia-smi if NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.index = cuda_index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            try:
                self.index = int(vis.split(",")[cuda_index])
            except (ValueError, IndexError):
                pass
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        self.proc = None

    def _nvml_init(self):
        import ctypes

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex failed")
        self.nvml, self.handle = lib, h

    def _poll(self):
        import ctypes

        lib, h = self.nvml, self.handle
        mhz, mx, mw, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0   # NVML_CLOCK_SM
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
            get_reasons(h, ctypes.byref(reasons))
            if ok:
                self.samples.append((float(mhz.value), float(mx.value), mw.value / 1000.0, int(reasons.value)))
            self.stop_flag.wait(0.02)

    def start(self):
        try:
            self._nvml_init()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        except Exception:
            self.nvml = None
        try:
            fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.sw_power_cap,"
                      "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={fields}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read_smi(self):
        bits = [0x4, 0x8, 0x20, 0x40]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                r = sum(b for b, v in zip(bits, parts[3:7]) if v.lower() == "active")
                self.samples.append((float(parts[0]), float(parts[1]), float(parts[2]), r))
            except (ValueError, IndexError):
                continue

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": "none"}
        reasons = set()
        for smp in self.samples:
            for bit, name in self.REASONS.items():
                if smp[3] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples),
                "power_w_max": max(s[2] for s in self.samples), "samples": len(self.samples),
                "reasons": sorted(reasons), "source": "nvml" if self.nvml is not None else "nvidia-smi"}


# ----------------------------------------------------------------------------- workloads
class GemmCase:
    def __init__(self, w, dev):
        import torch

        from gemm_bias_activation_gb300 import inputs

        self.w = w
        A, B, bias = inputs.gemm_inputs(w, seed=0)
        self.host = (A.pin_memory(), B.pin_memory(), bias.pin_memory())
        self.A, self.B, self.bias = (t.to(dev) for t in self.host)
        self.Y = torch.empty((w.M, w.N), dtype=A.dtype, device=dev)
        self.Y_host = torch.empty((w.M, w.N), dtype=A.dtype).pin_memory()
        self.units = w.flops() / 1e12  # TFLOP per step
        self.unit = "TFLOP/s"
        self.h2d = sum(t.numel() * t.element_size() for t in self.host)
        self.d2h = self.Y.numel() * self.Y.element_size()
        self.launches_per_step = 1

    def config(self):
        return {"workload": self.w.name, "M": self.w.M, "N": self.w.N, "K": self.w.K, "act": self.w.act}

    def run(self, stream):
        import gemm_bias_activation_gb300 as g

        st = g.coalesce_gemm_bias_act(self.w.M, self.w.N, self.w.K, g._dtype_code(self.A), self.A.data_ptr(),
                                      self.B.data_ptr(), self.bias.data_ptr(), self.Y.data_ptr(),
                                      g.ACT_CODES[self.w.act], stream.cuda_stream)
        if st != 0:
            raise g.CoalesceError(st, "coalesce_gemm_bias_act")

    def run_unfused(self, stream):
        """The unfused sequence of the fusion study: GEMM without bias or
        activation, then the separate in-place bias + activation pass."""
        import gemm_bias_activation_gb300 as g

        w = self.w
        st = g.coalesce_gemm_bias_act(w.M, w.N, w.K, g._dtype_code(self.A), self.A.data_ptr(), self.B.data_ptr(),
                                      None, self.Y.data_ptr(), g.COALESCE_ACT_NONE, stream.cuda_stream)
        if st == 0:
            st = g.coalesce_bias_act(w.M, w.N, g._dtype_code(self.Y), self.Y.data_ptr(), self.bias.data_ptr(),
                                     g.ACT_CODES[w.act], stream.cuda_stream)
        if st != 0:
            raise g.CoalesceError(st, "unfused sequence")

    def run_bias_act_only(self, stream):
        import gemm_bias_activation_gb300 as g

        w = self.w
        st = g.coalesce_bias_act(w.M, w.N, g._dtype_code(self.Y), self.Y.data_ptr(), self.bias.data_ptr(),
                                 g.ACT_CODES[w.act], stream.cuda_stream)
        if st != 0:
            raise g.CoalesceError(st, "coalesce_bias_act")

    def run_e2e(self, stream, chunks=8):
        """Host buffers in, host buffer out, through the C ABI: B and bias are
        copied once, then A and Y move in row chunks on their own copy streams
        so that the H2D copy of chunk i+1, the GEMM on chunk i and the D2H copy
        of chunk i-1 overlap.  The chunks' GEMMs alternate between `stream`
        and a second compute stream, so that a chunk's last partial wave of
        tiles shares the SMs with the next chunk's first.  Everything between
        the first copy and the last copy is inside the caller's events on
        `stream`."""
        import torch

        import gemm_bias_activation_gb300 as g

        w = self.w
        if not hasattr(self, "_pipe"):
            self._pipe = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream(),
                          [torch.cuda.Event() for _ in range(2 * chunks + 2)])
        s_in, s_out, s_c, ev = self._pipe
        compute = (stream, s_c)
        while w.M % chunks:
            chunks //= 2
        R = w.M // chunks
        ev[0].record(stream)
        s_in.wait_event(ev[0])
        with torch.cuda.stream(s_in):
            self.B.copy_(self.host[1], non_blocking=True)
            self.bias.copy_(self.host[2], non_blocking=True)
        esz = self.A.element_size()
        for c in range(chunks):
            rows = slice(c * R, (c + 1) * R)
            with torch.cuda.stream(s_in):
                self.A[rows].copy_(self.host[0][rows], non_blocking=True)
                ev[1 + c].record(s_in)
            cs = compute[c % 2]
            cs.wait_event(ev[1 + c])
            st = g.coalesce_gemm_bias_act(R, w.N, w.K, g._dtype_code(self.A), self.A.data_ptr() + c * R * w.K * esz,
                                          self.B.data_ptr(), self.bias.data_ptr(),
                                          self.Y.data_ptr() + c * R * w.N * esz, g.ACT_CODES[w.act], cs.cuda_stream)
            if st != 0:
                raise g.CoalesceError(st, "coalesce_gemm_bias_act")
            ev[1 + chunks + c].record(cs)
            s_out.wait_event(ev[1 + chunks + c])
            with torch.cuda.stream(s_out):
                self.Y_host[rows].copy_(self.Y[rows], non_blocking=True)
        ev[2 * chunks + 1].record(s_out)
        stream.wait_event(ev[2 * chunks + 1])

    def roofline(self, sec, peaks):
        if self.w.dtype == "f32":
            ffma = peaks["ffma"]
            return {"bound": "alu", "achieved": self.w.flops() / sec / 1e12, "peak": ffma["tflops"],
                    "unit": "TFLOP/s", "peak_source": ffma["source"]}
        return {"bound": "tensor", "achieved": self.w.flops() / sec / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "peak_source": f"{peaks['source']} bf16 burst"}

    def cpu_sample(self, rows=64):
        """Oracle on a bounded sample of rows; returns (units of work done, seconds, description)."""
        import numpy as np

        import oracle

        rows = max(1, min(rows, self.w.M))
        A = self.host[0][:rows].float().numpy().astype(np.float64)
        B = self.host[1].float().numpy().astype(np.float64)
        bias = self.host[2].float().numpy().astype(np.float64)
        t0 = time.perf_counter()
        oracle.gemm_bias_act(A, B, bias, self.w.act)
        dt = time.perf_counter() - t0
        return 2.0 * rows * self.w.N * self.w.K / 1e12, dt, f"{rows} of {self.w.M} rows (all {self.w.N} columns)"


class MlpCase:
    def __init__(self, w, dev):
        import torch

        from gemm_bias_activation_gb300 import inputs

        self.w = w
        x, Ws, bs = inputs.mlp_inputs(w, seed=0)
        self.host_x = x.pin_memory()
        self.host_W = Ws
        self.host_b = bs
        self.x = self.host_x.to(dev)
        self.W = [t.to(dev) for t in Ws]
        self.b = [t.to(dev) for t in bs]
        self.out = torch.empty((w.rows, w.H), dtype=x.dtype, device=dev)
        self.out_host = torch.empty((w.rows, w.H), dtype=x.dtype).pin_memory()
        self.units = w.rows / 1e6  # million rows per step
        self.unit = "Mrows/s"
        self.h2d = self.host_x.numel() * self.host_x.element_size()
        self.d2h = self.out.numel() * self.out.element_size()
        self.launches_per_step = 1

    def config(self):
        w = self.w
        return {"workload": w.name, "rows": w.rows, "D": w.D, "H": w.H, "L": w.L, "act": w.act}

    def run(self, stream):
        import gemm_bias_activation_gb300 as g

        w = self.w
        st = g.coalesce_mlp_fused(w.rows, w.D, w.H, w.L, self.x.data_ptr(), [t.data_ptr() for t in self.W],
                                  [t.data_ptr() for t in self.b], self.out.data_ptr(), g.ACT_CODES[w.act],
                                  stream.cuda_stream)
        if st != 0:
            raise g.CoalesceError(st, "coalesce_mlp_fused")

    def run_e2e(self, stream, chunks=8):
        """Host x in, host out back, in row chunks overlapped as for the GEMM."""
        import torch

        import gemm_bias_activation_gb300 as g

        w = self.w
        if not hasattr(self, "_pipe"):
            self._pipe = (torch.cuda.Stream(), torch.cuda.Stream(),
                          [torch.cuda.Event() for _ in range(2 * chunks + 2)])
        s_in, s_out, ev = self._pipe
        while w.rows % chunks:
            chunks //= 2
        R = w.rows // chunks
        ev[0].record(stream)
        s_in.wait_event(ev[0])
        esz = self.x.element_size()
        for c in range(chunks):
            rows = slice(c * R, (c + 1) * R)
            with torch.cuda.stream(s_in):
                self.x[rows].copy_(self.host_x[rows], non_blocking=True)
                ev[1 + c].record(s_in)
            stream.wait_event(ev[1 + c])
            st = g.coalesce_mlp_fused(R, w.D, w.H, w.L, self.x.data_ptr() + c * R * w.D * esz,
                                      [t.data_ptr() for t in self.W], [t.data_ptr() for t in self.b],
                                      self.out.data_ptr() + c * R * w.H * esz, g.ACT_CODES[w.act], stream.cuda_stream)
            if st != 0:
                raise g.CoalesceError(st, "coalesce_mlp_fused")
            ev[1 + chunks + c].record(stream)
            s_out.wait_event(ev[1 + chunks + c])
            with torch.cuda.stream(s_out):
                self.out_host[rows].copy_(self.out[rows], non_blocking=True)
        ev[2 * chunks + 1].record(s_out)
        stream.wait_event(ev[2 * chunks + 1])

    def roofline(self, sec, peaks):
        return {"bound": "hbm", "achieved": self.w.bytes_moved() / sec / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_source": f"{peaks['source']} copy bandwidth",
                "tflops": self.w.flops() / sec / 1e12}

    def cpu_sample(self, rows=4096):
        import numpy as np

        import oracle

        rows = max(1, min(rows, self.w.rows))
        x = self.host_x[:rows].float().numpy().astype(np.float64)
        Ws = [t.float().numpy().astype(np.float64) for t in self.host_W]
        bs = [t.float().numpy().astype(np.float64) for t in self.host_b]
        t0 = time.perf_counter()
        oracle.mlp_chain(x, Ws, bs, self.w.act)
        dt = time.perf_counter() - t0
        return rows / 1e6, dt, f"{rows} of {self.w.rows} rows"


class MlpTrainCase:
    """One training step of the chained MLP through the C ABI: the forward
    pass that stores every activation, then the backward pass (dx, dW, db)
    for a fixed synthetic loss gradient dout."""

    def __init__(self, w, dev):
        import torch

        from gemm_bias_activation_gb300 import inputs

        self.w = w
        x, Ws, bs = inputs.mlp_inputs(w, seed=0)
        dout = inputs.normal((w.rows, w.out_width), 0, 99, w.dtype, 1.0)
        self.host_x, self.host_dout = x.pin_memory(), dout.pin_memory()
        self.host_W, self.host_b = Ws, bs
        self.x, self.dout = self.host_x.to(dev), self.host_dout.to(dev)
        self.W = [t.to(dev) for t in Ws]
        self.b = [t.to(dev) for t in bs]
        self.h = [torch.empty((w.rows, w.H), dtype=x.dtype, device=dev) for _ in range(w.L - 1)]
        self.out = torch.empty((w.rows, w.out_width), dtype=x.dtype, device=dev)
        self.dx = torch.empty_like(self.x)
        self.dW = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in Ws]
        self.db = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in bs]
        self.dW_host = [torch.empty(t.shape, dtype=torch.float32).pin_memory() for t in Ws]
        self.db_host = [torch.empty(t.shape, dtype=torch.float32).pin_memory() for t in bs]
        self.units = w.rows / 1e6
        self.unit = "Mrows/s"
        self.h2d = sum(t.numel() * t.element_size() for t in (self.host_x, self.host_dout))
        self.d2h = sum(t.numel() * 4 for t in self.dW_host + self.db_host)
        # Kernels per step (memsets are not kernels), by the library's rules,
        # on the widths rounded up to multiples of 64 as the fused kernels run
        # them: the forward is one fused launch when every width is at most
        # 256 (weights beyond 160 KiB are streamed), else one GEMM per layer;
        # the backward is one fused launch when every layer has K <= 128 and
        # N <= 256, the dW accumulators and one max(K)-column accumulator fit
        # the 512 TMEM columns and the weights and two row tiles fit in shared
        # memory, else a column sum and two GEMMs per layer.
        widths = [w.D] + [w.H] * (w.L - 1) + [w.out_width]
        fused = all(d <= 256 for d in widths)
        padded = [(d + 63) // 64 * 64 for d in widths]
        ks, ns = padded[:-1], padded[1:]
        wbytes = 2 * sum(a * b for a, b in zip(ks, ns))
        bwd_fused = (fused and all(k <= 128 and n <= 256 for k, n in zip(ks, ns))
                     and max(ks) + sum(ns) <= 512 and wbytes + 2 * 256 * max(padded) + 4096 <= 232448)
        self.launches_per_step = (1 if fused else w.L) + (1 if bwd_fused else 3 * w.L)

    def config(self):
        w = self.w
        return {"workload": w.name, "rows": w.rows, "D": w.D, "H": w.H, "L": w.L, "act": w.act,
                "step": "forward storing activations + backward (dx, dW, db)"}

    def run(self, stream):
        import gemm_bias_activation_gb300 as g

        w = self.w
        dt = g._dtype_code(self.x)
        st = g.coalesce_mlp_forward_train(w.rows, w.D, w.H, w.out_width, w.L, dt, self.x.data_ptr(),
                                          [t.data_ptr() for t in self.W], [t.data_ptr() for t in self.b],
                                          [t.data_ptr() for t in self.h], self.out.data_ptr(), g.ACT_CODES[w.act],
                                          stream.cuda_stream)
        if st == 0:
            st = g.coalesce_mlp_backward(w.rows, w.D, w.H, w.out_width, w.L, dt, self.x.data_ptr(),
                                         [t.data_ptr() for t in self.W], [t.data_ptr() for t in self.h],
                                         self.dout.data_ptr(), self.dx.data_ptr(), [t.data_ptr() for t in self.dW],
                                         [t.data_ptr() for t in self.db], g.ACT_CODES[w.act], stream.cuda_stream)
        if st != 0:
            raise g.CoalesceError(st, "MLP training step")

    def run_e2e(self, stream, chunks=8):
        """Host x and dout in, the parameter gradients back to host memory."""
        import torch

        with torch.cuda.stream(stream):
            self.x.copy_(self.host_x, non_blocking=True)
            self.dout.copy_(self.host_dout, non_blocking=True)
        self.run(stream)
        with torch.cuda.stream(stream):
            for d, h in zip(self.dW + self.db, self.dW_host + self.db_host):
                h.copy_(d, non_blocking=True)

    def roofline(self, sec, peaks):
        return {"bound": "hbm", "achieved": self.w.train_bytes_moved() / sec / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_source": f"{peaks['source']} copy bandwidth",
                "tflops": self.w.train_flops() / sec / 1e12}

    def cpu_sample(self, rows=2048):
        import numpy as np

        import oracle

        rows = max(1, min(rows, self.w.rows))
        x = self.host_x[:rows].float().numpy().astype(np.float64)
        dout = self.host_dout[:rows].float().numpy().astype(np.float64)
        Ws = [t.float().numpy().astype(np.float64) for t in self.host_W]
        bs = [t.float().numpy().astype(np.float64) for t in self.host_b]
        t0 = time.perf_counter()
        oracle.mlp_backward(x, Ws, bs, dout, self.w.act)
        dt = time.perf_counter() - t0
        return rows / 1e6, dt, f"{rows} of {self.w.rows} rows"


def inputs_dtype(name):
    from gemm_bias_activation_gb300 import inputs

    return inputs.WORKLOADS[name].dtype


def make_case(name, dev, M=None, N=None, K=None, rows=None):
    import dataclasses

    from gemm_bias_activation_gb300 import inputs

    w = inputs.WORKLOADS[name]
    if isinstance(w, inputs.GemmWorkload):
        w = dataclasses.replace(w, M=M or w.M, N=N or w.N, K=K or w.K)
        return GemmCase(w, dev)
    w = dataclasses.replace(w, rows=rows or w.rows)
    return MlpTrainCase(w, dev) if w.train else MlpCase(w, dev)


# ----------------------------------------------------------------------------- timing
def time_steps(case, steps, warmup, stream, flush, e2e=False, fn=None):
    import torch

    if fn is None:
        fn = case.run_e2e if e2e else case.run
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn(stream)
        stream.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for s, e in evs:
            flush.zero_()  # writes 512 MiB: evicts the 129 MB L2 before every timed step
            s.record(stream)
            fn(stream)
            e.record(stream)
        stream.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def small_m_study(dev, stream, rows_list=(64, 4096, 8192, 65536), calls=20, reps=20):
    """Launch-bound regime of the 128-wide 3-layer MLP: per-call device time
    from a CUDA graph of `calls` back-to-back C-ABI calls (no Python dispatch
    inside the timed region), at the row counts the megakernel pages report."""
    import torch

    import gemm_bias_activation_gb300 as g
    from gemm_bias_activation_gb300 import inputs

    w = inputs.WORKLOADS["fp16_mlp3_softplus_128w_2p20rows"]
    res = {}
    for rows in rows_list:
        x, Ws, bs = inputs.mlp_inputs(w, seed=0, rows=rows)
        x, Ws, bs = x.to(dev), [t.to(dev) for t in Ws], [t.to(dev) for t in bs]
        out = torch.empty((rows, w.H), dtype=x.dtype, device=dev)
        with torch.cuda.stream(stream):
            g.mlp_fused(x, Ws, bs, out=out, stream=stream)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(calls):
                    g.mlp_fused(x, Ws, bs, out=out)
            for _ in range(3):
                graph.replay()
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                stream.synchronize()
                ts.append(e0.elapsed_time(e1) / calls * 1e3)
        res[str(rows)] = {"us_per_call": statistics.median(ts)}
    return res


def fp32_sweep(dev, stream, flush, ffma_tflops, sizes=(256, 512, 1024, 2048, 4096), reps=100):
    """The FP32 square GEMM + bias + GELU sweep: median of `reps` device-timed
    calls at each size, the L2 flushed before each."""
    res = {}
    for n in sizes:
        c = make_case(f"fp32_gemm_bias_gelu_{n}", dev)
        ms = time_steps(c, reps, 3, stream, flush)
        med = statistics.median(ms)
        tf = c.units / (med / 1e3)
        res[str(n)] = {"ms_median": med, "tflops": tf, "frac_of_ffma_peak": tf / ffma_tflops}
        del c
    return res


def measure_ffma_peak(dev, stream, local, reps=5, iters=1 << 19):
    """The FP32 FMA rate of this GPU, measured: the library's FMA-chain kernel
    (coalesce_measure_ffma: 4 blocks x 256 threads per SM, 16 independent
    chains per thread, no memory traffic) timed with CUDA events on the
    launching stream, median of `reps` launches after one warm-up, with the
    SM clock sampled meanwhile.  The SM count is the device's own.  Also
    returned, for context: the derived figure, SMs x 128 FP32 lanes x 2 FLOP
    x the maximum SM clock."""
    import ctypes

    import torch

    import gemm_bias_activation_gb300 as g

    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    flop = ctypes.c_double(0.0)
    lib = g.load_library()

    def launch():
        st = lib.coalesce_measure_ffma(iters, ctypes.c_void_p(sink.data_ptr()), ctypes.byref(flop),
                                       ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise g.CoalesceError(st, "coalesce_measure_ffma")

    launch()
    stream.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        stream.synchronize()
        ts.append(e0.elapsed_time(e1))
    clk = clocks.stop()
    ms = statistics.median(ts)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = clk.get("sm_max_mhz") or 2070.0
    return {"tflops": flop.value / (ms / 1e3) / 1e12, "ms_median": ms, "flop_per_launch": flop.value,
            "source": f"measured: FMA-chain kernel on {sms} SMs (coalesce_measure_ffma)",
            "derived_tflops": sms * 128 * 2 * max_mhz * 1e6 / 1e12,
            "derived": f"{sms} SMs x 128 FP32 lanes x 2 FLOP x {max_mhz:.0f} MHz", "clocks": clk}


def sustained_leg(case, stream, local, seconds, peaks):
    """The workload back to back for about `seconds` (no flush between calls:
    its inputs are larger than L2 anyway), timed with one pair of CUDA events,
    the SM clock, power and throttle reasons sampled meanwhile.  This is the
    rate the GPU keeps up once it sits at its power cap, next to the per-step
    burst figure of the headline."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(3):
            case.run(stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        case.run(stream)
        e1.record(stream)
        stream.synchronize()
        calls = max(10, int(seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
        clocks = ClockSampler(local)
        clocks.start()
        e0.record(stream)
        for _ in range(calls):
            case.run(stream)
        e1.record(stream)
        stream.synchronize()
        clk = clocks.stop()
    ms = e0.elapsed_time(e1) / calls
    value = case.units / (ms / 1e3)
    out = {"value": value, "unit": case.unit, "ms_per_call": ms, "calls": calls, "seconds": ms * calls / 1e3,
           "clocks": clk}
    if clk.get("sm_mhz"):
        out["kcycles_per_call_at_median_clock"] = ms * clk["sm_mhz"]
    if isinstance(case, GemmCase) and case.w.dtype != "f32":
        out["peak"] = peaks["bf16_tflops_sustained"]
        out["peak_source"] = f"{peaks['source']} bf16 sustained"
        out["frac"] = value / out["peak"]
    return out


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    """The largest of every rank's x (a time), on every rank: the job takes as
    long as its slowest replica."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, max_ms, world):
    """Whole-job throughput of `world` replicas that each process
    `units_per_rank` per step (weak scaling), timed by the slowest rank."""
    return world * units_per_rank / (max_ms / 1e3)


def calibrated_cpu_sample(case, seconds):
    """Run the oracle on a row sample sized to take about `seconds` on this host."""
    probe = 64 if isinstance(case, GemmCase) else 8192
    units, dt, _ = case.cpu_sample(probe)
    rows = int(probe * max(1.0, seconds / max(dt, 1e-3)))
    return case.cpu_sample(rows)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- arms
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch  # noqa: F401

    from gemm_bias_activation_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    if isinstance(w, inputs.GemmWorkload):
        case = GemmCase.__new__(GemmCase)
        case.w = w
        case.host = inputs.gemm_inputs(w, seed=0)
        unit = "TFLOP/s"
        cfg = {"workload": args.workload, "M": w.M, "N": w.N, "K": w.K, "act": w.act}
    else:
        case = MlpCase.__new__(MlpCase)
        case.w = w
        case.host_x, case.host_W, case.host_b = inputs.mlp_inputs(w, seed=0)
        unit = "Mrows/s"
        cfg = {"workload": args.workload, "rows": w.rows, "D": w.D, "H": w.H, "L": w.L, "act": w.act}
    # each step: a row sample sized so that the whole run takes about two minutes
    probe = 64 if isinstance(case, GemmCase) else 8192
    _, dt0, _ = case.cpu_sample(probe)
    per_step = 120.0 / (args.warmup + args.steps)
    rows = max(1, int(probe * per_step / max(dt0, 1e-3)))
    times, work = [], 0.0
    sample = ""
    for i in range(args.warmup + args.steps):
        units, dt, sample = case.cpu_sample(rows)
        if i >= args.warmup:
            times.append(dt)
            work = units
    sec = statistics.mean(times)
    value = work / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": unit, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    import gemm_bias_activation_gb300 as g

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g.build()
    g.load_library()
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(max(1, args.flush_mb * 1024 * 1024 // 4), dtype=torch.float32, device=dev)

    case = make_case(args.workload, dev, args.M, args.N, args.K, args.rows)
    fp32_needed = case.w.dtype == "f32" or (not args.no_extras and world == 1 and (
        not args.no_fp32_sweep or any(inputs_dtype(n) == "f32" for n in args.extras)))
    if fp32_needed:
        peaks["ffma"] = measure_ffma_peak(dev, stream, local)

    # headline: device-resident inputs
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t_wall0 = time.perf_counter()
    ms = time_steps(case, args.steps, args.warmup, stream, flush)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    barrier(world)
    st = g.coalesce_device_status(stream.cuda_stream)
    if st != 0:
        raise g.CoalesceError(st, "device status after timed region")
    mean_ms = max_over_ranks(statistics.mean(ms), world)
    med_ms = max_over_ranks(statistics.median(ms), world)
    value = job_throughput(case.units, mean_ms, world)

    # end to end through the public API with host buffers
    if args.no_e2e:
        e2e_ms = float("nan")
        e2e_value = None
    else:
        ms_e2e = time_steps(case, max(3, min(20, args.steps)), 1, stream, flush, e2e=True)
        e2e_ms = max_over_ranks(statistics.mean(ms_e2e), world)
        e2e_value = job_throughput(case.units, e2e_ms, world)

    fusion = None
    if isinstance(case, GemmCase) and not args.no_fusion_study:
        ms_unf = time_steps(case, max(5, min(50, args.steps)), 3, stream, flush, fn=case.run_unfused)
        ms_ba = time_steps(case, max(5, min(50, args.steps)), 3, stream, flush, fn=case.run_bias_act_only)
        fusion = {"fused_ms": statistics.median(ms), "unfused_ms": statistics.median(ms_unf),
                  "bias_act_pass_ms": statistics.median(ms_ba),
                  "speedup": statistics.median(ms_unf) / statistics.median(ms),
                  "unfused": "GEMM (bias=NULL, act=NONE) then coalesce_bias_act in place"}

    sustained = None
    if args.sustained_s > 0:
        barrier(world)
        sustained = sustained_leg(case, stream, local, args.sustained_s, peaks)

    roof = case.roofline(mean_ms / 1e3, peaks)
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(case)

    line = {
        "metric": METRIC, "value": value, "unit": case.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "ms_per_step_median": med_ms,
        "ms_per_step_p10_p90": [sorted(ms)[max(0, len(ms) // 10)], sorted(ms)[min(len(ms) - 1, (9 * len(ms)) // 10)]],
        "wall_s_timed_region": wall, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": case.w.dtype, "data": "synthetic",
        "config": dict(case.config(), l2=(f"{args.flush_mb} MiB buffer written before every timed step; "
                                          "inputs also larger than L2"),
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": case.unit, "h2d_bytes_per_step": case.h2d,
                "d2h_bytes_per_step": case.d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * case.launches_per_step,
        "clocks": clk,
        "sustained": sustained,
        "fusion_study": fusion,
        "peaks": {k: peaks.get(k) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "source", "ffma")},
    }

    if not args.no_extras and world == 1:
        extras = {}
        for name in args.extras:
            if name == args.workload:
                continue
            c = make_case(name, dev)
            ms_x = time_steps(c, args.steps, args.warmup, stream, flush)
            sec = statistics.mean(ms_x) / 1e3
            r = c.roofline(sec, peaks)
            r["frac"] = r["achieved"] / r["peak"]
            r["traffic"] = measured_traffic(c)
            extras[name] = {"value": c.units / sec, "unit": c.unit, "ms_per_step": sec * 1e3,
                            "ms_median": statistics.median(ms_x), "roofline": r}
            if isinstance(c, GemmCase) and not args.no_fusion_study:
                ms_u = time_steps(c, max(5, min(50, args.steps)), 3, stream, flush, fn=c.run_unfused)
                extras[name]["fusion_study"] = {"fused_ms": statistics.median(ms_x),
                                                "unfused_ms": statistics.median(ms_u),
                                                "speedup": statistics.median(ms_u) / statistics.median(ms_x)}
            if args.extras_e2e:
                ms_e = time_steps(c, 5, 2, stream, flush, e2e=True)
                extras[name]["e2e"] = {"value": c.units / (statistics.mean(ms_e) / 1e3), "unit": c.unit,
                                       "h2d_bytes_per_step": c.h2d, "d2h_bytes_per_step": c.d2h}
            del c
            torch.cuda.empty_cache()
        line["workloads"] = extras

    if not args.no_extras and world == 1 and not args.no_small_m:
        line["small_m_graph"] = {"workload": "fp16_mlp3_softplus_128w (rows varied)",
                                 "method": "CUDA graph of 20 back-to-back calls, median of 20 replays, L2 warm",
                                 "rows": small_m_study(dev, stream)}

    if not args.no_extras and world == 1 and not args.no_fp32_sweep:
        line["fp32_sweep"] = {"workload": "fp32_gemm_bias_gelu_N (M = N = K)",
                              "method": "median of 100 calls, 512 MiB L2 flush before each",
                              "peak_tflops": peaks["ffma"]["tflops"], "peak_source": peaks["ffma"]["source"],
                              "sizes": fp32_sweep(dev, stream, flush, peaks["ffma"]["tflops"])}

    if rank == 0 and not args.no_cpu_baseline:
        units, dt, sample = calibrated_cpu_sample(case, 12.0)
        line["cpu_baseline"] = {"value": units / dt, "unit": case.unit, "cores": cpu_cores(), "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE)
    p.add_argument("--extras", nargs="*", default=["fp32_gemm_bias_gelu_4096", "fp16_mlp3_softplus_128w_2p20rows",
                                                   "fp16_mlp5_softplus_64w_2p22rows",
                                                   "fp16_mlp3_softplus_128w_2p20rows_train"])
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-fp32-sweep", action="store_true")
    p.add_argument("--no-fusion-study", action="store_true")
    p.add_argument("--no-small-m", action="store_true")
    p.add_argument("--flush-mb", type=int, default=512, help="L2 flush buffer written before each step (0: none)")
    p.add_argument("--M", type=int, default=None, help="override the GEMM workload's M (profiling a smaller case)")
    p.add_argument("--N", type=int, default=None)
    p.add_argument("--K", type=int, default=None)
    p.add_argument("--rows", type=int, default=None, help="override the MLP workload's row count")
    p.add_argument("--no-extras-e2e", dest="extras_e2e", action="store_false")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sustained-s", type=float, default=3.0,
                   help="seconds of back-to-back calls for the sustained leg (0: skip it)")
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
