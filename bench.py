#!/usr/bin/env python
"""Benchmark of the MXFP8 routed-expert hot path on GB300.

The reported line is the largest configuration that fits one GPU: the routed SwiGLU expert
forward + backward (G=2 experts, M=65600 tokens split 39360/26240, D=5120, H=8192; gate/up
weights [2, 8192, 5120], down [2, 5120, 8192]; synthetic bf16 data, random weights).  One step
is one pass of the whole path through the C ABI (libmxfp8moe.so):

    quantize x (row + token-wise) and the three expert weights (plain + transposed)
    gate/up grouped GEMMs with the SwiGLU and its MXFP8 quantization fused in the epilogue
    down grouped GEMM
    quantize dY; down dgrad and wgrad; SwiGLU backward with dh1, dh3 quantized in the same kernel
    dx = dh1 Wg + dh3 Wu (one GEMM); gate and up wgrads

`value` = algorithmic GEMM FLOPs of the step (9 x 2*M*D*H) / step time with the inputs resident
in HBM.  `e2e` = the same metric with the inputs copied in from pinned host memory and the
outputs (y, dx, dWg, dWu, dWd) copied back inside every step.  `roofline` is the kernel with the
largest share of the step time.  The same invocation also measures (extra keys): the tiny,
Llama4-Scout-like and imbalanced-experts fwd+bwd configurations, the quantization bandwidth
sweep, bf16 cuBLAS baselines, SQNR against the unquantized product, and the CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

Multi-GPU: independent replicas (the path has no exchange step), one process per GPU under
torchrun; the max step time over ranks sets `value`.  --impl reference times the CPU oracle
(fp64, plain C, OpenMP over the host cores) on a bounded sample of the same workload and prints
the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP8 grouped-GEMM fwd+bwd TFLOP/s & % MXFP8 peak; quantize GB/s vs HBM"
FP8_OVER_BF16 = 2.0      # nominal dense fp8 / bf16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
NOMINAL_FP8_TFLOPS = 4500.0
L2_BYTES = 129 * 2 ** 20

WORKLOAD_TEXT = {
    "swiglu": "SwiGLU routed expert fwd+bwd: G=2, M=65600 (39360/26240), D=5120, H=8192, gate/up W[2,8192,5120], "
              "down W[2,5120,8192]; gate/up GEMMs with the SwiGLU and its MXFP8 quantization fused into the "
              "epilogue, 9 GEMMs, the SwiGLU backward and the quantization of dh1, dh3 in one kernel",
    "swiglu_unfused": "SwiGLU routed expert fwd+bwd as swiglu, with separate gate and up GEMMs, the SwiGLU and "
                      "its backward in torch bf16 and separate ROW|COL quantizations of h, dh1, dh3",
    "scout": "Llama4-Scout-like routed experts fwd+bwd: G=8, K=5120, N=8192, M=16384 tokens, Zipf(1.1) group "
             "sizes in 32-token chunks (seed 0)",
    "imbalanced": "Fine-grained imbalanced experts fwd+bwd: G=16, K=7168, N=2048, M=32768, group 1 = 13120 tokens, "
                  "groups 0/7/15 empty, 1% x100 activation outliers",
    "tiny": "Tiny: G=2, A[256,256], offs [128,256], W[2,128,256] (latency-bound; parity case)",
    "scout_w32": "Llama4-Scout-like routed experts fwd+bwd with the expert weights quantized with one scale per "
                 "32x32 block (one quantization for the forward and the dgrad)",
    "scout_stab": "Llama4-Scout-like routed experts fwd+bwd with the stability variants: random Hadamard "
                  "transform of both wgrad operands along the tokens, stochastic rounding of the output gradient",
    "scout_mb4": "Llama4-Scout-like routed experts, one optimizer step of 4 microbatches (seeds 0-3): W quantized "
                 "once (prequantized-weight cache), then fwd+bwd per microbatch",
}
CONFIG_NAMES = {"tiny": "C1", "scout": "C2", "swiglu": "C3", "imbalanced": "C4"}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the dominant kernel of the
# SwiGLU step, from a one-pass ncu capture of this command, valid only while the GEMM sources hash
# to the recorded value (the kernel is then unchanged since the counters were taken).
DOMINANT_TRAFFIC = {"kernel": "grouped_mm_pair_kernel", "bytes_per_launch": 3133892147, "src_sha": "d244b0c85f4bdfba"}


def kernel_src_sha() -> str:
    h = hashlib.sha256()
    for f in ("grouped_mm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "mxfp8_precision_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="swiglu", choices=sorted(WORKLOAD_TEXT) + ["sweep"],
                    help="swiglu (default: the reported line); the others are extra measurements")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--no-baseline", action="store_true", help="skip the cuBLAS bf16 comparison")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other configurations and the sweep (headline only)")
    return ap.parse_args(argv)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest value over all ranks (the slowest rank's time sets the job's throughput)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks during the timed region
class ClockSampler:
    """Read-only SM clock / power / clock-event-reason samples every ~5 ms through NVML (ctypes,
    in-process), so a sub-second timed region still gets tens of samples; nvidia-smi polling as a
    fallback.  Nothing is set: only query calls are made."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.samples = []
        self.period = period_s
        self.stop_evt = threading.Event()
        self.source = None
        self.sm_max = None
        self.proc = None
        self.thread = None
        try:
            self._init_nvml(device_index)
            self.source = f"nvml every {period_s * 1e3:.0f} ms"
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
        except Exception:  # noqa: BLE001 - any NVML failure: fall back to nvidia-smi
            self._init_smi(device_index)
        if self.thread is not None:
            self.thread.start()

    def _init_nvml(self, device_index):
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(device_index)
        ok = False
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", None)
        dev = getattr(props, "pci_device_id", None)
        if bus is not None and dom is not None and dev is not None:
            ident = f"{dom:08X}:{bus:02X}:{dev:02X}.0".encode()
            ok = L.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(ident), ctypes.byref(h)) == 0
        if not ok and getattr(props, "uuid", None) is not None:
            ident = ("GPU-" + str(props.uuid)).encode()
            ok = L.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(ident), ctypes.byref(h)) == 0
        if not ok and not os.environ.get("CUDA_VISIBLE_DEVICES"):
            ok = L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(h)) == 0
        if not ok:
            raise OSError("no NVML handle for the device")
        mx = ctypes.c_uint()
        if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.sm_max = float(mx.value)
        self.L, self.h = L, h
        fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else L.nvmlDeviceGetCurrentClocksThrottleReasons

    def _poll_nvml(self):
        L, h = self.L, self.h
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_evt.is_set():
            t = time.time()
            c = float(clk.value) if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 else None
            p = pw.value / 1000.0 if L.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
            r = int(rs.value) if self.reasons_fn(h, ctypes.byref(rs)) == 0 else 0
            self.samples.append((t, c, p, r))
            time.sleep(self.period)

    def _init_smi(self, device_index):
        fields = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active"]
        cmd = ["nvidia-smi", "-i", str(device_index), "--query-gpu=" + ",".join(fields),
               "--format=csv,noheader,nounits", "-lms", "20"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.source = "nvidia-smi every 20 ms"
        self.thread = threading.Thread(target=self._read_smi, daemon=True)

    def _read_smi(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        for line in self.proc.stdout:
            p = [s.strip() for s in line.split(",")]
            if len(p) == 4:
                self.sm_max = num(p[1]) or self.sm_max
                r = int(p[3], 16) if p[3].startswith("0x") else 0
                self.samples.append((time.time(), num(p[0]), num(p[2]), r))

    def stop(self):
        self.stop_evt.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no clock samples"], "samples": 0,
                    "source": self.source}
        sm = [s[1] for s in win if s[1] is not None]
        pw = [s[2] for s in win if s[2] is not None]
        bits = 0
        for s in win:
            bits |= s[3]
        reasons = sorted(name for b, name in self.REASONS.items() if bits & b)
        counts = {name: sum(1 for s in win if s[3] & b) for b, name in self.REASONS.items() if bits & b}
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": self.sm_max, "reasons": reasons,
                "reason_samples": counts, "samples": len(win), "sm_mhz_min": min(sm) if sm else None,
                "power_w_median": float(np.median(pw)) if pw else None, "power_w_max": max(pw) if pw else None,
                "source": self.source}


# ---------------------------------------------------------------- steps, through the C ABI
def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def gemm_kernel_of(out_width: int) -> str:
    """The library's kernel for a plain fwd / dgrad / wgrad whose output is out_width columns wide."""
    return "grouped_mm_pair_kernel" if out_width >= 256 else "grouped_mm_kernel<128>"


def _blocked_expert_bytes(rows, cols):
    return ((rows + 127) // 128) * 128 * ((cols + 127) // 128) * 4


class _CallList:
    """A list of C-ABI calls (name, function, argument tuple) run back to back on one stream."""

    def run(self, stream, events=None):
        for name, fn, args in self.calls:
            if events is not None:
                events[name][0].record(stream)
            rc = fn(*args, ctypes.c_void_p(stream.cuda_stream))
            if rc != 0:
                raise RuntimeError(f"{name}: {self.mx._lib.STATUS_NAMES.get(rc, rc)}")
            if events is not None:
                events[name][1].record(stream)

    def check_status(self):
        self.mx.read_status(self.status, type(self).__name__)


class Step(_CallList):
    """One grouped-GEMM problem: quantize A (row + token-wise), W (plain + transposed), dOut (row +
    token-wise); fwd, dgrad, wgrad."""

    def __init__(self, w: dict, device, w_block32: bool = False, stability: bool = False,
                 skip_w_quant: bool = False, shared=None):
        import mxfp8_precision_moe_gb300 as mx

        L = mx.load()
        self.mx, self.L = mx, L
        G, M, N, K = w["G"], w["M"], w["N"], w["K"]
        self.G, self.M, self.N, self.K = G, M, N, K
        u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=device)
        bf = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=device)
        self.A, self.D = w["A"].to(device), w["dOut"].to(device)
        self.W = shared.W if shared is not None else w["W"].to(device)
        self.offs = w["offs"].to(device)
        self.sizes = list(map(int, w["sizes"]))
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        sb, sc = mx.mxfp8_scale_bytes, mx.mxfp8_scale_bytes_colgroups
        self.aq, self.as_ = u8(M, K), u8(sb(M, K, G, 1))
        self.aTq, self.aTs = u8(K, M), u8(sc(K, M, G))
        if shared is not None:
            self.wq, self.ws, self.wTq, self.wTs = shared.wq, shared.ws, shared.wTq, shared.wTs
        else:
            self.wq, self.ws = u8(G, N, K), u8(G, _blocked_expert_bytes(N, K))
            self.wTq, self.wTs = u8(G, K, N), u8(G, _blocked_expert_bytes(K, N))
        self.dq, self.ds = u8(M, N), u8(sb(M, N, G, 1))
        self.dTq, self.dTs = u8(N, M), u8(sc(N, M, G))
        self.out, self.dA, self.dW = bf(M, N), bf(M, K), bf(G, N, K)
        P, st, RC = _ptr, _ptr(self.status), 3
        calls = [
            ("quant_A", L.mxfp8_quantize_2d, (P(self.A), M, K, RC, 1, P(self.offs), G, P(self.aq), P(self.as_),
                                              P(self.aTq), P(self.aTs), st)),
            ("quant_W", L.mxfp8_quantize_3d_experts, (P(self.W), G, N, K, RC | (4 if w_block32 else 0), 1,
                                                      P(self.wq), P(self.ws), P(self.wTq), P(self.wTs), st)),
            ("fwd", L.mxfp8_grouped_mm_fwd, (P(self.aq), P(self.as_), P(self.wq), P(self.ws), P(self.offs), G, M,
                                             N, K, P(self.out), st)),
            ("quant_dOut", L.mxfp8_quantize_2d, (P(self.D), M, N, RC, 1, P(self.offs), G, P(self.dq), P(self.ds),
                                                 P(self.dTq), P(self.dTs), st)),
            ("dgrad", L.mxfp8_grouped_mm_dgrad, (P(self.dq), P(self.ds), P(self.wTq), P(self.wTs), P(self.offs), G,
                                                 M, N, K, P(self.dA), st)),
            ("wgrad", L.mxfp8_grouped_mm_wgrad, (P(self.dTq), P(self.dTs), P(self.aTq), P(self.aTs), P(self.offs), G,
                                                 M, N, K, P(self.dW), st)),
        ]
        if stability:
            # Hadamard transform of both wgrad operands along the tokens (one seed), stochastic
            # rounding of both dOut copies
            seed = 0x5EED
            byname = dict((c[0], c) for c in calls)
            byname["quant_A"] = ("quant_A", L.mxfp8_quantize_2d_opts,
                                 (P(self.A), M, K, RC, 1, P(self.offs), G, 4, seed, P(self.aq), P(self.as_),
                                  P(self.aTq), P(self.aTs), st))
            byname["quant_dOut"] = ("quant_dOut", L.mxfp8_quantize_2d_opts,
                                    (P(self.D), M, N, RC, 1, P(self.offs), G, 1 | 4, seed, P(self.dq), P(self.ds),
                                     P(self.dTq), P(self.dTs), st))
            calls = [byname[c[0]] for c in calls]
        if skip_w_quant or shared is not None:
            calls = [c for c in calls if c[0] != "quant_W"]
        self.calls = calls
        f = 2.0 * M * N * K
        self.gemm_flops = {"fwd": f, "dgrad": f, "wgrad": f}
        self.flops = 3 * f
        e8 = 1 + 1 / 32  # e4m3 code + E8M0 scale bytes per element
        self.gemm_bytes = {"fwd": (M * K + G * N * K) * e8 + 2 * M * N,
                           "dgrad": (M * N + G * N * K) * e8 + 2 * M * K,
                           "wgrad": (N * M + K * M) * e8 + 2 * G * N * K}
        qb = lambda e: e * (2 + 2 + 2 / 32)
        self.bytes = {"quant_A": qb(M * K), "quant_W": qb(G * N * K), "quant_dOut": qb(M * N)}
        quant = "quant_tile_kernel<ROW|COL" + (", ext>" if stability else ">")
        self.kernel_of = {"quant_A": quant, "quant_W": "quant_tile_kernel<ROW|COL" + ("|32x32>" if w_block32 else ">"),
                          "quant_dOut": quant, "fwd": gemm_kernel_of(N), "dgrad": gemm_kernel_of(K),
                          "wgrad": gemm_kernel_of(K)}

    def inputs(self):
        return [self.A, self.W, self.D, self.offs]

    def outputs(self):
        return [self.out, self.dA, self.dW]


class StepGroup(_CallList):
    """Several grouped-GEMM problems back to back as one step (microbatches sharing W)."""

    def __init__(self, parts: list, device):
        self.parts = []
        for i, w in enumerate(parts):
            self.parts.append(Step(w, device, shared=self.parts[0] if i else None))
        self.calls, self.gemm_flops, self.gemm_bytes, self.bytes, self.kernel_of = [], {}, {}, {}, {}
        for i, st in enumerate(self.parts):
            for name, fn, argv in st.calls:
                key = f"mb{i}.{name}"
                self.calls.append((key, fn, argv))
                self.kernel_of[key] = st.kernel_of[name]
                if name in st.gemm_flops:
                    self.gemm_flops[key] = st.gemm_flops[name]
                    self.gemm_bytes[key] = st.gemm_bytes[name]
                else:
                    self.bytes[key] = st.bytes[name]
        self.flops = sum(st.flops for st in self.parts)
        p0 = self.parts[0]
        self.G, self.M, self.N, self.K, self.mx, self.sizes = p0.G, p0.M, p0.N, p0.K, p0.mx, p0.sizes

    def check_status(self):
        for st in self.parts:
            st.check_status()


def swiglu_backward_bf16(dh: torch.Tensor, h1: torch.Tensor, h3: torch.Tensor):
    """(dh1, dh3) of h = silu(h1) * h3 with torch's bf16 autograd ops (the unfused comparison route)."""
    dh3 = dh * torch.nn.functional.silu(h1)
    dh1 = torch.ops.aten.silu_backward(dh * h3, h1)
    return dh1, dh3


class SwiGLUStep(_CallList):
    """One fwd+bwd of the SwiGLU routed expert y = (silu(x Wg^T) * (x Wu^T)) Wd^T through the C ABI.

    fused:   the gate/up GEMMs write h1, h3 and h already quantized both ways (one kernel); in the
             backward one kernel computes dh1, dh3 and quantizes both both ways, and one GEMM gives
             dx = dh1 Wg + dh3 Wu;
    unfused: two forward GEMMs, h = silu(h1) * h3 in torch bf16, a ROW|COL quantization of h; in the
             backward the SwiGLU backward in torch bf16 ops and two ROW|COL quantizations.
    Both run the down GEMM, and in the backward: dY quantized both ways, down dgrad and wgrad, the
    gate/up dgrads and wgrads.  Entries whose name starts with "torch." are torch elementwise glue,
    not library kernels.  skip_w_quant: the expert weights arrive prequantized (their quantization
    happens once per optimizer step, outside the step)."""

    def __init__(self, s: dict, device, fused: bool = True, skip_w_quant: bool = False):
        import mxfp8_precision_moe_gb300 as mx

        L = mx.load()
        self.mx, self.L = mx, L
        G, M, D, H = s["G"], s["M"], s["D"], s["H"]
        self.G, self.M, self.D, self.H = G, M, D, H
        self.sizes = list(map(int, s["sizes"]))
        u8 = lambda *sh: torch.empty(sh, dtype=torch.uint8, device=device)
        bf = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)
        P = _ptr
        sb, sc = mx.mxfp8_scale_bytes, mx.mxfp8_scale_bytes_colgroups
        self.x, self.dY, self.offs = s["x"].to(device), s["dY"].to(device), s["offs"].to(device)
        self.W = {n: s[n].to(device) for n in ("Wg", "Wu", "Wd")}
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        st = P(self.status)
        RC = 3
        tok = lambda cols: (u8(M, cols), u8(sb(M, cols, G, 1)), u8(cols, M), u8(sc(cols, M, G)))
        xq = tok(D)
        wq = {}
        for n, (r, c) in (("Wg", (H, D)), ("Wu", (H, D)), ("Wd", (D, H))):
            wq[n] = (u8(G, r, c), u8(G, _blocked_expert_bytes(r, c)), u8(G, c, r), u8(G, _blocked_expert_bytes(c, r)))
        self.wq = wq
        h1, h3 = bf(M, H), bf(M, H)
        hq = tok(H)
        dYq = tok(D)
        dh, dh1, dh3 = bf(M, H), bf(M, H), bf(M, H)
        a1, a3 = tok(H), tok(H)
        self.y, self.dx, dx2 = bf(M, D), bf(M, D), bf(M, D)
        self.dWg, self.dWu, self.dWd = bf(G, H, D), bf(G, H, D), bf(G, D, H)
        self.h1 = h1
        self.keep = [xq, h1, h3, hq, dYq, dh, dh1, dh3, a1, a3, dx2]
        offs, x, dY = P(self.offs), P(self.x), P(self.dY)
        q = lambda t4: tuple(P(t) for t in t4)
        y, dx, dWg, dWu, dWd = self.y, self.dx, self.dWg, self.dWu, self.dWd

        def glue(fn):
            def call(*args):
                fn()
                return 0
            return call

        def swiglu_fwd_torch():
            torch.mul(torch.nn.functional.silu(h1), h3, out=dh)  # dh holds h in the forward

        def swiglu_bwd_torch():
            g1, g3 = swiglu_backward_bf16(dh, h1, h3)
            dh1.copy_(g1)
            dh3.copy_(g3)

        calls = [("quant_x", L.mxfp8_quantize_2d, (x, M, D, RC, 1, offs, G, *q(xq), st))]
        if not skip_w_quant:
            for n, (r, c) in (("Wg", (H, D)), ("Wu", (H, D)), ("Wd", (D, H))):
                calls.append((f"quant_{n}", L.mxfp8_quantize_3d_experts,
                              (P(self.W[n]), G, r, c, RC, 1, *q(wq[n]), st)))
        if fused:
            calls.append(("gateup_swiglu", L.mxfp8_grouped_mm_swiglu_fwd,
                          (*q(xq)[:2], *q(wq["Wg"])[:2], *q(wq["Wu"])[:2], offs, G, M, H, D, P(h1), P(h3),
                           *q(hq), st)))
        else:
            calls += [("fwd_gate", L.mxfp8_grouped_mm_fwd, (*q(xq)[:2], *q(wq["Wg"])[:2], offs, G, M, H, D, P(h1), st)),
                      ("fwd_up", L.mxfp8_grouped_mm_fwd, (*q(xq)[:2], *q(wq["Wu"])[:2], offs, G, M, H, D, P(h3), st)),
                      ("torch.swiglu", glue(swiglu_fwd_torch), ()),
                      ("quant_h", L.mxfp8_quantize_2d, (P(dh), M, H, RC, 1, offs, G, *q(hq), st))]
        calls += [
            ("fwd_down", L.mxfp8_grouped_mm_fwd, (*q(hq)[:2], *q(wq["Wd"])[:2], offs, G, M, D, H, P(y), st)),
            ("quant_dY", L.mxfp8_quantize_2d, (dY, M, D, RC, 1, offs, G, *q(dYq), st)),
            ("dgrad_down", L.mxfp8_grouped_mm_dgrad, (*q(dYq)[:2], *q(wq["Wd"])[2:], offs, G, M, D, H, P(dh), st)),
            ("wgrad_down", L.mxfp8_grouped_mm_wgrad, (*q(dYq)[2:], *q(hq)[2:], offs, G, M, D, H, P(dWd), st)),
        ]
        if fused:
            calls.append(("swiglu_bwd_quant", L.mxfp8_swiglu_bwd_quantize,
                          (P(dh), P(h1), P(h3), M, H, offs, G, *q(a1), *q(a3), st)))
            calls.append(("dgrad_gate_up", L.mxfp8_grouped_mm_dgrad2,
                          (*q(a1)[:2], *q(wq["Wg"])[2:], *q(a3)[:2], *q(wq["Wu"])[2:], offs, G, M, H, D, P(dx), st)))
        else:
            calls += [("torch.swiglu_bwd", glue(swiglu_bwd_torch), ()),
                      ("quant_dh1", L.mxfp8_quantize_2d, (P(dh1), M, H, RC, 1, offs, G, *q(a1), st)),
                      ("quant_dh3", L.mxfp8_quantize_2d, (P(dh3), M, H, RC, 1, offs, G, *q(a3), st)),
                      ("dgrad_gate", L.mxfp8_grouped_mm_dgrad, (*q(a1)[:2], *q(wq["Wg"])[2:], offs, G, M, H, D, P(dx), st)),
                      ("dgrad_up", L.mxfp8_grouped_mm_dgrad, (*q(a3)[:2], *q(wq["Wu"])[2:], offs, G, M, H, D, P(dx2), st)),
                      ("torch.add", glue(lambda: dx.add_(dx2)), ())]
        calls += [
            ("wgrad_gate", L.mxfp8_grouped_mm_wgrad, (*q(a1)[2:], *q(xq)[2:], offs, G, M, H, D, P(dWg), st)),
            ("wgrad_up", L.mxfp8_grouped_mm_wgrad, (*q(a3)[2:], *q(xq)[2:], offs, G, M, H, D, P(dWu), st)),
        ]
        self.calls = calls
        f1 = 2.0 * M * D * H
        self.gemm_flops = {n: (2 * f1 if n in ("gateup_swiglu", "dgrad_gate_up") else f1) for n, _, _ in calls
                           if n.startswith(("fwd_", "dgrad_", "wgrad_", "gateup"))}
        self.flops = 9 * f1
        e8 = 1 + 1 / 32  # e4m3 code + E8M0 scale bytes per element
        gb = {"fwd_gate": (M * D + G * H * D) * e8 + 2 * M * H, "fwd_up": (M * D + G * H * D) * e8 + 2 * M * H,
              "gateup_swiglu": (M * D + 2 * G * H * D) * e8 + 4 * M * H + 2 * M * H * e8,
              "fwd_down": (M * H + G * D * H) * e8 + 2 * M * D, "dgrad_down": (M * D + G * D * H) * e8 + 2 * M * H,
              "wgrad_down": (D * M + H * M) * e8 + 2 * G * D * H,
              "dgrad_gate_up": 2 * (M * H + G * H * D) * e8 + 2 * M * D,
              "dgrad_gate": (M * H + G * H * D) * e8 + 2 * M * D, "dgrad_up": (M * H + G * H * D) * e8 + 2 * M * D,
              "wgrad_gate": (H * M + D * M) * e8 + 2 * G * H * D, "wgrad_up": (H * M + D * M) * e8 + 2 * G * H * D}
        self.gemm_bytes = {n: gb[n] for n in self.gemm_flops}
        qb = lambda e: e * (2 + 2 + 2 / 32)
        self.bytes = {"quant_x": qb(M * D), "quant_Wg": qb(G * H * D), "quant_Wu": qb(G * H * D),
                      "quant_Wd": qb(G * D * H), "quant_dY": qb(M * D)}
        if fused:
            # reads dh, h1, h3; writes dh1 and dh3 codes both ways with their scales
            self.bytes["swiglu_bwd_quant"] = M * H * (6 + 2 * (2 + 2 / 32))
        else:
            self.bytes.update(quant_h=qb(M * H), quant_dh1=qb(M * H), quant_dh3=qb(M * H))
        ko = {}
        for n, _, _ in calls:
            if n.startswith("torch."):
                ko[n] = n
            elif n.startswith("wgrad_"):
                ko[n] = gemm_kernel_of(D if n in ("wgrad_gate", "wgrad_up") else H)
            elif n == "gateup_swiglu":
                ko[n] = "grouped_mm_pair_kernel<swiglu epilogue>"
            elif n == "dgrad_gate_up":
                ko[n] = ("grouped_mm_pair_kernel<two-operand dgrad>" if D >= 256
                         else "grouped_mm_kernel<128, two-operand dgrad>")
            elif n.startswith(("fwd_", "dgrad_")):
                ko[n] = gemm_kernel_of(D if n in ("fwd_down", "dgrad_gate", "dgrad_up") else H)
            elif n == "swiglu_bwd_quant":
                ko[n] = "quant_tile_kernel<ROW|COL, swiglu backward>"
            else:
                ko[n] = "quant_tile_kernel<ROW|COL>"
        self.kernel_of = ko

    def inputs(self):
        return [self.x, self.dY, self.W["Wg"], self.W["Wu"], self.W["Wd"], self.offs]

    def outputs(self):
        return [self.y, self.dx, self.dWg, self.dWu, self.dWd]


# ---------------------------------------------------------------- timing
def time_step(step, stream, steps: int, warmup: int, world: int = 1, device=None, sample_clocks: bool = False):
    """Warm-up, then `steps` timed passes bracketed by a barrier and a synchronize on both sides.
    Returns (ms for all steps, mean ms per call, clock summary or None)."""
    for _ in range(max(warmup, 3)):
        step.run(stream)
    torch.cuda.synchronize()
    step.check_status()
    names = [c[0] for c in step.calls]
    ev = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for n in names}
          for _ in range(steps)]
    sampler = ClockSampler(device.index) if sample_clocks else None
    if sampler is not None:
        time.sleep(0.05)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for i in range(steps):
        step.run(stream, ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = None
    if sampler is not None:
        sampler.stop()
        clocks = sampler.summary(wall0, wall1)
    step.check_status()
    ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    per = {n: float(np.mean([e[n][0].elapsed_time(e[n][1]) for e in ev])) for n in names}
    return ms, per, clocks


def kernel_table(step, per, ms_step, pk):
    """Per call: time and throughput against its roofline; per kernel function: share of the step."""
    fp8_burst = pk["bf16"] * FP8_OVER_BF16
    calls = {}
    for n, t in per.items():
        d = {"ms": round(t, 4), "kernel": step.kernel_of[n]}
        if n in step.gemm_flops:
            tf = step.gemm_flops[n] / t / 1e9
            d.update(tflops=round(tf, 1), frac_fp8_peak=round(tf / fp8_burst, 3))
        elif n in step.bytes:
            gbs = step.bytes[n] / t / 1e6
            d.update(gbs=round(gbs, 1), frac_hbm=round(gbs / pk["hbm"], 3))
        calls[n] = d
    kernels = {}
    for n, t in per.items():
        k = kernels.setdefault(step.kernel_of[n], {"launches_per_step": 0, "ms_per_step": 0.0, "flops": 0.0,
                                                   "bytes": 0.0})
        k["launches_per_step"] += 1
        k["ms_per_step"] += t
        k["flops"] += step.gemm_flops.get(n, 0.0)
        k["bytes"] += step.bytes.get(n, 0.0)
    for k in kernels.values():
        k["share"] = round(k["ms_per_step"] / ms_step, 4)
        if k["flops"]:
            k["tflops"] = round(k["flops"] / k["ms_per_step"] / 1e9, 1)
            k["frac_fp8_peak"] = round(k["tflops"] / fp8_burst, 3)
        if k["bytes"]:
            k["gbs"] = round(k["bytes"] / k["ms_per_step"] / 1e6, 1)
            k["frac_hbm"] = round(k["gbs"] / pk["hbm"], 3)
        k["ms_per_step"] = round(k["ms_per_step"], 4)
        del k["flops"], k["bytes"]
    return calls, kernels


def roofline_of(step, per, kernels, pk, traffic_info=None):
    """The roofline object for the kernel with the largest share of the step time."""
    name = max((k for k in kernels if not k.startswith("torch.")), key=lambda k: kernels[k]["share"])
    launches = [n for n in per if step.kernel_of[n] == name]
    t_mean = float(np.mean([per[n] for n in launches]))
    flops = sum(step.gemm_flops.get(n, 0.0) for n in launches)
    if flops:
        peak = pk["bf16"] * FP8_OVER_BF16
        achieved = flops / len(launches) / t_mean / 1e9
        r = {"bound": "tensor", "kernel": name, "achieved": round(achieved, 1), "peak": round(peak, 1),
             "unit": "TFLOP/s", "frac": round(achieved / peak, 3),
             "frac_of_sustained_peak": round(achieved / (pk["bf16_sus"] * FP8_OVER_BF16), 3),
             "frac_of_nominal_4p5": round(achieved / NOMINAL_FP8_TFLOPS, 3),
             "peak_note": f"{pk['src']} burst bf16 {pk['bf16']} TFLOP/s x {FP8_OVER_BF16} (nominal dense fp8/bf16 "
                          f"ratio), of measured; sustained {pk['bf16_sus']} x {FP8_OVER_BF16} and the nominal "
                          f"{NOMINAL_FP8_TFLOPS:.0f} TFLOP/s beside it",
             "launches_per_step": len(launches), "mean_launch_ms": round(t_mean, 4),
             "algorithmic_per_launch": f"{flops / len(launches) / 1e12:.4f} TFLOP (2*M*N*K)"}
    else:
        nbytes = sum(step.bytes.get(n, 0.0) for n in launches)
        achieved = nbytes / len(launches) / t_mean / 1e6
        r = {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
             "frac": round(achieved / pk["hbm"], 3), "peak_note": f"{pk['src']} copy bandwidth",
             "launches_per_step": len(launches), "mean_launch_ms": round(t_mean, 4)}
    t = traffic_info or {}
    ok = t.get("kernel") == name and t.get("bytes_per_launch") and t.get("src_sha") == kernel_src_sha()
    r["traffic"] = t["bytes_per_launch"] if ok else None
    if flops and hasattr(step, "gemm_bytes"):
        algo = sum(step.gemm_bytes[n] for n in launches) / len(launches)
        r["algorithmic_bytes_per_launch"] = int(algo)
        if r["traffic"]:
            r["traffic_over_algorithmic"] = round(r["traffic"] / algo, 2)
    return r


# ---------------------------------------------------------------- information: SQNR vs the unquantized product
def _sqnr(ref: torch.Tensor, got: torch.Tensor) -> float:
    num = float((ref.double() ** 2).sum())
    den = float(((ref.double() - got.double()) ** 2).sum())
    return round(10.0 * np.log10(num / den), 2) if den > 0 else float("inf")


def _sample_rows(sizes, n_per_group, seed):
    rng = np.random.default_rng(seed)
    ends = np.cumsum(sizes)
    rows, groups = [], []
    for g, m in enumerate(sizes):
        if m:
            lo = int(ends[g] - m)
            r = np.unique(rng.integers(lo, lo + m, n_per_group))
            rows += list(map(int, r))
            groups += [g] * len(r)
    return rows, groups


def sqnr_step(step) -> dict:
    """SQNR (dB) of the MXFP8 fwd/dgrad/wgrad outputs against the fp64 product of the unquantized bf16
    inputs, on sampled rows (fwd, dgrad) and sampled dW rows of every group (wgrad)."""
    rows, groups = _sample_rows(step.sizes, 8, 7)
    A, W, D = step.A.double(), step.W, step.D.double()
    ref_o = torch.stack([A[r] @ W[g].double().T for r, g in zip(rows, groups)])
    ref_a = torch.stack([D[r] @ W[g].double() for r, g in zip(rows, groups)])
    idx = torch.tensor(rows, device=A.device)
    ends = np.cumsum(step.sizes)
    ref_w, got_w = [], []
    ns = torch.arange(0, step.N, max(1, step.N // 8), device=A.device)
    for g, m in enumerate(step.sizes):
        if m:
            lo, hi = int(ends[g] - m), int(ends[g])
            ref_w.append(D[lo:hi, ns].T @ A[lo:hi])
            got_w.append(step.dW[g, ns].double())
    return {"fwd": _sqnr(ref_o, step.out[idx]), "dgrad": _sqnr(ref_a, step.dA[idx]),
            "wgrad": _sqnr(torch.cat(ref_w), torch.cat(got_w))}


def sqnr_swiglu(step) -> dict:
    """SQNR (dB) of the expert's y and of the gate GEMM output h1 against fp64 from the unquantized bf16
    inputs (h = silu(h1) * h3 in fp64), on sampled token rows."""
    rows, groups = _sample_rows(step.sizes, 16, 8)
    x = step.x.double()
    ref_y, ref_h1 = [], []
    for r, g in zip(rows, groups):
        h1 = x[r] @ step.W["Wg"][g].double().T
        h3 = x[r] @ step.W["Wu"][g].double().T
        ref_h1.append(h1)
        ref_y.append((torch.nn.functional.silu(h1) * h3) @ step.W["Wd"][g].double().T)
    idx = torch.tensor(rows, device=x.device)
    return {"y": _sqnr(torch.stack(ref_y), step.y[idx]), "h1": _sqnr(torch.stack(ref_h1), step.h1[idx])}


# ---------------------------------------------------------------- bf16 cuBLAS baselines (per-group torch.mm)
def _time_fn(fn, stream, reps=5, warmup=2):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def bf16_baseline_step(step, stream) -> dict:
    """fwd, dgrad and wgrad of one grouped GEMM problem in bf16 as a per-group cuBLAS torch.mm loop."""
    ends = np.cumsum(step.sizes)
    A, W, D = step.A, step.W, step.D
    out, dA, dW = torch.empty_like(step.out), torch.empty_like(step.dA), torch.empty_like(step.dW)
    spans = [(g, int(e - m), int(e)) for g, (m, e) in enumerate(zip(step.sizes, ends)) if m]

    def fwd():
        for g, lo, hi in spans:
            torch.mm(A[lo:hi], W[g].t(), out=out[lo:hi])

    def dgrad():
        for g, lo, hi in spans:
            torch.mm(D[lo:hi], W[g], out=dA[lo:hi])

    def wgrad():
        for g, lo, hi in spans:
            torch.mm(D[lo:hi].t(), A[lo:hi], out=dW[g])

    t = {n: _time_fn(f, stream) for n, f in (("fwd", fwd), ("dgrad", dgrad), ("wgrad", wgrad))}
    f = step.gemm_flops["fwd"]
    return {"kernel": "cuBLAS bf16, per-group torch.mm loop (torch._grouped_mm is not used: it failed on this "
                      "GPU in an earlier run)",
            "ms": {k: round(v, 4) for k, v in t.items()}, "ms_fwd_bwd": round(sum(t.values()), 4),
            "tflops": {k: round(f / v / 1e9, 1) for k, v in t.items()}}


def bf16_baseline_swiglu(step, stream) -> dict:
    """The SwiGLU expert fwd+bwd in bf16: 9 per-group cuBLAS torch.mm GEMMs, torch's silu * mul, its
    autograd backward ops and the dx add."""
    ends = np.cumsum(step.sizes)
    x, dY, Wg, Wu, Wd = step.x, step.dY, step.W["Wg"], step.W["Wu"], step.W["Wd"]
    M, D, H = step.M, step.D, step.H
    bf = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=x.device)
    h1, h3, h, y, dh, dx, dx2 = bf(M, H), bf(M, H), bf(M, H), bf(M, D), bf(M, H), bf(M, D), bf(M, D)
    dWg, dWu, dWd = torch.empty_like(Wg), torch.empty_like(Wu), torch.empty_like(Wd)
    spans = [(g, int(e - m), int(e)) for g, (m, e) in enumerate(zip(step.sizes, ends)) if m]

    def gemms_fwd():
        for g, lo, hi in spans:
            torch.mm(x[lo:hi], Wg[g].t(), out=h1[lo:hi])
            torch.mm(x[lo:hi], Wu[g].t(), out=h3[lo:hi])

    def swiglu():
        torch.mul(torch.nn.functional.silu(h1), h3, out=h)

    def down_fwd():
        for g, lo, hi in spans:
            torch.mm(h[lo:hi], Wd[g].t(), out=y[lo:hi])

    def down_bwd():
        for g, lo, hi in spans:
            torch.mm(dY[lo:hi], Wd[g], out=dh[lo:hi])
            torch.mm(dY[lo:hi].t(), h[lo:hi], out=dWd[g])

    grads = {}

    def swiglu_bwd():
        grads["d1"], grads["d3"] = swiglu_backward_bf16(dh, h1, h3)

    def front_bwd(d1, d3):
        for g, lo, hi in spans:
            torch.mm(d1[lo:hi], Wg[g], out=dx[lo:hi])
            torch.mm(d3[lo:hi], Wu[g], out=dx2[lo:hi])
            torch.mm(d1[lo:hi].t(), x[lo:hi], out=dWg[g])
            torch.mm(d3[lo:hi].t(), x[lo:hi], out=dWu[g])

    def whole():
        gemms_fwd(); swiglu(); down_fwd(); down_bwd(); swiglu_bwd()
        front_bwd(grads["d1"], grads["d3"])
        dx.add_(dx2)

    def gemms_only():
        gemms_fwd(); down_fwd(); down_bwd()
        front_bwd(dh, dh)

    t_all = _time_fn(whole, stream, reps=3)
    t_gemm = _time_fn(gemms_only, stream, reps=3)
    return {"kernel": "cuBLAS bf16 per-group torch.mm (9 GEMMs) + torch SwiGLU, its backward and the dx add",
            "ms_step": round(t_all, 4), "ms_gemms": round(t_gemm, 4),
            "tflops_gemms": round(step.flops / t_gemm / 1e9, 1)}


# ---------------------------------------------------------------- the CPU oracle (cpu_baseline / reference arm)
def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5)
        for line in r.stdout.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """A bounded sample of the SwiGLU expert's gate GEMM (x Wg^T, K = D = 5120) run by the CPU oracle
    from the bf16 inputs: 128 token rows of each expert times 128 weight rows of that expert, the
    quantization of exactly those operands included (the oracle's exhaustive E4M3 encoding is
    serial; its GEMM loops run on OpenMP threads).  One rep = 2 * 256 * 128 * 5120 GEMM FLOPs."""

    ROWS, COLS = 128, 128

    def __init__(self, s_cpu: dict):
        import oracle

        oracle.lib()
        self.o = oracle
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        ends = np.cumsum(s_cpu["sizes"])
        starts = ends - np.asarray(s_cpu["sizes"])
        self.x = np.concatenate([bits(s_cpu["x"][int(lo):int(lo) + self.ROWS]) for lo in starts])
        self.w = [bits(s_cpu["Wg"][g][:self.COLS]) for g in range(s_cpu["G"])]
        self.ends = np.arange(1, s_cpu["G"] + 1) * self.ROWS
        self.flops = 2.0 * self.x.shape[0] * self.COLS * self.x.shape[1]

    def rep(self) -> float:
        o = self.o
        aq, as_ = o.quantize_rows(self.x)
        wq = [o.quantize_rows(w) for w in self.w]
        o.grouped_mm_rows(aq, as_, np.stack([q for q, _ in wq]), np.stack([s for _, s in wq]), self.ends)
        return self.flops


def oracle_rate(sample: OracleSample, threads: int, seconds: float):
    """Reps of the sample for about `seconds` with `threads` OpenMP threads: (TFLOP/s, reps, s)."""
    sample.o.set_num_threads(threads)
    flops, n, t0 = 0.0, 0, time.perf_counter()
    while True:
        flops += sample.rep()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return flops / el / 1e12, n, el


def cpu_baseline(s_cpu: dict) -> dict:
    sample = OracleSample(s_cpu)
    cores = host_cores()
    multi, n_m, el_m = oracle_rate(sample, cores, 10.0)
    single, n_s, el_s = oracle_rate(sample, 1, 10.0)
    return {"value": multi, "unit": "TFLOP/s", "cores": min(cores, OracleSample.ROWS), "kind": "oracle",
            "sample": f"gate GEMM x Wg^T of the SwiGLU expert on {sample.x.shape[0]} token rows x {sample.COLS} "
                      f"weight rows per expert, K=5120, quantization of those operands included: {n_m} reps in "
                      f"{el_m:.1f} s with {cores} OpenMP threads (the rows of a group are split across threads)",
            "single_thread": {"value": single, "cores": 1, "reps": n_s, "seconds": round(el_s, 1)},
            "host": {"cpu_model": cpu_model(), "cores": cores}}


# ---------------------------------------------------------------- end to end through host buffers
def host_link(device, nbytes: int = 256 << 20, reps: int = 4) -> dict:
    """Pinned-host <-> device copy rates of this box's link (GB/s): each direction alone, then both
    directions at once on two streams; the e2e step's copies cannot run faster than these."""
    h_src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def timed(h2d: bool, d2h: bool) -> float:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_out.wait_event(e0)
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s_in):
                    d_a.copy_(h_src, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    h_dst.copy_(d_b, non_blocking=True)
        s_in.wait_stream(s_out)
        e1.record(s_in)
        torch.cuda.synchronize()
        return reps * nbytes / (e0.elapsed_time(e1) * 1e6)

    timed(True, True)  # first touch of the pinned pages
    both = timed(True, True)
    return {"h2d_gbs": round(timed(True, False), 1), "d2h_gbs": round(timed(False, True), 1),
            "both_gbs_each": round(both, 1), "bytes_per_copy": nbytes}


def run_e2e(make_step, step, stream, world, device, n_steps: int):
    """The step with its inputs copied in from pinned host memory and its outputs copied out, as a
    3-stream pipeline over two device buffer sets: the copy-in of step i+1 and the copy-out of step
    i-1 overlap the kernels of step i (events order each buffer set's reuse)."""
    sets = [step, make_step()]
    h_in = [t.cpu().pin_memory() for t in step.inputs()]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in st.outputs()] for st in sets]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    mk = lambda: torch.cuda.Event(enable_timing=True)

    def pipeline(n: int):
        """n steps of the pipeline; returns its events (per step: copy-in, kernels, copy-out start/end)."""
        ev = {k: [mk() for _ in range(n)] for k in ("in0", "in1", "k0", "k1", "out0", "out1")}
        for i in range(n):
            st = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["k1"][i - 2])        # inputs of set i%2 no longer read
                ev["in0"][i].record(s_in)
                for d, h in zip(st.inputs(), h_in):
                    d.copy_(h, non_blocking=True)
                ev["in1"][i].record(s_in)
            stream.wait_event(ev["in1"][i])
            if i >= 2:
                stream.wait_event(ev["out1"][i - 2])        # outputs of set i%2 already copied out
            ev["k0"][i].record(stream)
            st.run(stream)
            ev["k1"][i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["k1"][i])
                ev["out0"][i].record(s_out)
                for h, d in zip(h_out[i % 2], st.outputs()):
                    h.copy_(d, non_blocking=True)
                ev["out1"][i].record(s_out)
        s_in.wait_stream(s_out)
        return ev

    # untimed warm-up: both buffer sets through the whole pipeline, copies included (the first copies of
    # a run, after the device had gone idle, have been seen at a tenth of the link's rate)
    pipeline(4)
    if world > 1:
        torch.cuda.synchronize()
        torch.distributed.barrier()
    # one GPU: the timed steps follow the warm-up with no idle gap; x0 marks the end of every warm-up
    # operation in stream order, and the timed copies start after it
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_in.wait_stream(stream)
    s_in.wait_stream(s_out)
    x0.record(s_in)
    host0 = time.perf_counter()
    ev = pipeline(n_steps)
    x1.record(s_in)
    host_ms = (time.perf_counter() - host0) * 1e3 / n_steps  # the host's enqueue time per step
    torch.cuda.synchronize()
    in_start, h2d_done, comp_start, comp_done, out_start, d2h_done = (
        ev[k] for k in ("in0", "in1", "k0", "k1", "out0", "out1"))
    for st in sets:
        st.check_status()
    xms = max_over_ranks(x0.elapsed_time(x1) / n_steps, world, device)
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = sum(t.numel() * t.element_size() for t in h_out[0])

    # each leg of the pipeline alone, on the step's own buffers
    def alone(fn, s) -> float:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        with torch.cuda.stream(s):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    legs = {"copy_in_ms": alone(lambda: [d.copy_(h, non_blocking=True) for d, h in zip(step.inputs(), h_in)], s_in),
            "kernels_ms": alone(lambda: step.run(stream), stream),
            "copy_out_ms": alone(lambda: [h.copy_(d, non_blocking=True) for h, d in zip(h_out[0], step.outputs())],
                                 s_out)}
    # the same legs inside the pipeline (median over the steps)
    med = lambda a, b: float(np.median([a[i].elapsed_time(b[i]) for i in range(n_steps)]))
    legs.update(piped_copy_in_ms=med(in_start, h2d_done), piped_kernels_ms=med(comp_start, comp_done),
                piped_copy_out_ms=med(out_start, d2h_done))
    legs = {k: round(v, 3) for k, v in legs.items()}
    # when each leg of the first steps started and ended (ms after the pipeline's first event)
    at = lambda e: round(x0.elapsed_time(e), 2)
    timeline = [{"in": [at(in_start[i]), at(h2d_done[i])],
                 "kernels": [at(comp_start[i]), at(comp_done[i])], "out": [at(out_start[i]), at(d2h_done[i])]}
                for i in range(min(n_steps, 4))]
    legs["copy_in_gbs"] = round(bi / (legs["copy_in_ms"] * 1e6), 1)
    legs["copy_out_gbs"] = round(bo / (legs["copy_out_ms"] * 1e6), 1)
    link = host_link(device)
    # with both directions busy, each step's copies need at least this long on this machine's link
    link["copy_ms_per_step"] = round(max(bi, bo) / (link["both_gbs_each"] * 1e6), 3)
    return {"value": round(world * step.flops / xms / 1e9, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(xms, 3), "steps": n_steps, "warmup_steps": 4,
            "pipeline": "copy-in, kernels and copy-out on 3 streams over 2 device buffer sets",
            "alone": legs, "timeline_ms": timeline, "host_enqueue_ms_per_step": round(host_ms, 3), "host_link": link}


# ---------------------------------------------------------------- native (GPU) arm
def make_step(name: str, dev):
    from mxfp8_precision_moe_gb300 import synth

    if name in ("swiglu", "swiglu_unfused"):
        s = synth.workload("swiglu", seed=0, device=dev)
        return (lambda: SwiGLUStep(s, dev, fused=name == "swiglu")), s
    if name == "scout_mb4":
        mbs = [synth.workload("scout", seed=i, device=dev) for i in range(4)]
        for w in mbs[1:]:
            w["W"] = mbs[0]["W"]  # one weight tensor for the whole optimizer step
        return (lambda: StepGroup(mbs, dev)), mbs[0]
    base = {"scout_w32": "scout", "scout_stab": "scout"}.get(name, name)
    w = synth.workload(base, seed=0, device=dev)
    return (lambda: Step(w, dev, w_block32=name == "scout_w32", stability=name == "scout_stab")), w


def step_flops(w: dict, name: str) -> float:
    if name in ("swiglu", "swiglu_unfused"):
        return 9 * 2.0 * w["M"] * w["D"] * w["H"]
    f = 3 * 2.0 * w["M"] * w["N"] * w["K"]
    return 4 * f if name == "scout_mb4" else f


def measure_config(name: str, dev, stream, pk, steps: int, warmup: int, baseline: bool) -> dict:
    """One extra configuration: its step timed, per-kernel table, SQNR and (optionally) bf16 baselines."""
    factory, w = make_step(name, dev)
    step = factory()
    ms, per, _ = time_step(step, stream, steps, warmup, device=dev)
    ms_step = ms / steps
    calls, kernels = kernel_table(step, per, ms_step, pk)
    gemm_ms = sum(per[n] for n in step.gemm_flops)
    fp8_burst = pk["bf16"] * FP8_OVER_BF16
    d = {"config": CONFIG_NAMES.get(name), "workload": WORKLOAD_TEXT[name], "ms_per_step": round(ms_step, 4),
         "tflops": round(step.flops / ms_step / 1e9, 1),
         "frac_fp8_peak_step": round(step.flops / ms_step / 1e9 / fp8_burst, 3),
         "frac_fp8_peak_gemms_only": round(step.flops / gemm_ms / 1e9 / fp8_burst, 3),
         "roofline": roofline_of(step, per, kernels, pk), "calls": calls, "kernels": kernels,
         "group_sizes": step.sizes}
    if isinstance(step, Step):
        d["sqnr_db"] = sqnr_step(step)
        if baseline:
            b = bf16_baseline_step(step, stream)
            nw = Step(w, dev, skip_w_quant=True)
            ms_nw, _, _ = time_step(nw, stream, steps, warmup, device=dev)
            del nw
            b["mxfp8_ms_step_W_prequantized"] = round(ms_nw / steps, 4)
            b["mxfp8_over_bf16"] = {
                "gemms_only": round(b["ms_fwd_bwd"] / gemm_ms, 3),
                "step_with_W_quantization": round(b["ms_fwd_bwd"] / ms_step, 3),
                "step_with_W_prequantized": round(b["ms_fwd_bwd"] / (ms_nw / steps), 3)}
            d["baseline_bf16"] = b
    del step
    torch.cuda.empty_cache()
    return d


def run_native(args, rank, world, local):
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    stream = torch.cuda.current_stream(dev)
    factory, w = make_step(args.workload, dev)
    step = factory()
    ms, per, clocks = time_step(step, stream, args.steps, args.warmup, world, dev, sample_clocks=True)
    ms_step = ms / args.steps
    calls, kernels = kernel_table(step, per, ms_step, pk)
    headline = args.workload == "swiglu"
    roof = roofline_of(step, per, kernels, pk, DOMINANT_TRAFFIC if headline else None)
    fp8_burst = pk["bf16"] * FP8_OVER_BF16
    gemm_ms = sum(per[n] for n in step.gemm_flops)
    flops = step_flops(w, args.workload)

    extras = {}
    if rank == 0 and world == 1:
        if isinstance(step, SwiGLUStep):
            extras["sqnr_db"] = sqnr_swiglu(step)
        elif isinstance(step, Step):
            extras["sqnr_db"] = sqnr_step(step)
        if not args.no_baseline and isinstance(step, SwiGLUStep) and headline:
            b = bf16_baseline_swiglu(step, stream)
            nw = SwiGLUStep(w, dev, fused=True, skip_w_quant=True)
            ms_nw, _, _ = time_step(nw, stream, args.steps, args.warmup, device=dev)
            del nw
            b["mxfp8_ms_step_W_prequantized"] = round(ms_nw / args.steps, 4)
            b["mxfp8_over_bf16"] = {"gemms_only": round(b["ms_gemms"] / gemm_ms, 3),
                                    "step_with_W_quantization": round(b["ms_step"] / ms_step, 3),
                                    "step_with_W_prequantized": round(b["ms_step"] / (ms_nw / args.steps), 3)}
            b["pages_context"] = "~1.8x over compiled BF16 for MoE shapes (MXFP8 training for MoEs; GB200)"
            extras["baseline_bf16"] = b
        elif not args.no_baseline and isinstance(step, Step):
            extras["baseline_bf16"] = bf16_baseline_step(step, stream)

    e2e = None
    if not args.no_e2e and hasattr(step, "inputs"):
        e2e = run_e2e(factory, step, stream, world, dev, n_steps=max(4, args.steps))  # as many steps as the kernel timing
    del step
    torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_extras and headline:
        extras["configs"] = {}
        for name in ("tiny", "scout", "imbalanced"):
            extras["configs"][CONFIG_NAMES[name]] = measure_config(name, dev, stream, pk, 50, 5,
                                                                   baseline=not args.no_baseline and name == "scout")
        extras["configs"]["C5"] = run_sweep(args)

    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(world * flops / ms_step / 1e9, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "config": CONFIG_NAMES.get(args.workload),
                   "group_sizes": list(map(int, w["sizes"])), "parallelism": f"replicas x{world}",
                   "l2": "inputs and working set far larger than L2 (129 MiB): no flush needed",
                   "frac_fp8_peak_step": round(flops / ms_step / 1e9 / fp8_burst, 3),
                   "frac_fp8_peak_gemms_only": round(flops / gemm_ms / 1e9 / fp8_burst, 3),
                   "frac_nominal_4p5_step": round(flops / ms_step / 1e9 / NOMINAL_FP8_TFLOPS, 3),
                   "peak_note": f"fractions of the {pk['src']} burst bf16 x {FP8_OVER_BF16} = {fp8_burst:.1f} TFLOP/s "
                                "unless named nominal (4.5 PFLOP/s dense fp8)"},
        "roofline": roof,
        "calls": calls,
        "kernels": kernels,
        "hbm_peak_gbs": pk["hbm"],
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(1 for n in per if not n.startswith("torch.")),
    }
    line.update(extras)
    return line, w


def run_sweep(args) -> dict:
    """Quantization bandwidth over the sweep shapes: bf16 [M,K] row, column, row+column (one read) and
    32x32 blocks, plus 3D expert weights [16,8192,5120] plain, transposed and both, and the stability
    variants; GB/s of algorithmic bytes (2 read + per direction 1 code + 1/32 scale byte per element)."""
    import mxfp8_precision_moe_gb300 as mx
    from mxfp8_precision_moe_gb300 import synth

    L = mx.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    stream = torch.cuda.current_stream(dev)
    sp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rows = []

    def time_call(fn, argv, nbytes, label, shape):
        for _ in range(3):
            fn(*argv, ctypes.c_void_p(stream.cuda_stream))
        torch.cuda.synchronize()
        n = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            rc = fn(*argv, ctypes.c_void_p(stream.cuda_stream))
            if rc != 0:
                raise RuntimeError(f"{label}: status {rc}")
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        gbs = nbytes / ms / 1e6
        rows.append({"shape": shape, "dirs": label, "us": round(ms * 1e3, 1), "gbs": round(gbs, 1),
                     "frac_hbm": round(gbs / pk["hbm"], 3)})

    u8 = lambda *shape: torch.empty(shape, dtype=torch.uint8, device=dev)
    for M in synth.SWEEP_M:
        for K in synth.SWEEP_K:
            x = synth.log_uniform_rows(M, K, seed=M + K, device=dev)
            q, qT = u8(M, K), u8(K, M)
            s_r, s_c = u8(mx.mxfp8_scale_bytes(M, K, 1, 1)), u8(mx.mxfp8_scale_bytes_colgroups(K, M, 1))
            s32 = u8(M // 32, K // 32)
            E = M * K
            for label, dirs, lay, out in (("row", 1, 1, (q, s_r, None, None)), ("col", 2, 1, (None, None, qT, s_c)),
                                          ("row+col", 3, 1, (q, s_r, qT, s_c)), ("32x32", 4, 0, (q, s32, None, None))):
                nb = E * (2 + 1 + 1 / 32) if label in ("row", "col") else \
                    E * (2 + 2 + 2 / 32) if label == "row+col" else E * (2 + 1 + 1 / 1024)
                time_call(L.mxfp8_quantize_2d, (sp(x), M, K, dirs, lay, None, 0, *[sp(t) for t in out], None), nb,
                          label, [M, K])
            del x, q, qT, s_r, s_c, s32
    # stability variants (mxfp8_quantize_2d_opts) on one activation shape, both copies
    M, K = 16384, 5120
    x = synth.log_uniform_rows(M, K, seed=M + K, device=dev)
    q, qT = u8(M, K), u8(K, M)
    s_r, s_c = u8(mx.mxfp8_scale_bytes(M, K, 1, 1)), u8(mx.mxfp8_scale_bytes_colgroups(K, M, 1))
    for label, opts in (("row+col SR", 1), ("row+col RHT(col)", 4), ("row+col RHT(row,col)", 6),
                        ("row+col SR+RHT(col)", 5)):
        time_call(L.mxfp8_quantize_2d_opts, (sp(x), M, K, 3, 1, None, 0, opts, 0x5EED, sp(q), sp(s_r), sp(qT),
                                             sp(s_c), None), M * K * (2 + 2 + 2 / 32), label, [M, K])
    del x, q, qT, s_r, s_c
    G, N, K = 16, 8192, 5120
    w = synth.randn_bf16((G, N, K), 1.0, seed=7, device=dev)
    q, s3 = u8(G, N, K), u8(G, _blocked_expert_bytes(N, K))
    qT, sT = u8(G, K, N), u8(G, _blocked_expert_bytes(K, N))
    E = G * N * K
    for label, dirs, out in (("3d plain", 1, (q, s3, None, None)), ("3d transposed", 2, (None, None, qT, sT)),
                             ("3d both", 3, (q, s3, qT, sT)), ("3d 32x32 both", 7, (q, s3, qT, sT))):
        nb = E * (2 + 2 + 2 / 32) if dirs & 3 == 3 else E * (2 + 1 + 1 / 32)
        time_call(L.mxfp8_quantize_3d_experts, (sp(w), G, N, K, dirs, 1, *[sp(t) for t in out], None), nb, label,
                  [G, N, K])
    del w, q, s3, qT, sT
    torch.cuda.empty_cache()
    plain = [r["frac_hbm"] for r in rows if "SR" not in r["dirs"] and "RHT" not in r["dirs"]]
    return {"config": "C5", "metric": "MXFP8 quantize GB/s (sweep)", "unit": "GB/s", "hbm_peak_gbs": pk["hbm"],
            "peak_note": f"{pk['src']} copy bandwidth",
            "workload": "quantization sweep: [M,K] M in 8192..131072, K in {5120, 8192}; 3D [16,8192,5120]; "
                        "N(0,1)*10^U(-4,4) per row",
            "min_frac_hbm_plain": min(plain), "best_frac_hbm": max(plain), "sweep": rows}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the machine's host cores (rank 0 only): each step is one rep of
    a bounded sample of the SwiGLU expert's gate GEMM, quantization included (OracleSample)."""
    if rank != 0:
        return
    from mxfp8_precision_moe_gb300 import synth

    s = synth.workload("swiglu", seed=0, device="cpu")
    sample = OracleSample(s)
    cores = host_cores()
    sample.o.set_num_threads(cores)
    for _ in range(args.warmup):
        sample.rep()
    flops, t0 = 0.0, time.perf_counter()
    for _ in range(args.steps):
        flops += sample.rep()
    el = time.perf_counter() - t0
    val = flops / el / 1e12
    desc = (f"one rep per step: gate GEMM x Wg^T of the SwiGLU expert on {sample.x.shape[0]} token rows x "
            f"{sample.COLS} weight rows per expert, K=5120, quantization of those operands included")
    line = {
        "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD_TEXT["swiglu"], "config": "C3"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": min(cores, OracleSample.ROWS), "kind": "oracle",
                         "sample": desc, "host": {"cpu_model": cpu_model(), "cores": cores}},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return
    if args.workload == "sweep":
        if rank == 0:
            print(json.dumps(run_sweep(args)), flush=True)
        return
    res = run_native(args, rank, world, local)
    if rank == 0 and res is not None:
        line, w = res
        if not args.no_cpu and world == 1 and args.workload == "swiglu":
            w_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in w.items()}
            line["cpu_baseline"] = cpu_baseline(w_cpu)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
