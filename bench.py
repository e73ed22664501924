#!/usr/bin/env python
"""Benchmark of the MXFP8 routed-expert hot path on GB300.

One step = one pass of the whole path over one batch of the Llama4-Scout-like
routed-expert workload (G=8 experts, K=5120, N=8192, M=16384 tokens in
Zipf(1.1) groups; synthetic bf16 data, random weights):
    quantize A row+column  -> quantize W plain+transposed -> grouped GEMM fwd
    quantize dOut row+column -> grouped GEMM dgrad -> grouped GEMM wgrad
every call through the C ABI (libmxfp8moe.so).  `value` = algorithmic fwd+bwd
GEMM FLOPs (3 x 2*M*N*K) / step time, with inputs resident in HBM; `e2e` = the
same metric with the inputs copied from pinned host memory and the results
copied back inside every step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Multi-GPU: independent replicas (the path has no exchange step), one process
per GPU under torchrun; the max step time over ranks sets `value`.
--impl reference times the CPU oracle (fp64, plain C) on a bounded sample of
the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP8 grouped-GEMM fwd+bwd TFLOP/s & % MXFP8 peak; quantize GB/s vs HBM"
WORKLOAD = ("Llama4-Scout-like routed experts fwd+bwd: G=8, K=5120, N=8192, M=16384 tokens, "
            "Zipf(1.1) group sizes in 32-token chunks (seed 0)")
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
L2_BYTES = 129 * 2 ** 20

# DRAM traffic of one grouped-GEMM forward launch on this workload, from the
# ncu capture summarised in profiles/grouped_mm_fwd_scout.md, valid only while
# the kernel sources hash to the value recorded with it.
FWD_TRAFFIC = {"bytes": 771875584, "src_sha": "d06a053bdd32ff51"}


WORKLOAD_TEXT = {
    "scout": WORKLOAD,
    "imbalanced": "Fine-grained imbalanced experts fwd+bwd: G=16, K=7168, N=2048, M=32768, group 1 = 13120 tokens, "
                  "groups 0/7/15 empty, 1% x100 activation outliers",
    "swiglu": "SwiGLU routed expert fwd+bwd: G=2, M=65600 (39360/26240), D=5120, H=8192, gate/up W[2,8192,5120], "
              "down W[2,5120,8192]; gate/up GEMMs with the SwiGLU and its MXFP8 quantization fused into the "
              "epilogue, 9 GEMMs, the SwiGLU backward and the quantization of dh1, dh3 in one kernel",
    "swiglu_unfused": "SwiGLU routed expert fwd+bwd as swiglu, with separate gate and up GEMMs, the SwiGLU and "
                      "its backward in torch bf16 and separate ROW|COL quantizations of h, dh1, dh3",
    "swiglu_standin": "SwiGLU routed expert GEMMs: G=2, M=65600 (39360/26240), gate/up W[2,8192,5120], "
                      "down W[2,5120,8192]; 9 grouped GEMMs, seeded stand-ins for the SwiGLU intermediates",
    "tiny": "Tiny: G=2, A[256,256], offs [128,256], W[2,128,256] (latency-bound; parity case)",
    "scout_w32": WORKLOAD + "; expert weights quantized with one scale per 32x32 block (one quantization for "
                            "the forward and the dgrad)",
    "scout_stab": WORKLOAD + "; stability variants: random Hadamard transform of both wgrad operands along the "
                             "tokens, stochastic rounding of the output gradient",
    "scout_mb4": "Llama4-Scout-like routed experts, one optimizer step of 4 microbatches (G=8, K=5120, N=8192, "
                 "M=16384 tokens each, Zipf(1.1) group sizes in 32-token chunks, seeds 0-3): W quantized once "
                 "(prequantized-weight cache), then fwd+bwd per microbatch",
}


def workload_parts(name: str, dev) -> list:
    """The grouped-GEMM problems one step of a workload runs (each: quantize A, W, dOut; fwd, dgrad, wgrad)."""
    from mxfp8_precision_moe_gb300 import synth

    if name in ("scout", "imbalanced", "tiny"):
        return [synth.workload(name, seed=0, device=dev)]
    if name in ("scout_w32", "scout_stab"):
        return [synth.workload("scout", seed=0, device=dev)]
    if name in ("swiglu", "swiglu_unfused"):
        return [synth.workload("swiglu", seed=0, device=dev)]
    if name == "scout_mb4":
        mbs = [synth.workload("scout", seed=i, device=dev) for i in range(4)]
        for w in mbs[1:]:
            w["W"] = mbs[0]["W"]  # one weight tensor for the whole optimizer step
        return mbs
    # swiglu_standin: the expert's 9 GEMMs as three plain problems with seeded intermediates
    s = synth.workload("swiglu", seed=0, device=dev)
    G, M, D, H = s["G"], s["M"], s["D"], s["H"]
    h = synth.randn_bf16((M, H), 1.0, seed=50, device=dev)      # stands in for silu(x Wg^T) * (x Wu^T)
    dh1 = synth.randn_bf16((M, H), 1e-3, seed=51, device=dev)   # stands in for the gate-branch gradient
    dh3 = synth.randn_bf16((M, H), 1e-3, seed=52, device=dev)   # stands in for the up-branch gradient
    common = dict(G=G, M=M, sizes=s["sizes"], offs=s["offs"])
    return [dict(common, N=H, K=D, A=s["x"], W=s["Wg"], dOut=dh1),
            dict(common, N=H, K=D, A=s["x"], W=s["Wu"], dOut=dh3),
            dict(common, N=D, K=H, A=h, W=s["Wd"], dOut=s["dY"])]


def step_inputs(step, parts) -> list:
    """The bf16 input tensors one step reads."""
    if hasattr(step, "x"):
        return [step.x, step.dY, *step.W.values()]
    return [t for p in parts for t in (p["A"], p["W"], p["dOut"])]


def kernel_src_sha() -> str:
    h = hashlib.sha256()
    for f in ("grouped_mm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "mxfp8_precision_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--no-baseline", action="store_true", help="skip the cuBLAS bf16 comparison leg")
    ap.add_argument("--workload", default="scout", choices=["scout", "imbalanced", "swiglu", "swiglu_unfused", "swiglu_standin", "tiny", "scout_mb4", "scout_w32", "scout_stab",
                             "sweep"],
                    help="scout (default, the reported line); the others are extra measurements")
    return ap.parse_args()


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
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        ident = str(device_index)
        try:
            bus = getattr(torch.cuda.get_device_properties(device_index), "pci_bus_id", None)
            if bus:
                ident = bus
        except Exception:
            pass
        cmd = ["nvidia-smi", "-i", ident, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [p for t, p in self.samples if t0 <= t <= t1] or [p for _, p in self.samples[-5:]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[3 + i].lower() == "active"})
        pw = [num(p[2]) for p in win if num(p[2]) is not None]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- the step, through the C ABI
class Step:
    """Device buffers of one replica and the C-ABI calls of one pass of the path."""

    def __init__(self, w: dict, device, shared_w: "Step | None" = None, w_block32: bool = False,
                 stability: bool = False):
        import mxfp8_precision_moe_gb300 as mx

        L = mx.load()
        self.mx, self.L = mx, L
        G, M, N, K = w["G"], w["M"], w["N"], w["K"]
        self.G, self.M, self.N, self.K = G, M, N, K
        u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=device)
        bf = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=device)
        self.A, self.W, self.D = w["A"].to(device), w["W"].to(device), w["dOut"].to(device)
        self.offs = w["offs"].to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        sb = mx.mxfp8_scale_bytes
        sc = mx.mxfp8_scale_bytes_colgroups
        self.aq, self.as_ = u8(M, K), u8(sb(M, K, G, 1))
        self.aTq, self.aTs = u8(K, M), u8(sc(K, M, G))
        ce = lambda r, c: ((r + 127) // 128) * 128 * ((c + 127) // 128) * 4
        if shared_w is None:
            self.wq, self.ws = u8(G, N, K), u8(G, ce(N, K))
            self.wTq, self.wTs = u8(G, K, N), u8(G, ce(K, N))
        else:  # prequantized weights of another microbatch of the same optimizer step
            self.W = shared_w.W
            self.wq, self.ws, self.wTq, self.wTs = shared_w.wq, shared_w.ws, shared_w.wTq, shared_w.wTs
        self.dq, self.ds = u8(M, N), u8(sb(M, N, G, 1))
        self.dTq, self.dTs = u8(N, M), u8(sc(N, M, G))
        self.out, self.dA, self.dW = bf(M, N), bf(M, K), bf(G, N, K)
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        st = P(self.status)
        RC = 3  # MXFP8_ROW | MXFP8_COL
        self.calls = [
            ("quant_A", L.mxfp8_quantize_2d, (P(self.A), M, K, RC, 1, P(self.offs), G, P(self.aq), P(self.as_),
                                              P(self.aTq), P(self.aTs), st)),
            ("quant_W", L.mxfp8_quantize_3d_experts, (P(self.W), G, N, K, RC | (4 if w_block32 else 0), 1,
                                                      P(self.wq), P(self.ws),
                                                      P(self.wTq), P(self.wTs), st)),
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
            # the stability variants: Hadamard transform of both wgrad operands along the tokens (A's and
            # dOut's column-wise copies, one seed), stochastic rounding of both dOut copies
            seed = 0x5EED
            calls = dict((c[0], c) for c in self.calls)
            calls["quant_A"] = ("quant_A", L.mxfp8_quantize_2d_opts,
                                (P(self.A), M, K, RC, 1, P(self.offs), G, 4, seed, P(self.aq), P(self.as_),
                                 P(self.aTq), P(self.aTs), st))
            calls["quant_dOut"] = ("quant_dOut", L.mxfp8_quantize_2d_opts,
                                   (P(self.D), M, N, RC, 1, P(self.offs), G, 1 | 4, seed, P(self.dq), P(self.ds),
                                    P(self.dTq), P(self.dTs), st))
            self.calls = [calls[c[0]] for c in self.calls]
        # kernels each call launches (one each: the quantize kernels also write the blocked padding)
        self.launches = {"quant_A": 1, "quant_W": 1, "fwd": 1, "quant_dOut": 1, "dgrad": 1, "wgrad": 1}
        self.flops = 3 * 2.0 * M * N * K
        self.bytes = {"quant_A": M * K * (2 + 1 + 1 + 2 / 32), "quant_W": G * N * K * (2 + 1 + 1 + 2 / 32),
                      "quant_dOut": M * N * (2 + 1 + 1 + 2 / 32)}
        if shared_w is not None:
            self.calls = [c for c in self.calls if c[0] != "quant_W"]
            del self.launches["quant_W"], self.bytes["quant_W"]
        self.gemm_flops = {"fwd": 2.0 * M * N * K, "dgrad": 2.0 * M * N * K, "wgrad": 2.0 * M * N * K}

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
        self.mx.read_status(self.status, "bench step")


class StepGroup:
    """Several grouped-GEMM problems run back to back as one step (the SwiGLU expert's three)."""

    def __init__(self, parts: list, device, share_w: bool = False):
        self.parts = []
        for w in parts:
            self.parts.append(Step(w, device, self.parts[0] if (share_w and self.parts) else None))
        self.calls, self.gemm_flops, self.bytes, self.launches = [], {}, {}, {}
        for i, st in enumerate(self.parts):
            for name, fn, argv in st.calls:
                key = f"p{i}.{name}"
                self.calls.append((key, fn, argv))
                self.launches[key] = st.launches[name]
                if name in st.gemm_flops:
                    self.gemm_flops[key] = st.gemm_flops[name]
                else:
                    self.bytes[key] = st.bytes[name]
        self.flops = sum(st.flops for st in self.parts)
        p0 = self.parts[0]
        self.G, self.M, self.N, self.K, self.mx = p0.G, p0.M, p0.N, p0.K, p0.mx

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
        for st in self.parts:
            st.check_status()


def swiglu_backward_bf16(dh: torch.Tensor, h1: torch.Tensor, h3: torch.Tensor):
    """(dh1, dh3) of h = silu(h1) * h3 with torch's bf16 autograd ops (the unfused comparison route)."""
    dh3 = dh * torch.nn.functional.silu(h1)
    dh1 = torch.ops.aten.silu_backward(dh * h3, h1)
    return dh1, dh3


class SwiGLUStep:
    """One fwd+bwd of the SwiGLU routed expert y = (silu(x Wg^T) * (x Wu^T)) Wd^T through the C ABI.

    fused:   the gate/up GEMMs write h1, h3 and h already quantized both ways (one kernel); in the
             backward one kernel computes dh1, dh3 and quantizes both both ways, and one GEMM gives
             dx = dh1 Wg + dh3 Wu;
    unfused: two forward GEMMs, h = silu(h1) * h3 in torch bf16, a ROW|COL quantization of h; in the
             backward the SwiGLU backward in torch bf16 ops and two ROW|COL quantizations.
    Both run the down GEMM, and in the backward: dY quantized both ways, down dgrad and wgrad, two
    dgrads (summed) and two wgrads.  Entries whose name starts with "torch." are torch elementwise
    glue, not library kernels."""

    def __init__(self, s: dict, device, fused: bool):
        import mxfp8_precision_moe_gb300 as mx

        L = mx.load()
        self.mx, self.L = mx, L
        G, M, D, H = s["G"], s["M"], s["D"], s["H"]
        self.G, self.M, self.N, self.K = G, M, H, D
        u8 = lambda *sh: torch.empty(sh, dtype=torch.uint8, device=device)
        bf = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        sb, sc = mx.mxfp8_scale_bytes, mx.mxfp8_scale_bytes_colgroups
        ce = lambda r, c: ((r + 127) // 128) * 128 * ((c + 127) // 128) * 4
        self.x, self.dY, self.offs = s["x"].to(device), s["dY"].to(device), s["offs"].to(device)
        self.W = {n: s[n].to(device) for n in ("Wg", "Wu", "Wd")}
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        st = P(self.status)
        RC = 3
        tok = lambda cols: (u8(M, cols), u8(sb(M, cols, G, 1)), u8(cols, M), u8(sc(cols, M, G)))
        xq = tok(D)
        wq = {}
        for n, (r, c) in (("Wg", (H, D)), ("Wu", (H, D)), ("Wd", (D, H))):
            wq[n] = (u8(G, r, c), u8(G, ce(r, c)), u8(G, c, r), u8(G, ce(c, r)))
        h1, h3 = bf(M, H), bf(M, H)
        hq = tok(H)
        dYq = tok(D)
        dh, dh1, dh3 = bf(M, H), bf(M, H), bf(M, H)
        a1, a3 = tok(H), tok(H)
        y, dx, dx2 = bf(M, D), bf(M, D), bf(M, D)
        dWg, dWu, dWd = bf(G, H, D), bf(G, H, D), bf(G, D, H)
        self.keep = [xq, wq, h1, h3, hq, dYq, dh, dh1, dh3, a1, a3, y, dx, dx2, dWg, dWu, dWd]
        offs, x, dY = P(self.offs), P(self.x), P(self.dY)
        q = lambda t4: tuple(P(t) for t in t4)

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
        for n, (r, c) in (("Wg", (H, D)), ("Wu", (H, D)), ("Wd", (D, H))):
            calls.append((f"quant_{n}", L.mxfp8_quantize_3d_experts, (P(self.W[n]), G, r, c, RC, 1, *q(wq[n]), st)))
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
        else:
            calls += [("torch.swiglu_bwd", glue(swiglu_bwd_torch), ()),
                      ("quant_dh1", L.mxfp8_quantize_2d, (P(dh1), M, H, RC, 1, offs, G, *q(a1), st)),
                      ("quant_dh3", L.mxfp8_quantize_2d, (P(dh3), M, H, RC, 1, offs, G, *q(a3), st))]
        if fused:
            calls.append(("dgrad_gate_up", L.mxfp8_grouped_mm_dgrad2,
                          (*q(a1)[:2], *q(wq["Wg"])[2:], *q(a3)[:2], *q(wq["Wu"])[2:], offs, G, M, H, D, P(dx), st)))
        else:
            calls += [
                ("dgrad_gate", L.mxfp8_grouped_mm_dgrad, (*q(a1)[:2], *q(wq["Wg"])[2:], offs, G, M, H, D, P(dx), st)),
                ("dgrad_up", L.mxfp8_grouped_mm_dgrad, (*q(a3)[:2], *q(wq["Wu"])[2:], offs, G, M, H, D, P(dx2), st)),
                ("torch.add", glue(lambda: dx.add_(dx2)), ())]
        calls += [
            ("wgrad_gate", L.mxfp8_grouped_mm_wgrad, (*q(a1)[2:], *q(xq)[2:], offs, G, M, H, D, P(dWg), st)),
            ("wgrad_up", L.mxfp8_grouped_mm_wgrad, (*q(a3)[2:], *q(xq)[2:], offs, G, M, H, D, P(dWu), st)),
        ]
        self.calls = calls
        self.launches = {n: (0 if n.startswith("torch.") else 1) for n, _, _ in calls}
        f1 = 2.0 * M * D * H
        self.gemm_flops = {n: (2 * f1 if n in ("gateup_swiglu", "dgrad_gate_up") else f1) for n, _, _ in calls
                           if n.startswith(("fwd_", "dgrad_", "wgrad_", "gateup"))}
        self.flops = 9 * f1
        qb = lambda e: e * (2 + 1 + 1 + 2 / 32)
        self.bytes = {"quant_x": qb(M * D), "quant_Wg": qb(G * H * D), "quant_Wu": qb(G * H * D),
                      "quant_Wd": qb(G * D * H), "quant_dY": qb(M * D)}
        if fused:
            # reads dh, h1, h3; writes dh1 and dh3 codes both ways with their scales
            self.bytes["swiglu_bwd_quant"] = M * H * (6 + 2 * (2 + 2 / 32))
        else:
            self.bytes.update(quant_h=qb(M * H), quant_dh1=qb(M * H), quant_dh3=qb(M * H))
        self.roofline_key = "gateup_swiglu" if fused else "fwd_gate"
        self.roofline_name = "grouped_mm_swiglu_fwd (gate+up, fused epilogue)" if fused else "grouped_mm_fwd (gate)"

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
        self.mx.read_status(self.status, "bench SwiGLU step")


# ---------------------------------------------------------------- oracle sample (CPU baseline / reference arm)
def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class OracleProbe:
    """Sampled outputs of the three GEMMs computed by the CPU oracle from the bf16
    inputs (quantization included): one probe = one element of out, one of dA
    and one of dW.  Algorithmic FLOPs of a probe: 2*(K + N + M_g)."""

    def __init__(self, w_cpu: dict, seed: int = 0):
        import oracle

        oracle.lib()
        self.o = oracle
        self.w = w_cpu
        self.ends = np.cumsum(w_cpu["sizes"])
        self.starts = self.ends - np.asarray(w_cpu["sizes"])
        self.nonempty = [g for g, s in enumerate(w_cpu["sizes"]) if s > 0]
        self.rng = np.random.default_rng(seed)

    def probe(self) -> float:
        o, w, rng = self.o, self.w, self.rng
        M, N, K = w["M"], w["N"], w["K"]
        m = int(rng.integers(0, M))
        g = int(np.searchsorted(self.ends, m, side="right"))
        n, k = int(rng.integers(0, N)), int(rng.integers(0, K))
        qa, sa = o.quantize_vec(_bits(w["A"][m]))
        qw, sw = o.quantize_vec(_bits(w["W"][g, n]))
        o.dot(qa, sa, qw, sw)                                   # out[m, n]
        qd, sd = o.quantize_vec(_bits(w["dOut"][m]))
        qt, st = o.quantize_vec(_bits(w["W"][g, :, k]))
        o.dot(qd, sd, qt, st)                                   # dA[m, k]
        gg = self.nonempty[int(rng.integers(0, len(self.nonempty)))]
        lo, hi = int(self.starts[gg]), int(self.ends[gg])
        q1, s1 = o.quantize_vec(_bits(w["dOut"][lo:hi, n]))
        q2, s2 = o.quantize_vec(_bits(w["A"][lo:hi, k]))
        o.dot(q1, s1, q2, s2)                                   # dW[gg][n, k]
        return 2.0 * (K + N + (hi - lo))


def oracle_rate(w_cpu: dict, seconds: float, seed: int = 0):
    """Run probes for about `seconds`; return (TFLOP/s, probes, elapsed)."""
    pr = OracleProbe(w_cpu, seed)
    flops, n, t0 = 0.0, 0, time.perf_counter()
    while True:
        flops += pr.probe()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return flops / el / 1e12, n, el


def cpu_cores_used() -> int:
    return 1  # the probes call the oracle's single-threaded scalar routines


# ---------------------------------------------------------------- native (GPU) arm
def run_native(args, rank, world, local):
    from mxfp8_precision_moe_gb300 import synth

    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    parts = workload_parts(args.workload, dev)
    w = parts[0]
    if args.workload in ("swiglu", "swiglu_unfused"):
        step = SwiGLUStep(w, dev, fused=args.workload == "swiglu")
    elif len(parts) == 1:
        step = Step(w, dev, w_block32=args.workload == "scout_w32", stability=args.workload == "scout_stab")
    else:
        step = StepGroup(parts, dev, share_w=args.workload == "scout_mb4")
    single = isinstance(step, Step)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        step.run(stream)
    torch.cuda.synchronize()
    step.check_status()

    names = [c[0] for c in step.calls]
    ev = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for n in names}
          for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    time.sleep(0.3)  # let the sampler start
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step.run(stream, ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall1 = time.time()
    sampler.stop()
    step.check_status()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    per = {n: float(np.mean([e[n][0].elapsed_time(e[n][1]) for e in ev])) for n in names}
    clocks = sampler.summary(wall0, wall1)

    # bf16 baseline: per-group cuBLAS torch.mm loop for the forward (same bf16 inputs)
    base = None
    if rank == 0 and not args.no_baseline and single:
        ends = np.cumsum(w["sizes"])
        out_b = torch.empty_like(step.out)

        def bf16_fwd():
            lo = 0
            for g, hi in enumerate(ends):
                if hi > lo:
                    torch.mm(step.A[lo:hi], step.W[g].t(), out=out_b[lo:hi])
                lo = int(hi)

        for _ in range(3):
            bf16_fwd()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(20):
            bf16_fwd()
        b1.record(stream)
        torch.cuda.synchronize()
        bms = b0.elapsed_time(b1) / 20
        base = {"kernel": "cuBLAS bf16 per-group torch.mm loop, forward", "ms": round(bms, 4),
                "tflops": round(step.gemm_flops["fwd"] / bms / 1e9, 1)}

    # end to end: host (pinned) inputs copied in and results copied out inside every step, as a
    # 3-stream pipeline over two device buffer sets: the copy-in of step i+1 and the copy-out of
    # step i-1 overlap the kernels of step i (events order each buffer set's reuse)
    e2e = None
    if not args.no_e2e and single:
        sets = [step, Step(w, dev)]
        hA, hW, hD = (t.cpu().pin_memory() for t in (step.A, step.W, step.D))
        hoffs = step.offs.cpu().pin_memory()
        hout = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (st.out, st.dA, st.dW))
                for st in sets]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        n_e2e = max(4, min(20, args.steps // 10))
        mk = lambda: torch.cuda.Event(enable_timing=False)
        h2d_done = [mk() for _ in range(n_e2e)]
        comp_done = [mk() for _ in range(n_e2e)]
        d2h_done = [mk() for _ in range(n_e2e)]
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(s_in)
        for i in range(n_e2e):
            st = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])       # inputs of set i%2 no longer read
                st.A.copy_(hA, non_blocking=True)
                st.W.copy_(hW, non_blocking=True)
                st.D.copy_(hD, non_blocking=True)
                st.offs.copy_(hoffs, non_blocking=True)
                h2d_done[i].record(s_in)
            stream.wait_event(h2d_done[i])
            if i >= 2:
                stream.wait_event(d2h_done[i - 2])           # outputs of set i%2 already copied out
            st.run(stream)
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                for h, d in zip(hout[i % 2], (st.out, st.dA, st.dW)):
                    h.copy_(d, non_blocking=True)
                d2h_done[i].record(s_out)
        s_out.wait_event(d2h_done[n_e2e - 1])
        x1.record(s_out)
        torch.cuda.synchronize()
        for st in sets:
            st.check_status()
        xms = max_over_ranks(x0.elapsed_time(x1) / n_e2e, world, dev)
        bi = sum(t.numel() * t.element_size() for t in (hA, hW, hD, hoffs))
        bo = sum(t.numel() * t.element_size() for t in hout[0])
        e2e = {"value": round(world * step.flops / xms / 1e9, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": round(xms, 3), "steps": n_e2e,
               "pipeline": "copy-in, kernels and copy-out on 3 streams over 2 device buffer sets"}

    if rank != 0:
        return None
    ms_step = ms / args.steps
    fp8_peak = pk["bf16_sus"] * FP8_OVER_BF16
    fwd_key = getattr(step, "roofline_key", "fwd" if single else "p0.fwd")
    fwd_ms = per[fwd_key]
    achieved = step.gemm_flops[fwd_key] / fwd_ms / 1e9
    traffic = FWD_TRAFFIC["bytes"] if (FWD_TRAFFIC["src_sha"] == kernel_src_sha() and args.workload == "scout") else None
    kernels = {}
    for n in names:
        d = {"ms": round(per[n], 4)}
        if n in step.gemm_flops:
            tf = step.gemm_flops[n] / per[n] / 1e9
            d.update(tflops=round(tf, 1), frac_fp8_peak=round(tf / fp8_peak, 3))
        elif n in step.bytes:
            gbs = step.bytes[n] / per[n] / 1e6
            d.update(gbs=round(gbs, 1), frac_hbm=round(gbs / pk["hbm"], 3))
        kernels[n] = d  # entries named torch.* are torch elementwise glue: time only
    line = {
        "metric": METRIC,
        "value": round(world * step.flops / ms_step / 1e9, 2),
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
        "config": {"workload": WORKLOAD_TEXT[args.workload], "G": step.G, "M": step.M, "N": step.N, "K": step.K,
                   "group_sizes": list(map(int, w["sizes"])), "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({L2_BYTES // 2**20} MiB): A, W, dOut = "
                         f"{sum(t.numel() * 2 for t in {id(t): t for t in step_inputs(step, parts)}.values()) // 2**20} "
                         "MiB bf16 per step" if args.workload != "tiny" else "tiny: L2-resident (latency-bound case)",
                   "frac_fp8_peak_step": round(step.flops / ms_step / 1e9 / fp8_peak, 3)},
        "roofline": {"bound": "tensor", "kernel": getattr(step, "roofline_name", "grouped_mm_fwd" + ("" if single else " (gate)")),
                     "achieved": round(achieved, 1),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 3),
                     "traffic": traffic,
                     "peak_note": f"{pk['src']} sustained bf16 {pk['bf16_sus']} TFLOP/s x {FP8_OVER_BF16} "
                                  "(nominal dense fp8/bf16 ratio)"},
        "kernels": kernels,
        "hbm_peak_gbs": pk["hbm"],
        "baseline_bf16": base,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(step.launches.values()),
    }
    return line, w


def main():
    args = parse_args()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload == "sweep":
        if rank == 0:
            print(json.dumps(run_sweep(args)), flush=True)
        return
    res = run_native(args, rank, world, local)
    if rank == 0 and res is not None:
        line, w = res
        if not args.no_cpu and world == 1 and args.workload == "scout":
            w_cpu = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in w.items()}
            rate, n, el = oracle_rate(w_cpu, 15.0)
            line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
                                    "sample": f"{n} probes (one element each of out, dA, dW, quantization "
                                              f"included) in {el:.1f} s"}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_sweep(args) -> dict:
    """Quantization bandwidth over the sweep shapes: bf16 [M,K] row, column, row+column (one read) and
    32x32 blocks, plus 3D expert weights [16,8192,5120] plain, transposed and both; GB/s of
    algorithmic bytes (2 read + per direction 1 code + 1/32 scale byte per element)."""
    import mxfp8_precision_moe_gb300 as mx
    from mxfp8_precision_moe_gb300 import synth

    L = mx.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    stream = torch.cuda.current_stream(dev)
    sp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rows = []
    sampler = ClockSampler(dev.index)
    time.sleep(0.3)
    wall0 = time.time()

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

    for M in synth.SWEEP_M:
        for K in synth.SWEEP_K:
            x = synth.log_uniform_rows(M, K, seed=M + K, device=dev)
            u8 = lambda *shape: torch.empty(shape, dtype=torch.uint8, device=dev)
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
    u8 = lambda *shape: torch.empty(shape, dtype=torch.uint8, device=dev)
    q, qT = u8(M, K), u8(K, M)
    s_r, s_c = u8(mx.mxfp8_scale_bytes(M, K, 1, 1)), u8(mx.mxfp8_scale_bytes_colgroups(K, M, 1))
    for label, opts in (("row+col SR", 1), ("row+col RHT(col)", 4), ("row+col RHT(row,col)", 6),
                        ("row+col SR+RHT(col)", 5)):
        time_call(L.mxfp8_quantize_2d_opts, (sp(x), M, K, 3, 1, None, 0, opts, 0x5EED, sp(q), sp(s_r), sp(qT), sp(s_c),
                                             None), M * K * (2 + 2 + 2 / 32), label, [M, K])
    del x, q, qT, s_r, s_c
    G, N, K = 16, 8192, 5120
    w = synth.randn_bf16((G, N, K), 1.0, seed=7, device=dev)
    ce = lambda r, c: ((r + 127) // 128) * 128 * ((c + 127) // 128) * 4
    q, s3 = torch.empty((G, N, K), dtype=torch.uint8, device=dev), torch.empty((G, ce(N, K)), dtype=torch.uint8, device=dev)
    qT, sT = torch.empty((G, K, N), dtype=torch.uint8, device=dev), torch.empty((G, ce(K, N)), dtype=torch.uint8, device=dev)
    E = G * N * K
    for label, dirs, out in (("3d plain", 1, (q, s3, None, None)), ("3d transposed", 2, (None, None, qT, sT)),
                             ("3d both", 3, (q, s3, qT, sT)), ("3d 32x32 both", 7, (q, s3, qT, sT))):
        nb = E * (2 + 2 + 2 / 32) if dirs & 3 == 3 else E * (2 + 1 + 1 / 32)
        time_call(L.mxfp8_quantize_3d_experts, (sp(w), G, N, K, dirs, 1, *[sp(t) for t in out], None), nb, label,
                  [G, N, K])
    wall1 = time.time()
    sampler.stop()
    best = max(r["frac_hbm"] for r in rows)
    return {"metric": "MXFP8 quantize GB/s (sweep)", "unit": "GB/s", "hbm_peak_gbs": pk["hbm"],
            "clocks": sampler.summary(wall0, wall1),
            "peak_note": f"{pk['src']} copy bandwidth", "data": "synthetic",
            "config": {"workload": "quantization sweep: [M,K] M in 8192..131072, K in {5120, 8192}; "
                                   "3D [16,8192,5120]; N(0,1)*10^U(-4,4) per row"},
            "best_frac_hbm": best, "sweep": rows}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the machine's host cores (rank 0 only)."""
    if rank != 0:
        return
    from mxfp8_precision_moe_gb300 import synth

    w = synth.workload("scout", seed=0, device="cpu")
    pr = OracleProbe(w, seed=1)
    t0 = time.perf_counter()
    pr.probe()
    t_probe = time.perf_counter() - t0
    per_step = max(1, int(90.0 / ((args.steps + args.warmup) * max(t_probe, 1e-3))))
    for _ in range(args.warmup):
        for _ in range(per_step):
            pr.probe()
    flops, t0 = 0.0, time.perf_counter()
    for _ in range(args.steps):
        for _ in range(per_step):
            flops += pr.probe()
    el = time.perf_counter() - t0
    val = flops / el / 1e12
    sample = f"{per_step} probe(s) per step (one element each of out, dA, dW from the bf16 inputs)"
    line = {
        "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cpu_cores_used(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
