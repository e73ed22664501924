"""The SwiGLU routed expert as three chained MXFP8 grouped GEMMs (gate, up, down) with the
elementwise SwiGLU in torch, forward and backward, against the same chain computed by the
oracle (its own quantization, fp64 GEMMs, the glue in fp64 with bf16 rounding of every
intermediate).  No GPU value feeds the oracle.

Tolerance: the per-GEMM bound 1e-2|o| + 1e-3 rms(o) holds for every single GEMM
(test_gpu_grouped_mm.py).  Chained, the bf16 intermediates of the GPU (torch CUDA glue) and of
the oracle (fp64 rounded to bf16) can differ by one bf16 ulp, which can move an element
across an E4M3 rounding boundary in the next quantization (one E4M3 ulp = 1/8 relative).  The
chain therefore asserts a relative Frobenius error below 2e-2 and the elementwise bound with
5x the per-GEMM coefficients on 99.9% of the elements.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._util import f64, require_gpu, sizes_to_ends, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def bf16_round(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def o_fwd(A, W, sizes):
    aq, as_ = oracle.quantize_rows(u16(A))
    wq, ws = zip(*[oracle.quantize_rows(u16(W[g])) for g in range(W.shape[0])])
    return oracle.grouped_mm_rows(aq, as_, np.stack(wq), np.stack(ws), sizes_to_ends(sizes))


def o_dgrad(D, W, sizes):
    dq, ds = oracle.quantize_rows(u16(D))
    wTq, wTs = zip(*[oracle.quantize_cols(u16(W[g])) for g in range(W.shape[0])])
    return oracle.grouped_mm_rows(dq, ds, np.stack(wTq), np.stack(wTs), sizes_to_ends(sizes))


def o_wgrad(D, A, sizes):
    dTq, dTs = oracle.quantize_cols(u16(D))
    aTq, aTs = oracle.quantize_cols(u16(A))
    return oracle.grouped_mm_wgrad(dTq, dTs, aTq, aTs, sizes_to_ends(sizes))


def chain_close(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel < 2e-2, f"{what}: relative Frobenius error {rel:.3g}"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    ok = np.abs(got - ref) <= 5e-2 * np.abs(ref) + 5e-3 * rms
    assert ok.mean() >= 0.999, f"{what}: {int((~ok).sum())}/{ok.size} elements outside the chain bound"


def test_swiglu_expert_chain_fwd_bwd(mx):
    sizes = [384, 256]
    G, M, D, H = 2, sum(sizes), 256, 512
    x = synth.randn_bf16((M, D), 1.0, seed=61)
    Wg = synth.randn_bf16((G, H, D), 0.05, seed=62)
    Wu = synth.randn_bf16((G, H, D), 0.05, seed=63)
    Wd = synth.randn_bf16((G, D, H), 0.05, seed=64)
    dY = synth.randn_bf16((M, D), 1e-2, seed=65)
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")

    # ---- GPU: three differentiable MXFP8 grouped GEMMs, SwiGLU glue in torch (bf16)
    xg = x.cuda().requires_grad_(True)
    Wgg, Wug, Wdg = (t.cuda().requires_grad_(True) for t in (Wg, Wu, Wd))
    h1 = mx.to_mxfp8_then_scaled_grouped_mm(xg, Wgg, offs)
    h3 = mx.to_mxfp8_then_scaled_grouped_mm(xg, Wug, offs)
    h = torch.nn.functional.silu(h1) * h3
    y = mx.to_mxfp8_then_scaled_grouped_mm(h, Wdg, offs)
    y.backward(dY.cuda())
    torch.cuda.synchronize()

    # ---- oracle chain: fp64 GEMMs; the glue in fp64 with a bf16 rounding after each elementwise
    # op, the same places the bf16 torch glue rounds (silu(h1) and the product; in the backward
    # dh*silu(h1), dh*h3 and the silu derivative product)
    o_h1 = bf16_round(o_fwd(x, Wg, sizes))
    o_h3 = bf16_round(o_fwd(x, Wu, sizes))
    h1d, h3d = o_h1.double().numpy(), o_h3.double().numpy()
    sig = 1.0 / (1.0 + np.exp(-h1d))
    silu = bf16_round(h1d * sig).double().numpy()
    o_h = bf16_round(silu * h3d)
    o_y = o_fwd(o_h, Wd, sizes)
    # backward: dh = dY Wd (dgrad); dWd = dY^T h (wgrad); then the SwiGLU backward
    o_dh = bf16_round(o_dgrad(dY, Wd, sizes))
    o_dWd = o_wgrad(dY, o_h, sizes)
    dhd = o_dh.double().numpy()
    d_h3 = bf16_round(dhd * silu)                                          # d/dh3 of silu(h1) * h3
    d_silu = bf16_round(dhd * h3d).double().numpy()
    d_h1 = bf16_round(d_silu * sig * (1.0 + h1d * (1.0 - sig)))            # silu derivative
    o_dx = o_dgrad(d_h1, Wg, sizes) + o_dgrad(d_h3, Wu, sizes)
    o_dWg = o_wgrad(d_h1, x, sizes)
    o_dWu = o_wgrad(d_h3, x, sizes)

    chain_close(f64(y), o_y, "y")
    chain_close(f64(Wdg.grad), o_dWd, "dW_down")
    chain_close(f64(Wgg.grad), o_dWg, "dW_gate")
    chain_close(f64(Wug.grad), o_dWu, "dW_up")
    chain_close(f64(xg.grad), o_dx, "dx")
