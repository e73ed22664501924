"""The SwiGLU routed expert as three chained MXFP8 grouped GEMMs (gate, up, down) with the
elementwise SwiGLU in torch, forward and backward, against the same chain computed by the
oracle (its own quantization, fp64 GEMMs, the glue in fp64 with bf16 rounding of every
intermediate); and the fused expert (mxfp8_swiglu_expert: gate/up GEMMs with the SwiGLU and
its quantization in the epilogue) against the same oracle chain.  No GPU value feeds the oracle.

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
from tests._util import assert_gemm_close, f64, require_gpu, sizes_to_ends, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def bf16_round(a: np.ndarray) -> torch.Tensor:
    """bf16 round-to-nearest-even of fp64 values, one rounding (the oracle's pinned routine)."""
    b = oracle.bf16_from_f64(np.ascontiguousarray(a, np.float64))
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)


def as_bf16(b: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16) as a bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


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


SIZES = [384, 256]
G, D, H = 2, 256, 512
M = sum(SIZES)


def inputs():
    x = synth.randn_bf16((M, D), 1.0, seed=61)
    Wg = synth.randn_bf16((G, H, D), 0.05, seed=62)
    Wu = synth.randn_bf16((G, H, D), 0.05, seed=63)
    Wd = synth.randn_bf16((G, D, H), 0.05, seed=64)
    dY = synth.randn_bf16((M, D), 1e-2, seed=65)
    return x, Wg, Wu, Wd, dY


def oracle_chain(x, Wg, Wu, Wd, dY, sizes):
    """The expert on the oracle: fp64 GEMMs of oracle-quantized operands, each rounded once to
    bf16, and the oracle's SwiGLU stages (swiglu_bf16 and swiglu_bwd_bf16: fp64 with a bf16
    rounding after each elementwise op, pinned in test_oracle_swiglu.py)."""
    o_h1 = bf16_round(o_fwd(x, Wg, sizes))
    o_h3 = bf16_round(o_fwd(x, Wu, sizes))
    o_h = as_bf16(oracle.swiglu_bf16(u16(o_h1), u16(o_h3)))               # the oracle's pinned SwiGLU stage
    o = dict(y=o_fwd(o_h, Wd, sizes))
    # backward: dh = dY Wd (dgrad); dWd = dY^T h (wgrad); then the oracle's SwiGLU backward stage
    o_dh = bf16_round(o_dgrad(dY, Wd, sizes))
    o["dWd"] = o_wgrad(dY, o_h, sizes)
    d_h1, d_h3 = (as_bf16(t) for t in oracle.swiglu_bwd_bf16(u16(o_dh), u16(o_h1), u16(o_h3)))
    o["dx"] = o_dgrad(d_h1, Wg, sizes) + o_dgrad(d_h3, Wu, sizes)
    o["dWg"] = o_wgrad(d_h1, x, sizes)
    o["dWu"] = o_wgrad(d_h3, x, sizes)
    return o


def gpu_leaves(x, Wg, Wu, Wd):
    return [t.cuda().requires_grad_(True) for t in (x, Wg, Wu, Wd)]


def offs_dev():
    return torch.tensor(sizes_to_ends(SIZES).astype(np.int32), device="cuda")


def check_chain(o, y, xg, Wgg, Wug, Wdg):
    chain_close(f64(y), o["y"], "y")
    chain_close(f64(Wdg.grad), o["dWd"], "dW_down")
    chain_close(f64(Wgg.grad), o["dWg"], "dW_gate")
    chain_close(f64(Wug.grad), o["dWu"], "dW_up")
    chain_close(f64(xg.grad), o["dx"], "dx")


def test_swiglu_expert_chain_fwd_bwd(mx):
    """Three differentiable MXFP8 grouped GEMMs with the SwiGLU glue in torch (bf16)."""
    x, Wg, Wu, Wd, dY = inputs()
    offs = offs_dev()
    xg, Wgg, Wug, Wdg = gpu_leaves(x, Wg, Wu, Wd)
    h1 = mx.to_mxfp8_then_scaled_grouped_mm(xg, Wgg, offs)
    h3 = mx.to_mxfp8_then_scaled_grouped_mm(xg, Wug, offs)
    h = torch.nn.functional.silu(h1) * h3
    y = mx.to_mxfp8_then_scaled_grouped_mm(h, Wdg, offs)
    y.backward(dY.cuda())
    torch.cuda.synchronize()
    check_chain(oracle_chain(x, Wg, Wu, Wd, dY, SIZES), y, xg, Wgg, Wug, Wdg)


def test_fused_swiglu_expert_fwd_bwd(mx):
    """The fused expert (gate/up GEMMs with SwiGLU + quantization in the epilogue, down GEMM
    on the fused kernel's codes, fused SwiGLU backward, one dgrad for dx) against the same oracle
    chain, and against the unfused chain on the GPU."""
    x, Wg, Wu, Wd, dY = inputs()
    offs = offs_dev()
    xg, Wgg, Wug, Wdg = gpu_leaves(x, Wg, Wu, Wd)
    y = mx.mxfp8_swiglu_expert(xg, Wgg, Wug, Wdg, offs)
    y.backward(dY.cuda())
    torch.cuda.synchronize()
    check_chain(oracle_chain(x, Wg, Wu, Wd, dY, SIZES), y, xg, Wgg, Wug, Wdg)

    ug = gpu_leaves(x, Wg, Wu, Wd)
    h = torch.nn.functional.silu(mx.to_mxfp8_then_scaled_grouped_mm(ug[0], ug[1], offs)) * \
        mx.to_mxfp8_then_scaled_grouped_mm(ug[0], ug[2], offs)
    yu = mx.to_mxfp8_then_scaled_grouped_mm(h, ug[3], offs)
    yu.backward(dY.cuda())
    torch.cuda.synchronize()
    for a, b, what in ((y, yu, "y"), (Wgg.grad, ug[1].grad, "dWg"), (Wug.grad, ug[2].grad, "dWu"),
                       (Wdg.grad, ug[3].grad, "dWd")):
        assert_gemm_close(f64(a), f64(b), what=f"fused vs unfused {what}")
    # dx: the fused route sums dh1 Wg + dh3 Wu in one accumulator, the unfused one rounds each
    # product to bf16 before adding, which is off by more than one GEMM's bound where they cancel
    chain_close(f64(xg.grad), f64(ug[0].grad), "fused vs unfused dx")


def test_fused_swiglu_expert_prequantized_weights(mx):
    """Weights through an Mxfp8WeightCache give bit-identical results to on-the-fly quantization."""
    x, Wg, Wu, Wd, dY = inputs()
    offs = offs_dev()
    outs = []
    cache = mx.Mxfp8WeightCache()
    leaves_w = gpu_leaves(x, Wg, Wu, Wd)[1:]
    for kw in ({}, {"weight_cache": cache}, {"weight_cache": cache}):
        xg = x.cuda().requires_grad_(True)
        for w in leaves_w:
            w.grad = None
        y = mx.mxfp8_swiglu_expert(xg, *leaves_w, offs, **kw)
        y.backward(dY.cuda())
        torch.cuda.synchronize()
        outs.append([y.detach().clone(), xg.grad.clone()] + [w.grad.clone() for w in leaves_w])
    assert cache.misses == 3 and cache.hits == 3
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(outs[1], outs[2]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
