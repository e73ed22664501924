"""SwiGLU routed expert on the MXFP8 path, with the SwiGLU and its quantization fused
into the gate/up GEMM epilogue.

"feat(moe): add MoK MXFP8 expert support" names the expert's gate, up and down
weights and their MXFP8 quadruples; "MXFP8 (Micro-scaling FP8)", "Neutralizing
quantization overhead" fuses an activation's quantization into the kernel that
produces it.  Per group g of tokens:

    h1 = x Wg[g]^T,  h3 = x Wu[g]^T,  h = silu(h1) * h3,  y = h Wd[g]^T

Forward: x is quantized along D (and along the tokens for the wgrads); one fused
kernel runs both gate and up GEMMs and writes h1, h3 (bf16, kept for the backward)
and h already quantized along H (for the down GEMM) and along the tokens (for the
down wgrad); the down GEMM reads those codes directly.  Backward: dY is quantized
both ways; dgrad and wgrad of the down GEMM; one kernel computes the SwiGLU backward
(dh1, dh3 at the rounding points of the bf16 autograd ops for ``silu(h1) * h3``) and
quantizes both results both ways; one GEMM for dx = dh1 Wg + dh3 Wu; the wgrads of
gate and up.  Quantization is the identity for gradients.
"""
from __future__ import annotations

import torch

from . import (COL, ROW, SCALES_BLOCKED, _check_quad, _offsets, mxfp8_check_offsets, mxfp8_grouped_mm_dgrad,
               mxfp8_grouped_mm_dgrad2, mxfp8_grouped_mm_fwd, mxfp8_grouped_mm_swiglu_fwd, mxfp8_grouped_mm_wgrad,
               mxfp8_quantize_2d, mxfp8_swiglu_bwd_quantize, new_status, quantize_expert_weights, read_status)


class _Mxfp8SwiGLUExpert(torch.autograd.Function):

    @staticmethod
    def forward(ctx, x, Wg, Wu, Wd, offs, qg, qu, qd, check_offsets):
        need_dx = ctx.needs_input_grad[0]
        need_dw = any(ctx.needs_input_grad[1:4])
        st = None
        if check_offsets:
            # the token-wise copies of the wgrads need group sizes that are multiples of 32
            st = new_status(x.device)
            mxfp8_check_offsets(offs, x.shape[0], 32 if need_dw else 1, st)
        xq, xs, xTq, xTs = mxfp8_quantize_2d(x.contiguous(), ROW | (COL if need_dw else 0), SCALES_BLOCKED, offs,
                                             st)
        qg = _check_quad(qg, Wg, need_dx) if qg is not None else quantize_expert_weights(Wg)
        qu = _check_quad(qu, Wu, need_dx) if qu is not None else quantize_expert_weights(Wu)
        qd = _check_quad(qd, Wd, True) if qd is not None else quantize_expert_weights(Wd)
        h1, h3, hq, hs, hTq, hTs = mxfp8_grouped_mm_swiglu_fwd(xq, xs, qg[0], qg[1], qu[0], qu[1], offs,
                                                               token_wise=ctx.needs_input_grad[3], dev_status=st)
        y = mxfp8_grouped_mm_fwd(hq, hs, qd[0], qd[1], offs, dev_status=st)
        if st is not None:
            read_status(st, "mxfp8_swiglu_expert (group offsets)")
        ctx.save_for_backward(xTq, xTs, h1, h3, hTq, hTs, qg[2], qg[3], qu[2], qu[3], qd[2], qd[3], offs)
        return y

    @staticmethod
    def backward(ctx, dY):
        xTq, xTs, h1, h3, hTq, hTs, gTq, gTs, uTq, uTs, dTq, dTs, offs = ctx.saved_tensors
        need_dx, need_dWg, need_dWu, need_dWd = ctx.needs_input_grad[:4]
        need_front = need_dx or need_dWg or need_dWu
        dirs = (ROW if need_front else 0) | (COL if need_dWd else 0)
        dq, ds, dTq_, dTs_ = mxfp8_quantize_2d(dY.contiguous().to(torch.bfloat16), dirs, SCALES_BLOCKED, offs)
        dWd = mxfp8_grouped_mm_wgrad(dTq_, dTs_, hTq, hTs, offs) if need_dWd else None
        dx = dWg = dWu = None
        if need_front:
            dh = mxfp8_grouped_mm_dgrad(dq, ds, dTq, dTs, offs)
            # the SwiGLU backward and the quantization of dh1, dh3 (both ways) in one kernel
            (a1q, a1s, a1Tq, a1Ts), (a3q, a3s, a3Tq, a3Ts) = mxfp8_swiglu_bwd_quantize(dh, h1, h3, offs)
            if need_dx:  # dx = dh1 Wg + dh3 Wu, one GEMM over both
                dx = mxfp8_grouped_mm_dgrad2(a1q, a1s, gTq, gTs, a3q, a3s, uTq, uTs, offs)
            if need_dWg:
                dWg = mxfp8_grouped_mm_wgrad(a1Tq, a1Ts, xTq, xTs, offs)
            if need_dWu:
                dWu = mxfp8_grouped_mm_wgrad(a3Tq, a3Ts, xTq, xTs, offs)
        return dx, dWg, dWu, dWd, None, None, None, None, None


def mxfp8_swiglu_expert(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, offs: torch.Tensor,
                        *, w_mxfp8=None, weight_cache=None, check_offsets: bool = True) -> torch.Tensor:
    """Differentiable SwiGLU routed expert: y[m] = (silu(x[m] Wg[g]^T) * (x[m] Wu[g]^T)) Wd[g]^T
    for rows m of group g.  x [M, D], Wg and Wu [G, H, D], Wd [G, D, H], all bf16; offs int32
    cumulative end rows; y [M, D] bf16.  Group sizes must be multiples of 32 when weight
    gradients are needed.  Prequantized weights: ``w_mxfp8 = (gate_quad, up_quad, down_quad)``
    (each as ``quantize_expert_weights`` returns) or an ``Mxfp8WeightCache``.  check_offsets: as for
    ``to_mxfp8_then_scaled_grouped_mm`` (a device check of offs, one stream synchronization per
    forward; bad offsets raise Mxfp8Error)."""
    for t in (x, Wg, Wu, Wd):
        if t.dtype != torch.bfloat16:
            raise ValueError("mxfp8_swiglu_expert expects bf16 tensors")
    if offs.dtype != torch.int32:
        raise ValueError("offs must be int32")
    G, H, D = Wg.shape
    if tuple(Wu.shape) != (G, H, D) or tuple(Wd.shape) != (G, D, H) or x.dim() != 2 or x.shape[1] != D:
        raise ValueError("shapes: x [M, D], Wg and Wu [G, H, D], Wd [G, D, H]")
    _offsets(offs, G)
    if w_mxfp8 is not None and weight_cache is not None:
        raise ValueError("pass w_mxfp8 or weight_cache, not both")
    if weight_cache is not None:
        w_mxfp8 = tuple(weight_cache.get(W) for W in (Wg, Wu, Wd))
    qg, qu, qd = w_mxfp8 if w_mxfp8 is not None else (None, None, None)
    return _Mxfp8SwiGLUExpert.apply(x, Wg, Wu, Wd, offs, qg, qu, qd, bool(check_offsets))
