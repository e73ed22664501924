"""Prequantized expert weights on the GPU ("feat(moe): add MoK MXFP8 expert support": the
(weight_fp8, weight_scale, weight_t_fp8, weight_t_scale) quadruple, kept across microbatches
until the optimizer step).

- The quadruple equals the oracle's plain and transposed quantization of W, byte for byte.
- Microbatches through the cache give bit-identical outputs and gradients to the on-the-fly
  path, and W is quantized once per optimizer step.
- After an in-place optimizer update, the next microbatch sees the new weights.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._util import assert_gemm_close, f64, require_gpu, sizes_to_ends, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


SIZES = [96, 0, 160]
G, N, K = 3, 256, 192
M = sum(SIZES)


def offs_dev():
    return torch.tensor(sizes_to_ends(SIZES).astype(np.int32), device="cuda")


def test_quadruple_equals_oracle(mx):
    W = synth.randn_bf16((G, N, K), 0.02, seed=70)
    wq, ws, wTq, wTs = [u8(t) for t in mx.quantize_expert_weights(W.cuda())]
    for g in range(G):
        qo, so = oracle.quantize_rows(u16(W[g]))
        qTo, sTo = oracle.quantize_cols(u16(W[g]))
        assert np.array_equal(wq[g], qo) and np.array_equal(wTq[g], qTo)
        assert np.array_equal(ws[g], oracle.blocked_rowgroups(so, [N]))
        assert np.array_equal(wTs[g], oracle.blocked_rowgroups(sTo, [K]))


def step(mx, A, W, D, offs, **kw):
    A = A.clone().requires_grad_(True)
    out = mx.to_mxfp8_then_scaled_grouped_mm(A, W, offs, **kw)
    W.grad = None
    out.backward(D)
    torch.cuda.synchronize()
    return out.detach().clone(), A.grad.clone(), W.grad.clone()


def test_microbatches_through_cache_match_on_the_fly(mx):
    offs = offs_dev()
    W = torch.nn.Parameter(synth.randn_bf16((G, N, K), 0.02, seed=71).cuda())
    opt = torch.optim.SGD([W], lr=0.5)
    cache = mx.Mxfp8WeightCache()
    cache.attach(opt)
    for opt_step in range(2):
        for mb in range(3):
            A = synth.randn_bf16((M, K), 1.0, seed=100 + 10 * opt_step + mb).cuda()
            D = synth.randn_bf16((M, N), 1e-2, seed=200 + 10 * opt_step + mb).cuda()
            ref = step(mx, A, W, D, offs)
            got = step(mx, A, W, D, offs, weight_cache=cache)
            for r, g_, what in zip(ref, got, ("out", "dA", "dW")):
                assert torch.equal(r.view(torch.int16), g_.view(torch.int16)), f"step {opt_step} mb {mb}: {what}"
        assert cache.misses == opt_step + 1 and cache.hits == 2 * (opt_step + 1)
        W.grad = torch.ones_like(W) * 1e-3
        opt.step()                          # in-place update + post-step invalidation


def test_cached_step_against_oracle(mx):
    offs = offs_dev()
    W = torch.nn.Parameter(synth.randn_bf16((G, N, K), 0.02, seed=72).cuda())
    cache = mx.Mxfp8WeightCache()
    A = synth.randn_bf16((M, K), 1.0, seed=73)
    cache.get(W)
    out, _, _ = step(mx, A.cuda(), W, torch.zeros(M, N, dtype=torch.bfloat16, device="cuda"), offs,
                     weight_cache=cache)
    aq, as_ = oracle.quantize_rows(u16(A))
    wq, ws = zip(*[oracle.quantize_rows(u16(W[g].detach().cpu())) for g in range(G)])
    ref = oracle.grouped_mm_rows(aq, as_, np.stack(wq), np.stack(ws), sizes_to_ends(SIZES))
    assert_gemm_close(f64(out), ref, what="cached fwd")
    assert cache.hits == 1 and cache.misses == 1


def test_explicit_quadruple_and_validation(mx):
    offs = offs_dev()
    W = synth.randn_bf16((G, N, K), 0.02, seed=74).cuda()
    A = synth.randn_bf16((M, K), 1.0, seed=75).cuda()
    quad = mx.quantize_expert_weights(W)
    a = mx.to_mxfp8_then_scaled_grouped_mm(A, W, offs, w_mxfp8=quad)
    b = mx.to_mxfp8_then_scaled_grouped_mm(A, W, offs)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    with pytest.raises(ValueError):
        mx.to_mxfp8_then_scaled_grouped_mm(A, W, offs, w_mxfp8=(quad[0][:, :, :64].contiguous(),) + quad[1:])
    with pytest.raises(ValueError):
        mx.to_mxfp8_then_scaled_grouped_mm(A, W, offs, w_mxfp8=quad, weight_cache=mx.Mxfp8WeightCache())
