"""The SwiGLU backward with the quantization of dh1 and dh3 fused in (mxfp8_swiglu_bwd_quantize)
against the oracle's backward stage followed by its row- and token-wise quantization ("MXFP8
(Micro-scaling FP8)", "Neutralizing quantization overhead"; "feat(moe): add MoK MXFP8 expert
support").

The inputs dh, h1, h3 are the same bf16 tensors on both sides.  The kernel evaluates the
derivative in fp32, the oracle in fp64 with one rounding per op.  The products dh*h3 and
dh*silu of two bf16 values are exact in fp32, so the two sides can round a bf16 result
differently only where the exact value lies within the fp32 evaluation error of a bf16 rounding
midpoint:
- dh3 = bf16(dh * bf16(silu(h1))): only through silu, whose fp32 value x / (1 + expf(-x)) is
  within a few 2^-24 (relative) of the exact one;
- dh1 = bf16(bf16(dh*h3) * s * (1 + h1 (1 - s))), s = sigmoid(h1): the fp32 error of s (a few
  2^-24 relative) enters 1 - s absolutely, so the factor f = 1 + h1 (1 - s) carries an absolute
  error of about |h1| s 2^-22, which is large relative to f where f crosses zero (h1 near -1.28).
Every element farther than that error (times a safety factor) from a midpoint must give the same
bf16 value, so codes and scales are compared byte for byte outside those elements (and their
blocks); the excluded elements are a small fraction.  Everything else (padding included) is exact."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._mxcompare import compare_quantized
from tests._util import require_gpu, sizes_to_ends, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def near_midpoint(v, err):
    """Elements whose fp64 value v lies within err of a bf16 rounding midpoint."""
    a = np.abs(v)
    ex = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    q = np.ldexp(1.0, (ex - 7).astype(np.int64))          # bf16 quantum at |v|
    frac = a / q - np.floor(a / q)
    return (np.abs(frac - 0.5) * q <= err) & (a > 0)


def bwd_ties(dh_u16, h1_u16, h3_u16):
    """Masks of the dh1 and dh3 elements that fp32 evaluation may round to the other neighbour."""
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g, x, h3 = f(dh_u16), f(h1_u16), f(h3_u16)
    u = 2.0 ** -24
    sig = 1.0 / (1.0 + np.exp(-x))
    silu = x * sig
    ties3 = near_midpoint(silu, 16 * u * np.abs(silu))
    ds = f(oracle.bf16_from_f64(g * h3))                   # bf16(dh * h3): exact product, one rounding
    fac = 1.0 + x * (1.0 - sig)
    v1 = ds * sig * fac
    err1 = np.abs(ds) * sig * (np.abs(fac) * 8 * u + (np.abs(x) * sig + np.abs(x) * (1.0 - sig) + 1.0) * 8 * u)
    ties1 = near_midpoint(v1, 4 * err1 + 4 * u * np.abs(v1))
    return ties1, ties3


def inputs(M, H, seed):
    dh = synth.randn_bf16((M, H), 1e-2, seed=seed)
    h1 = synth.randn_bf16((M, H), 3.0, seed=seed + 1)
    h3 = synth.randn_bf16((M, H), 1.0, seed=seed + 2)
    return dh, h1, h3


@pytest.mark.parametrize("sizes,H", [([96, 0, 160, 32], 384), ([256], 128), ([128, 64], 416)])
def test_matches_oracle(mx, sizes, H):
    M = sum(sizes)
    dh, h1, h3 = inputs(M, H, seed=H + M)
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")
    st = mx.new_status()
    o1, o3 = mx.mxfp8_swiglu_bwd_quantize(dh.cuda(), h1.cuda(), h3.cuda(), offs, st)
    mx.read_status(st)
    ref = oracle.swiglu_bwd_quantized(u16(dh), u16(h1), u16(h3))
    ends = sizes_to_ends(sizes)
    ties = dict(zip(("dh1", "dh3"), bwd_ties(u16(dh), u16(h1), u16(h3))))
    for name, (q, s, qT, sT) in (("dh1", o1), ("dh3", o3)):
        t = ties[name]
        assert t.mean() < 2e-2, f"{name}: {t.mean():.4f} of the elements excluded"
        compare_quantized(u8(q), u8(s), ref[name + "_q"], ref[name + "_s"], "rows", ends, exact=True, exclude=t,
                          what=name + " rows")
        compare_quantized(u8(qT), u8(sT), ref[name + "T_q"], ref[name + "T_s"], "cols", ends, exact=True,
                          exclude=t.T, what=name + " cols")
        # and every element, ties included, within one E4M3 step
        kw = dict(exact=False, min_code_eq=0.999, min_scale_eq=0.999)
        compare_quantized(u8(q), u8(s), ref[name + "_q"], ref[name + "_s"], "rows", ends, what=name + " rows", **kw)
        compare_quantized(u8(qT), u8(sT), ref[name + "T_q"], ref[name + "T_s"], "cols", ends, what=name + " cols",
                          **kw)


def test_matches_unfused_gpu_path(mx):
    """The same step as torch's bf16 autograd ops followed by two ROW|COL quantizations."""
    sizes, H = [128, 96, 32], 256
    M = sum(sizes)
    dh, h1, h3 = [t.cuda() for t in inputs(M, H, seed=5)]
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")
    o1, o3 = mx.mxfp8_swiglu_bwd_quantize(dh, h1, h3, offs)
    # torch's bf16 autograd ops for h = silu(h1) * h3
    d3 = dh * torch.nn.functional.silu(h1)
    d1 = torch.ops.aten.silu_backward(dh * h3, h1)
    for fused, d in ((o1, d1), (o3, d3)):
        ref = mx.mxfp8_quantize_2d(d.contiguous(), mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs)
        torch.cuda.synchronize()
        assert (u8(fused[0]) == u8(ref[0])).mean() >= 0.999
        assert (u8(fused[2]) == u8(ref[2])).mean() >= 0.999


def test_argument_errors(mx):
    z = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    offs = torch.tensor([64], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        mx.mxfp8_swiglu_bwd_quantize(z, z, torch.zeros((64, 32), dtype=torch.bfloat16, device="cuda"), offs)
    bad = torch.zeros((48, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.Mxfp8Error, match="ALIGN"):
        mx.mxfp8_swiglu_bwd_quantize(bad, bad, bad, torch.tensor([48], dtype=torch.int32, device="cuda"))


def test_full_size_sampled(mx):
    """The SwiGLU expert's intermediate shape [65600, 8192] in two groups, sampled row blocks of
    dh1 / dh3 and token blocks of their transposes against the oracle."""
    sizes = synth.swiglu_group_sizes()
    M, H = sum(sizes), 8192
    dh = synth.randn_bf16((M, H), 1e-2, seed=21, device="cuda")
    h1 = synth.randn_bf16((M, H), 3.0, seed=22, device="cuda")
    h3 = synth.randn_bf16((M, H), 1.0, seed=23, device="cuda")
    ends = sizes_to_ends(sizes)
    starts = np.concatenate([[0], ends[:-1]])
    offs = torch.tensor(ends.astype(np.int32), device="cuda")
    st = mx.new_status()
    o1, o3 = mx.mxfp8_swiglu_bwd_quantize(dh, h1, h3, offs, st)
    mx.read_status(st)
    padded = np.concatenate([[0], np.cumsum([-(-int(m) // 128) * 128 for m in sizes])])
    rng = np.random.default_rng(9)
    q_g, q_o, s_g, s_o, tie = [], [], [], [], []
    for r in np.unique(np.concatenate([rng.integers(0, M, 64), starts, ends - 1])):
        r = int(r)
        g = int(np.searchsorted(ends, r, side="right"))
        j = int(rng.integers(0, H // 32))
        sl = slice(32 * j, 32 * j + 32)
        b = (u16(dh[r, sl]), u16(h1[r, sl]), u16(h3[r, sl]))
        d1, d3 = oracle.swiglu_bwd_bf16(*b)
        t1, t3 = bwd_ties(*b)
        pr = int(padded[g]) + r - int(starts[g])
        for d, t, (q, s, _, _) in ((d1, t1, o1), (d3, t3, o3)):
            qo, so = oracle.quantize_vec(d)
            q_o.append(qo); s_o.append(so[0]); tie.append(t)
            q_g.append(u8(q[r, sl])); s_g.append(int(s[oracle.blocked_offset(pr, j, H // 128)].item()))
    ct = int(padded[-1]) // 128
    for _ in range(32):
        g = int(rng.integers(0, len(sizes)))
        t0 = int(starts[g]) + 32 * int(rng.integers(0, sizes[g] // 32))
        c = int(rng.integers(0, H))
        b = (u16(dh[t0:t0 + 32, c]), u16(h1[t0:t0 + 32, c]), u16(h3[t0:t0 + 32, c]))
        d1, d3 = oracle.swiglu_bwd_bf16(*b)
        t1, t3 = bwd_ties(*b)
        cq = int(padded[g]) // 32 + (t0 - int(starts[g])) // 32
        for d, t, (_, _, qT, sT) in ((d1, t1, o1), (d3, t3, o3)):
            qo, so = oracle.quantize_vec(d)
            q_o.append(qo); s_o.append(so[0]); tie.append(t)
            q_g.append(u8(qT[c, t0:t0 + 32])); s_g.append(int(sT[oracle.blocked_offset(c, cq, ct)].item()))
    q_g, q_o, s_g, s_o, tie = np.stack(q_g), np.stack(q_o), np.array(s_g), np.array(s_o), np.stack(tie)
    clean = ~tie.any(axis=1)                    # sampled blocks without a possible rounding tie
    assert clean.mean() > 0.8
    assert np.array_equal(s_g[clean], s_o[clean]), "scales of tie-free blocks"
    assert np.array_equal(q_g[clean], q_o[clean]), "codes of tie-free blocks"
    assert np.all(np.abs(s_g.astype(int) - s_o.astype(int)) <= 1)
