"""Whole-tensor GPU parity at sizes where every persistent CTA runs several tiles.

The kernels are persistent: one CTA (or CTA pair) per SM walks a static tile order, reuses its
tensor-memory accumulator from tile to tile, and cycles its shared-memory stage ring many times.
The small cases of the other test files give a CTA at most one tile; here each GEMM mode and each
quantize direction runs at least three tiles per CTA (and several wraps of the stage ring), with
ragged and empty groups, and every output element is compared with the oracle:
- quantization: codes and blocked scales byte for byte (padding included);
- GEMMs: |gpu - o| <= 1e-2 |o| + 1e-3 rms(o) elementwise against the fp64 oracle (its
  matmul-per-group form, pinned to the scalar loops in test_oracle_layout_gemm.py);
- the fused SwiGLU gate/up epilogue: exact-arithmetic inputs, so h1, h3 equal the oracle's bf16
  values and h's codes and scales are byte-exact apart from silu rounding ties.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._mxcompare import compare_quantized
from tests._util import assert_gemm_close, f64, require_gpu, sizes_to_ends, u8, u16

pytestmark = pytest.mark.gpu

N_SM = 152


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def offs_dev(sizes):
    return torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")


def ceil(a, b):
    return -(-a // b)


# fwd / dgrad: ragged groups (any size), one empty
ROW_SIZES = [1000, 0, 2999, 1201, 2992]


def rowgrouped_tiles(sizes, n_out, bn=256):
    return sum(ceil(m, 128) for m in sizes) * ceil(n_out, bn)


def test_fwd_whole_tensor_several_tiles_per_cta(mx):
    sizes, N, K = ROW_SIZES, 2048, 512
    assert rowgrouped_tiles(sizes, N) >= 3 * N_SM
    M, G = sum(sizes), len(sizes)
    A = synth.randn_bf16((M, K), 1.0, seed=301)
    W = synth.randn_bf16((G, N, K), 0.02, seed=302)
    offs = offs_dev(sizes)
    st = mx.new_status()
    aq, as_, _, _ = mx.mxfp8_quantize_2d(A.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)
    wq, ws, _, _ = mx.mxfp8_quantize_3d_experts(W.cuda(), mx.ROW, mx.SCALES_BLOCKED, st)
    out = mx.mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs, dev_status=st)
    mx.read_status(st)
    oq, os_ = oracle.quantize_rows(u16(A))
    wo = [oracle.quantize_rows(u16(W[g])) for g in range(G)]
    ref = oracle.grouped_mm_rows_blas(oq, os_, np.stack([q for q, _ in wo]), np.stack([s for _, s in wo]),
                                      sizes_to_ends(sizes))
    assert_gemm_close(f64(out), ref, what="fwd (wrapping)")


def test_dgrad_whole_tensor_several_tiles_per_cta(mx):
    sizes, N, K = ROW_SIZES, 512, 2048
    assert rowgrouped_tiles(sizes, K) >= 3 * N_SM
    M, G = sum(sizes), len(sizes)
    D = synth.randn_bf16((M, N), 1e-3, seed=311)
    W = synth.randn_bf16((G, N, K), 0.02, seed=312)
    offs = offs_dev(sizes)
    st = mx.new_status()
    dq, ds, _, _ = mx.mxfp8_quantize_2d(D.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)
    _, _, wTq, wTs = mx.mxfp8_quantize_3d_experts(W.cuda(), mx.COL, mx.SCALES_BLOCKED, st)
    dA = mx.mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs, dev_status=st)
    mx.read_status(st)
    oq, os_ = oracle.quantize_rows(u16(D))
    wo = [oracle.quantize_cols(u16(W[g])) for g in range(G)]  # [K, N] per expert
    ref = oracle.grouped_mm_rows_blas(oq, os_, np.stack([q for q, _ in wo]), np.stack([s for _, s in wo]),
                                      sizes_to_ends(sizes))
    assert_gemm_close(f64(dA), ref, what="dgrad (wrapping)")


def test_dgrad2_whole_tensor_several_tiles_per_cta(mx):
    sizes, N, K = ROW_SIZES, 256, 2048
    assert rowgrouped_tiles(sizes, K) >= 3 * N_SM
    M, G = sum(sizes), len(sizes)
    ends = sizes_to_ends(sizes)
    offs = offs_dev(sizes)
    Ds = [synth.randn_bf16((M, N), 1.0, seed=321 + i) for i in range(2)]
    Ws = [synth.randn_bf16((G, N, K), 0.02, seed=323 + i) for i in range(2)]
    st = mx.new_status()
    q = [mx.mxfp8_quantize_2d(D.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)[:2] for D in Ds]
    wt = [mx.mxfp8_quantize_3d_experts(W.cuda(), mx.COL, mx.SCALES_BLOCKED, st)[2:] for W in Ws]
    dA = mx.mxfp8_grouped_mm_dgrad2(*q[0], *wt[0], *q[1], *wt[1], offs, dev_status=st)
    mx.read_status(st)
    ref = 0
    for D, W in zip(Ds, Ws):
        dq, ds = oracle.quantize_rows(u16(D))
        wo = [oracle.quantize_cols(u16(W[g])) for g in range(G)]
        ref = ref + oracle.grouped_mm_rows_blas(dq, ds, np.stack([a for a, _ in wo]), np.stack([b for _, b in wo]),
                                                ends)
    assert_gemm_close(f64(dA), ref, what="dgrad2 (wrapping)")


def test_wgrad_whole_tensor_several_tiles_per_cluster(mx):
    """The CTA-pair wgrad: 256 x 256 tiles per group (an empty group's tiles are zero fills), group
    sizes multiples of 32 but not of 128 (ragged last k-tiles), >= 3 tiles per cluster of 2."""
    sizes, N, K = [1024, 0, 2976, 1216, 2976], 2048, 2048
    G = len(sizes)
    assert G * ceil(N, 256) * ceil(K, 256) >= 3 * (N_SM // 2)
    M = sum(sizes)
    D = synth.randn_bf16((M, N), 1e-3, seed=331)
    A = synth.randn_bf16((M, K), 1.0, seed=332)
    offs = offs_dev(sizes)
    st = mx.new_status()
    _, _, dTq, dTs = mx.mxfp8_quantize_2d(D.cuda(), mx.COL, mx.SCALES_BLOCKED, offs, st)
    _, _, aTq, aTs = mx.mxfp8_quantize_2d(A.cuda(), mx.COL, mx.SCALES_BLOCKED, offs, st)
    dW = mx.mxfp8_grouped_mm_wgrad(dTq, dTs, aTq, aTs, offs, dev_status=st)
    mx.read_status(st)
    oq, os_ = oracle.quantize_cols(u16(D))
    aoq, aos = oracle.quantize_cols(u16(A))
    ref = oracle.grouped_mm_wgrad_blas(oq, os_, aoq, aos, sizes_to_ends(sizes))
    got = f64(dW)
    assert np.all(got[1] == 0.0), "empty group must give zero dW"
    assert_gemm_close(got, ref, what="wgrad (wrapping)")


def test_quantize_rowcol_grouped_whole_tensor(mx):
    """ROW|COL from one read, blocked scales with 5 token groups (an empty one), [8192, 2048]:
    64 x 16 = 1024 tiles over 2 CTAs per SM."""
    sizes, K = [1024, 0, 2976, 1216, 2976], 2048
    M = sum(sizes)
    assert ceil(M, 128) * ceil(K, 128) >= 3 * 2 * N_SM
    x = synth.log_uniform_rows(M, K, seed=341)
    ends = sizes_to_ends(sizes)
    st = mx.new_status()
    q, s, qT, sT = mx.mxfp8_quantize_2d(x.cuda(), mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs_dev(sizes), st)
    mx.read_status(st)
    qo, so = oracle.quantize_rows(u16(x))
    qTo, sTo = oracle.quantize_cols(u16(x))
    want_r = oracle.blocked_rowgroups(so, ends)
    want_c = oracle.blocked_colgroups(sTo, ends)
    assert np.array_equal(u8(q), qo), "row codes"
    assert np.array_equal(u8(qT), qTo), "column codes"
    assert np.array_equal(u8(s)[:want_r.size], want_r), "row scales (blocked, padding included)"
    assert np.array_equal(u8(sT)[:want_c.size], want_c), "column scales (blocked, padding included)"


def test_quantize_3d_whole_tensor(mx):
    """Expert weights [8, 1024, 2048] plain and transposed from one read: 1024 tiles."""
    G, N, K = 8, 1024, 2048
    w = synth.randn_bf16((G, N, K), 0.02, seed=351)
    st = mx.new_status()
    q, s, qT, sT = mx.mxfp8_quantize_3d_experts(w.cuda(), mx.ROW | mx.COL, mx.SCALES_BLOCKED, st)
    mx.read_status(st)
    q, s, qT, sT = u8(q), u8(s), u8(qT), u8(sT)
    for g in range(G):
        qo, so = oracle.quantize_rows(u16(w[g]))
        qTo, sTo = oracle.quantize_cols(u16(w[g]))
        assert np.array_equal(q[g], qo) and np.array_equal(qT[g], qTo), f"codes of expert {g}"
        assert np.array_equal(s[g], oracle.blocked_rowgroups(so, [N])), f"scales of expert {g}"
        assert np.array_equal(sT[g], oracle.blocked_rowgroups(sTo, [K])), f"transposed scales of expert {g}"


def exact_inputs(M, D, G, H, seed):
    """Few significant bits: every fp32 partial sum of the GEMMs is exact."""
    g = torch.Generator().manual_seed(seed)
    xv = torch.tensor([0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0])
    wv = torch.tensor([0.0, 1 / 16, -1 / 16, 1 / 8, -1 / 8, 1 / 4, -1 / 4])
    x = xv[torch.randint(0, 7, (M, D), generator=g)].to(torch.bfloat16)
    Wg = wv[torch.randint(0, 7, (G, H, D), generator=g)].to(torch.bfloat16)
    Wu = wv[torch.randint(0, 7, (G, H, D), generator=g)].to(torch.bfloat16)
    return x, Wg, Wu


def near_silu_ties(h1_u16, rel=2.0 ** -21):
    a = (h1_u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = np.abs(a / (1.0 + np.exp(-a)))
    ex = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    q = np.ldexp(1.0, (ex - 7).astype(np.int64))
    frac = v / q - np.floor(v / q)
    return (np.abs(frac - 0.5) * q <= v * rel) & (v > 0)


def test_swiglu_fused_whole_tensor_several_tiles_per_cta(mx):
    sizes, H, D = [1024, 0, 2976, 1216, 2976], 1024, 256
    G, M = len(sizes), sum(sizes)
    assert sum(ceil(m, 128) for m in sizes) * ceil(H, 128) >= 3 * N_SM
    x, Wg, Wu = exact_inputs(M, D, G, H, seed=361)
    offs = offs_dev(sizes)
    st = mx.new_status()
    xq, xs, _, _ = mx.mxfp8_quantize_2d(x.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)
    gq, gs, _, _ = mx.mxfp8_quantize_3d_experts(Wg.cuda(), mx.ROW, mx.SCALES_BLOCKED, st)
    uq, us, _, _ = mx.mxfp8_quantize_3d_experts(Wu.cuda(), mx.ROW, mx.SCALES_BLOCKED, st)
    h1, h3, hq, hs, hTq, hTs = mx.mxfp8_grouped_mm_swiglu_fwd(xq, xs, gq, gs, uq, us, offs, True, st)
    mx.read_status(st)
    ends = sizes_to_ends(sizes)
    o = oracle.swiglu_gate_up(u16(x), u16(Wg), u16(Wu), ends, blas=True)
    assert np.array_equal(u16(h1), o["h1"]) and np.array_equal(u16(h3), o["h3"])
    ties = near_silu_ties(o["h1"])
    compare_quantized(u8(hq), u8(hs), o["h_q"], o["h_s"], "rows", ends, exact=True, exclude=ties, what="h rows")
    compare_quantized(u8(hTq), u8(hTs), o["hT_q"], o["hT_s"], "cols", ends, exact=True, exclude=ties.T,
                      what="h tokens")
    assert ties.mean() < 1e-3
