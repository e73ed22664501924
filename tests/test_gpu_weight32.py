"""32x32-block weight quantization consumed by the grouped GEMMs ("MXFP8 (Micro-scaling FP8)",
"Low-precision Flash Attention", item 3: one scale per [32, 32] block makes the quantization
transpose invariant, so each tensor is quantized once and the backward uses its transpose).

- mxfp8_quantize_3d_experts(W, BLOCK32X32 | ROW | COL): q equals the oracle's 32x32 codes, qT
  is exactly q transposed, and both scale copies repeat the block scale on each row (column),
  byte for byte in the compact and in the blocked layout (padding included).
- The forward and dgrad GEMMs on those weights are within the GEMM bound of the oracle's fp64
  GEMMs of the same 32x32-dequantized weights; so is the composite op with weight_block32x32.
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


def oracle_w32(W):
    """Per expert: (codes [N, K], compact scales expanded per row [N, K/32], codes^T [K, N],
    scales of the transpose expanded per row [K, N/32])."""
    out = []
    for g in range(W.shape[0]):
        q, S = oracle.quantize_32x32(u16(W[g]))
        out.append((q, np.repeat(S, 32, axis=0), np.ascontiguousarray(q.T), np.repeat(S.T, 32, axis=0)))
    return out


@pytest.mark.parametrize("G,N,K", [(3, 160, 96), (2, 128, 256), (1, 32, 32), (2, 256, 416)])
@pytest.mark.parametrize("layout", ["compact", "blocked"])
def test_3d_block32_matches_oracle(mx, G, N, K, layout):
    W = synth.randn_bf16((G, N, K), 0.02, seed=N + K + G)
    W[0, :32, :32] *= 1000.0   # one loud block: its neighbours keep their own scales
    lay = mx.SCALES_COMPACT if layout == "compact" else mx.SCALES_BLOCKED
    status = mx.new_status()
    q, s, qT, sT = [u8(t) for t in mx.mxfp8_quantize_3d_experts(W.cuda(), mx.ROW | mx.COL | mx.BLOCK32X32,
                                                                 lay, status)]
    mx.read_status(status)
    for g, (qo, so, qTo, sTo) in enumerate(oracle_w32(W)):
        assert np.array_equal(q[g], qo) and np.array_equal(qT[g], qTo)
        assert np.array_equal(qT[g], q[g].T)
        if layout == "compact":
            assert np.array_equal(s[g], so) and np.array_equal(sT[g], sTo)
        else:
            assert np.array_equal(s[g], oracle.blocked_rowgroups(so, [N]))
            assert np.array_equal(sT[g], oracle.blocked_rowgroups(sTo, [K]))


def test_3d_block32_single_directions_match_fused(mx):
    W = synth.randn_bf16((2, 128, 192), 0.02, seed=5).cuda()
    both = mx.mxfp8_quantize_3d_experts(W, mx.ROW | mx.COL | mx.BLOCK32X32, mx.SCALES_BLOCKED)
    row = mx.mxfp8_quantize_3d_experts(W, mx.ROW | mx.BLOCK32X32, mx.SCALES_BLOCKED)
    col = mx.mxfp8_quantize_3d_experts(W, mx.COL | mx.BLOCK32X32, mx.SCALES_BLOCKED)
    torch.cuda.synchronize()
    assert torch.equal(both[0], row[0]) and torch.equal(both[1], row[1])
    assert torch.equal(both[2], col[2]) and torch.equal(both[3], col[3])
    with pytest.raises(mx.Mxfp8Error, match="LAYOUT"):
        mx.mxfp8_quantize_3d_experts(W, mx.BLOCK32X32, mx.SCALES_BLOCKED)


def test_gemms_on_block32_weights(mx):
    sizes = [96, 0, 160, 64]
    G, N, K = len(sizes), 256, 192
    M = sum(sizes)
    A = synth.randn_bf16((M, K), 1.0, seed=21)
    D = synth.randn_bf16((M, N), 1.0, seed=22)
    W = synth.randn_bf16((G, N, K), 0.02, seed=23)
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")
    wq, ws, wTq, wTs = mx.quantize_expert_weights(W.cuda(), block32x32=True)
    aq, as_, _, _ = mx.mxfp8_quantize_2d(A.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs)
    dq, ds, _, _ = mx.mxfp8_quantize_2d(D.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs)
    out = mx.mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs)
    dA = mx.mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs)
    torch.cuda.synchronize()
    o = oracle_w32(W)
    ends = sizes_to_ends(sizes)
    oaq, oas = oracle.quantize_rows(u16(A))
    odq, ods = oracle.quantize_rows(u16(D))
    ref = oracle.grouped_mm_rows(oaq, oas, np.stack([t[0] for t in o]), np.stack([t[1] for t in o]), ends)
    refd = oracle.grouped_mm_rows(odq, ods, np.stack([t[2] for t in o]), np.stack([t[3] for t in o]), ends)
    assert_gemm_close(f64(out), ref, what="fwd on 32x32 weights")
    assert_gemm_close(f64(dA), refd, what="dgrad on 32x32 weights")


def test_composite_with_block32_weights(mx):
    sizes = [128, 64, 96]
    G, N, K = len(sizes), 128, 256
    M = sum(sizes)
    A = synth.randn_bf16((M, K), 1.0, seed=31)
    W = synth.randn_bf16((G, N, K), 0.02, seed=32)
    dO = synth.randn_bf16((M, N), 1e-2, seed=33)
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")
    Ag, Wg = A.cuda().requires_grad_(True), W.cuda().requires_grad_(True)
    out = mx.to_mxfp8_then_scaled_grouped_mm(Ag, Wg, offs, weight_block32x32=True)
    out.backward(dO.cuda())
    torch.cuda.synchronize()
    o = oracle_w32(W)
    ends = sizes_to_ends(sizes)
    oaq, oas = oracle.quantize_rows(u16(A))
    odq, ods = oracle.quantize_rows(u16(dO))
    assert_gemm_close(f64(out), oracle.grouped_mm_rows(oaq, oas, np.stack([t[0] for t in o]),
                                                       np.stack([t[1] for t in o]), ends), what="out")
    assert_gemm_close(f64(Ag.grad), oracle.grouped_mm_rows(odq, ods, np.stack([t[2] for t in o]),
                                                           np.stack([t[3] for t in o]), ends), what="dA")
    # the weight gradient does not involve the weight quantization
    dTq, dTs = oracle.quantize_cols(u16(dO))
    aTq, aTs = oracle.quantize_cols(u16(A))
    assert_gemm_close(f64(Wg.grad), oracle.grouped_mm_wgrad(dTq, dTs, aTq, aTs, ends), what="dW")


def test_full_size_block32_sampled(mx):
    """The Scout expert weights [8, 8192, 5120] with 32x32 blocks, sampled blocks of both copies
    against the oracle, and sampled forward / dgrad outputs on those weights."""
    w = synth.workload("scout", seed=0, device="cuda")
    W, A, D, sizes = w["W"], w["A"], w["dOut"], w["sizes"]
    G, N, K, M = w["G"], w["N"], w["K"], w["M"]
    st = mx.new_status()
    wq, ws, wTq, wTs = mx.mxfp8_quantize_3d_experts(W, mx.ROW | mx.COL | mx.BLOCK32X32, mx.SCALES_BLOCKED, st)
    mx.read_status(st)
    rng = np.random.default_rng(13)
    Wc = W.cpu()                       # sampled blocks are sliced on the host
    for _ in range(12):
        g, bn, bk = int(rng.integers(0, G)), int(rng.integers(0, N // 32)), int(rng.integers(0, K // 32))
        qo, so = oracle.quantize_32x32(u16(Wc[g, 32 * bn:32 * bn + 32, 32 * bk:32 * bk + 32]))
        assert np.array_equal(u8(wq[g, 32 * bn:32 * bn + 32, 32 * bk:32 * bk + 32]), qo)
        assert np.array_equal(u8(wTq[g, 32 * bk:32 * bk + 32, 32 * bn:32 * bn + 32]), qo.T)
        for i in (0, 17, 31):
            assert int(ws[g, oracle.blocked_offset(32 * bn + i, bk, K // 128)].item()) == so[0, 0]
            assert int(wTs[g, oracle.blocked_offset(32 * bk + i, bn, N // 128)].item()) == so[0, 0]
    offs = w["offs"].cuda()
    ends = sizes_to_ends(sizes)
    aq, as_, _, _ = mx.mxfp8_quantize_2d(A, mx.ROW, mx.SCALES_BLOCKED, offs, st)
    dq, ds, _, _ = mx.mxfp8_quantize_2d(D, mx.ROW, mx.SCALES_BLOCKED, offs, st)
    out = mx.mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs, dev_status=st)
    dA = mx.mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs, dev_status=st)
    mx.read_status(st)
    ref, got, refd, gotd = [], [], [], []
    for r in rng.integers(0, M, 8):
        r = int(r)
        g = int(np.searchsorted(ends, r, side="right"))
        qa, sa = oracle.quantize_rows(u16(A[r:r + 1]))
        qd, sd = oracle.quantize_rows(u16(D[r:r + 1]))
        for bn in rng.integers(0, N // 32, 2):
            blk_q, blk_s = [], []
            for bk in range(K // 32):   # the 32 rows n of W[g] in block-row bn, all of K
                q32, s32 = oracle.quantize_32x32(u16(Wc[g, 32 * bn:32 * bn + 32, 32 * bk:32 * bk + 32]))
                blk_q.append(q32)
                blk_s.append(s32[0, 0])
            qrows = np.concatenate(blk_q, axis=1)                      # [32, K]
            srows = np.tile(np.array(blk_s, np.uint8), (32, 1))         # [32, K/32]
            n = int(rng.integers(0, 32))
            ref.append(oracle.dot(qa[0], sa[0], qrows[n], srows[n]))
            got.append(float(out[r, 32 * int(bn) + n].item()))
        # dgrad: dA[r, k] = sum_n dOut[r, n] W[g][n, k], column k of W through its 32x32 blocks
        k = int(rng.integers(0, K))
        bk = k // 32
        col_q, col_s = [], []
        for bn in range(N // 32):
            q32, s32 = oracle.quantize_32x32(u16(Wc[g, 32 * bn:32 * bn + 32, 32 * bk:32 * bk + 32]))
            col_q.append(q32[:, k - 32 * bk])
            col_s.append(s32[0, 0])
        refd.append(oracle.dot(qd[0], sd[0], np.concatenate(col_q), np.array(col_s, np.uint8)))
        gotd.append(float(dA[r, k].item()))
    assert_gemm_close(np.array(got), np.array(ref), what="fwd sampled on 32x32 weights")
    assert_gemm_close(np.array(gotd), np.array(refd), what="dgrad sampled on 32x32 weights")
