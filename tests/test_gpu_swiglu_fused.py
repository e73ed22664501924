"""The gate/up GEMMs with the SwiGLU and its MXFP8 quantization fused into the epilogue
(mxfp8_grouped_mm_swiglu_fwd) against the oracle's gate/up stage ("MXFP8 (Micro-scaling
FP8)", "Neutralizing quantization overhead": quantization fused into the kernel that
produces the activation; "feat(moe): add MoK MXFP8 expert support": gate/up/down weights).

Parity bars:
- h1, h3 (bf16 GEMM outputs): the GEMM bound |gpu - o| <= 1e-2 |o| + 1e-3 rms(o).
- Exact-arithmetic inputs (every fp32 accumulation exact, so h1 and h3 equal the oracle's):
  h_q, h_s, hT_q, hT_s byte for byte, padding included.  The only freedom left is silu in fp32
  versus fp64: the fp32 value x / (1 + expf(-x)) is within about 2^-22 (relative) of the exact
  one (expf within 2 ulp, the add and the divide within half an ulp each), so elements whose
  fp64 silu lies within 2^-21 of a bf16 rounding midpoint may round either way and are excluded.
- Random inputs: h1/h3 may differ from the oracle's by a bf16 ulp where fp32 accumulation
  crosses a rounding midpoint, and a one-ulp change of h moves its E4M3 code by at most one
  step (or its block scale by one).  So every dequantized element must lie within one E4M3
  step of the oracle's, every scale within one of the oracle's, and at least 99% of codes
  and 99.9% of scales must be identical.  The epilogue itself is then checked byte for byte:
  the oracle's SwiGLU stage and quantizations applied to the kernel's own bf16 h1, h3 must
  give h_q, h_s, hT_q, hT_s exactly, outside the silu rounding ties above.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._mxcompare import compare_quantized, e4m3_step
from tests._util import assert_gemm_close, f64, require_gpu, sizes_to_ends, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def offs_of(sizes):
    return torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")


def run_fused(mx, x, Wg, Wu, sizes, token_wise=True):
    offs = offs_of(sizes)
    status = mx.new_status()
    xq, xs, _, _ = mx.mxfp8_quantize_2d(x.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs)
    gq, gs, _, _ = mx.mxfp8_quantize_3d_experts(Wg.cuda(), mx.ROW, mx.SCALES_BLOCKED)
    uq, us, _, _ = mx.mxfp8_quantize_3d_experts(Wu.cuda(), mx.ROW, mx.SCALES_BLOCKED)
    out = mx.mxfp8_grouped_mm_swiglu_fwd(xq, xs, gq, gs, uq, us, offs, token_wise, status)
    torch.cuda.synchronize()
    return out, status


def near_silu_ties(h1_u16):
    """Elements whose fp64 silu(h1) lies within 2^-21 (relative) of a bf16 rounding midpoint."""
    a = (h1_u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = np.abs(a / (1.0 + np.exp(-a)))
    ex = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    q = np.ldexp(1.0, (ex - 7).astype(np.int64))       # bf16 quantum at v
    frac = v / q - np.floor(v / q)
    return (np.abs(frac - 0.5) * q <= v * 2.0 ** -21) & (v > 0)


CASES = [
    ([384, 0, 256, 96], 384, 256),   # 4 groups: an empty one, a 96-row tail tile
    ([160, 96], 160, 128),           # ragged H: the second column tile has 32 valid columns
    ([64], 128, 512),                # one group, 4 k-tiles
]


@pytest.mark.parametrize("sizes,H,D", CASES)
def test_fused_gate_up_random_inputs(mx, sizes, H, D):
    G, M = len(sizes), sum(sizes)
    x = synth.randn_bf16((M, D), 1.0, seed=80 + H)
    Wg = synth.randn_bf16((G, H, D), 0.08, seed=81 + H)
    Wu = synth.randn_bf16((G, H, D), 0.08, seed=82 + H)
    (h1, h3, hq, hs, hTq, hTs), status = run_fused(mx, x, Wg, Wu, sizes)
    mx.read_status(status)
    ends = sizes_to_ends(sizes)
    o = oracle.swiglu_gate_up(u16(x), u16(Wg), u16(Wu), ends)
    assert_gemm_close(f64(h1), o["h1_f64"], what="h1")
    assert_gemm_close(f64(h3), o["h3_f64"], what="h3")
    compare_quantized(u8(hq), u8(hs), o["h_q"], o["h_s"], "rows", ends, exact=False, what="h (row-wise)")
    compare_quantized(u8(hTq), u8(hTs), o["hT_q"], o["hT_s"], "cols", ends, exact=False, what="h (token-wise)")
    # the epilogue alone: the oracle's SwiGLU stage and quantizations applied to the kernel's own bf16
    # h1, h3 (so the GEMMs' fp32-vs-fp64 rounding no longer enters), byte for byte outside the elements
    # whose fp64 silu lies near a bf16 rounding midpoint
    hb = oracle.swiglu_bf16(u16(h1), u16(h3))
    ties = near_silu_ties(u16(h1))
    assert ties.mean() < 1e-3
    q_r, s_r = oracle.quantize_rows(hb)
    compare_quantized(u8(hq), u8(hs), q_r, s_r, "rows", ends, exact=True, exclude=ties, what="h rows (own h1, h3)")
    q_c, s_c = oracle.quantize_cols(hb)
    compare_quantized(u8(hTq), u8(hTs), q_c, s_c, "cols", ends, exact=True, exclude=ties.T,
                      what="h tokens (own h1, h3)")


def exact_inputs(M, D, G, H, seed):
    """Values with few significant bits: every partial sum of the GEMMs is exact in fp32."""
    g = torch.Generator().manual_seed(seed)
    xv = torch.tensor([0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0])
    wv = torch.tensor([0.0, 1 / 16, -1 / 16, 1 / 8, -1 / 8, 1 / 4, -1 / 4])
    x = xv[torch.randint(0, 7, (M, D), generator=g)].to(torch.bfloat16)
    Wg = wv[torch.randint(0, 7, (G, H, D), generator=g)].to(torch.bfloat16)
    Wu = wv[torch.randint(0, 7, (G, H, D), generator=g)].to(torch.bfloat16)
    return x, Wg, Wu


def test_fused_gate_up_exact_inputs_bit_exact(mx):
    sizes, H, D = [128, 64, 0, 192], 256, 256
    G, M = len(sizes), sum(sizes)
    x, Wg, Wu = exact_inputs(M, D, G, H, seed=90)
    (h1, h3, hq, hs, hTq, hTs), status = run_fused(mx, x, Wg, Wu, sizes)
    mx.read_status(status)
    ends = sizes_to_ends(sizes)
    o = oracle.swiglu_gate_up(u16(x), u16(Wg), u16(Wu), ends)
    assert np.array_equal(u16(h1), o["h1"]) and np.array_equal(u16(h3), o["h3"])
    ties = near_silu_ties(o["h1"])
    compare_quantized(u8(hq), u8(hs), o["h_q"], o["h_s"], "rows", ends, exact=True, exclude=ties, what="h rows")
    compare_quantized(u8(hTq), u8(hTs), o["hT_q"], o["hT_s"], "cols", ends, exact=True, exclude=ties.T,
                      what="h tokens")
    assert ties.mean() < 1e-3


def test_token_wise_requires_groups_of_32(mx):
    sizes, H, D = [48, 80], 128, 128
    G, M = len(sizes), sum(sizes)
    x = synth.randn_bf16((M, D), 1.0, seed=95)
    Wg = synth.randn_bf16((G, H, D), 0.08, seed=96)
    Wu = synth.randn_bf16((G, H, D), 0.08, seed=97)
    _, status = run_fused(mx, x, Wg, Wu, sizes, token_wise=True)
    with pytest.raises(mx.Mxfp8Error) as e:
        mx.read_status(status)
    assert e.value.status == 7  # MXFP8_ERR_OFFSETS
    # row-wise only: any group sizes
    (h1, h3, hq, hs, hTq, hTs), status = run_fused(mx, x, Wg, Wu, sizes, token_wise=False)
    mx.read_status(status)
    assert hTq is None and hTs is None
    ends = sizes_to_ends(sizes)
    o = oracle.swiglu_gate_up(u16(x), u16(Wg), u16(Wu), ends)
    assert_gemm_close(f64(h1), o["h1_f64"], what="h1")
    compare_quantized(u8(hq), u8(hs), o["h_q"], o["h_s"], "rows", ends, exact=False, what="h (row-wise)")


def test_fused_equals_unfused_gpu_path(mx):
    """Same GPU, two routes: the fused epilogue and (forward GEMM x2, torch bf16 SwiGLU,
    ROW|COL quantize).  h1/h3 come from the same MMA sequence; torch's bf16 silu evaluates
    the same fp32 expression, so the quantized bytes should agree almost everywhere."""
    sizes, H, D = [256, 128, 96], 256, 256
    G, M = len(sizes), sum(sizes)
    x = synth.randn_bf16((M, D), 1.0, seed=98)
    Wg = synth.randn_bf16((G, H, D), 0.08, seed=99)
    Wu = synth.randn_bf16((G, H, D), 0.08, seed=100)
    (h1, h3, hq, hs, hTq, hTs), status = run_fused(mx, x, Wg, Wu, sizes)
    mx.read_status(status)
    offs = offs_of(sizes)
    xq, xs, _, _ = mx.mxfp8_quantize_2d(x.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs)
    gq, gs, _, _ = mx.mxfp8_quantize_3d_experts(Wg.cuda(), mx.ROW, mx.SCALES_BLOCKED)
    uq, us, _, _ = mx.mxfp8_quantize_3d_experts(Wu.cuda(), mx.ROW, mx.SCALES_BLOCKED)
    r1 = mx.mxfp8_grouped_mm_fwd(xq, xs, gq, gs, offs)
    r3 = mx.mxfp8_grouped_mm_fwd(xq, xs, uq, us, offs)
    assert torch.equal(r1.view(torch.int16), h1.view(torch.int16))
    assert torch.equal(r3.view(torch.int16), h3.view(torch.int16))
    h = torch.nn.functional.silu(r1) * r3
    q, s, qT, sT = mx.mxfp8_quantize_2d(h, mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs)
    torch.cuda.synchronize()
    assert (u8(q) == u8(hq)).mean() >= 0.999
    assert (u8(qT) == u8(hTq)).mean() >= 0.999
    ends = sizes_to_ends(sizes)
    n_row = oracle.blocked_rowgroups_bytes(ends, H // 32)
    n_col = oracle.blocked_colgroups_bytes(H, ends)
    assert (u8(s)[:n_row] == u8(hs)[:n_row]).mean() >= 0.999
    assert (u8(sT)[:n_col] == u8(hTs)[:n_col]).mean() >= 0.999


def test_full_size_sampled(mx):
    """The SwiGLU expert's full gate/up shape (G=2, M=65600 as 39360 + 26240, D=5120, H=8192) in
    the launch configuration the bench times, sampled: row blocks of h (including the first and
    last row of each group) and token blocks of h^T, against the oracle's stage computed from the
    oracle's own dot products, with the random-input bars above; and byte for byte against the
    oracle's SwiGLU stage applied to the kernel's own h1, h3 on blocks without a silu rounding tie."""
    s = synth.workload("swiglu", seed=0, device="cuda")
    x, Wg, Wu, sizes = s["x"], s["Wg"], s["Wu"], s["sizes"]
    M, D, H = s["M"], s["D"], s["H"]
    ends = sizes_to_ends(sizes)
    starts = np.concatenate([[0], ends[:-1]])
    padded = np.concatenate([[0], np.cumsum([-(-int(m) // 128) * 128 for m in sizes])])
    (h1, h3, hq, hs, hTq, hTs), status = run_fused(mx, x, Wg, Wu, sizes)
    mx.read_status(status)
    rng = np.random.default_rng(12)
    xc, Wgc, Wuc = x.cpu(), Wg.cpu(), Wu.cpu()   # sampled rows are sliced on the host
    qx = {}

    def xrow(r):
        if r not in qx:
            qx[r] = oracle.quantize_rows(u16(xc[r:r + 1]))
        return qx[r]

    def h_oracle(r, g, cols):
        """The oracle's h1, h3 (fp64) and h (bf16 patterns) at row r, columns `cols`."""
        qa, sa = xrow(r)
        out = []
        for W in (Wgc, Wuc):
            qw, sw = oracle.quantize_rows(u16(W[g, cols[0]:cols[-1] + 1]))
            out.append(np.array([oracle.dot(qa[0], sa[0], qw[i], sw[i]) for i in range(len(cols))]))
        b1, b3 = oracle.bf16_from_f64(out[0]), oracle.bf16_from_f64(out[1])
        return out[0], out[1], oracle.swiglu_bf16(b1, b3)

    ref13, got13 = [], []
    q_o, q_g, s_o, s_g = [], [], [], []
    # the epilogue alone on the kernel's own bf16 h1, h3 of each sampled block (byte for byte on blocks
    # with no silu rounding tie)
    q_own, s_own, tie_own = [], [], []

    def own(b1, b3):
        qo, so = oracle.quantize_vec(oracle.swiglu_bf16(b1, b3))
        q_own.append(qo)
        s_own.append(so[0])
        tie_own.append(near_silu_ties(b1))

    rows = np.unique(np.concatenate([rng.integers(0, M, 10), starts, ends - 1]))
    for r in rows:
        r = int(r)
        g = int(np.searchsorted(ends, r, side="right"))
        j = int(rng.integers(0, H // 32))
        cols = list(range(32 * j, 32 * j + 32))
        o1, o3, h = h_oracle(r, g, cols)
        ref13 += [o1, o3]
        got13 += [f64(h1[r, 32 * j:32 * j + 32]), f64(h3[r, 32 * j:32 * j + 32])]
        qo, so = oracle.quantize_vec(h)
        q_o.append(qo)
        s_o.append(so[0])
        q_g.append(u8(hq[r, 32 * j:32 * j + 32]))
        own(u16(h1[r, 32 * j:32 * j + 32]), u16(h3[r, 32 * j:32 * j + 32]))
        pr = int(padded[g]) + r - int(starts[g])
        s_g.append(int(hs[oracle.blocked_offset(pr, j, H // 128)].item()))
    # token blocks of h^T: column c, 32 tokens of one group
    ct = int(padded[-1]) // 128
    for _ in range(6):
        g = int(rng.integers(0, len(sizes)))
        t0 = int(starts[g]) + 32 * int(rng.integers(0, sizes[g] // 32))
        c = int(rng.integers(0, H))
        hcol = np.array([h_oracle(t, g, [c])[2][0] for t in range(t0, t0 + 32)], np.uint16)
        qo, so = oracle.quantize_vec(hcol)
        q_o.append(qo)
        s_o.append(so[0])
        q_g.append(u8(hTq[c, t0:t0 + 32]))
        own(u16(h1[t0:t0 + 32, c]), u16(h3[t0:t0 + 32, c]))
        cq = int(padded[g]) // 32 + (t0 - int(starts[g])) // 32
        s_g.append(int(hTs[oracle.blocked_offset(c, cq, ct)].item()))
    assert_gemm_close(np.concatenate(got13), np.concatenate(ref13), what="h1/h3 sampled")
    q_o, q_g = np.stack(q_o), np.stack(q_g)
    s_o, s_g = np.array(s_o), np.array(s_g)
    tab = oracle.e4m3_table()
    dg = tab[q_g] * np.ldexp(1.0, s_g.astype(np.int64) - 127)[:, None]
    do = tab[q_o] * np.ldexp(1.0, s_o.astype(np.int64) - 127)[:, None]
    smax = np.maximum(s_g, s_o)[:, None].repeat(32, axis=1)
    assert np.all(np.abs(s_g.astype(int) - s_o.astype(int)) <= 1)
    assert np.all(np.abs(dg - do) <= e4m3_step(np.maximum(np.abs(dg), np.abs(do)), smax))
    assert (q_g == q_o).mean() >= 0.99 and (s_g == s_o).mean() >= 0.95
    clean = ~np.stack(tie_own).any(axis=1)
    assert clean.mean() > 0.8
    assert np.array_equal(np.array(s_own)[clean], s_g[clean]), "scales of tie-free blocks (own h1, h3)"
    assert np.array_equal(np.stack(q_own)[clean], q_g[clean]), "codes of tie-free blocks (own h1, h3)"
