"""Stability variants of the quantization ("MXFP8 (Micro-scaling FP8)", "Numerical stability":
random Hadamard transforms spread outliers before quantization; stochastic rounding removes the
bias of deterministic rounding) against the oracle, byte for byte.

Both sides draw the same Philox4x32-10 bytes (counter from the element's 2 x 8 block, key from the
seed; one byte per element, shared by its two copies) and evaluate the Hadamard butterflies in
fp32 in the same order, so codes and scales must agree exactly, padding of the blocked layouts
included.  The composite op's GEMMs
with these options are compared with the oracle's fp64 GEMMs of the oracle's operands within
the GEMM bound."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._util import assert_gemm_close, f64, require_gpu, sizes_to_ends, u8, u16

pytestmark = pytest.mark.gpu

SEED = 0x1234_5678_9ABC_DEF0


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def mixed_input(M, K, seed):
    """Rows of very different magnitude, tiny elements (the subnormal E4M3 range after scaling)
    and a few outliers."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, K), generator=g) * torch.pow(10.0, torch.rand((M, 1), generator=g) * 6 - 3)
    x[torch.rand((M, K), generator=g) < 0.05] *= 1e-3
    x[torch.rand((M, K), generator=g) < 0.01] *= 50.0
    return x.to(torch.bfloat16)


def oracle_opts(x, opts_gpu, seed):
    row_opts = (oracle.OPT_SR if opts_gpu & 1 else 0) | (oracle.OPT_RHT if opts_gpu & 2 else 0)
    col_opts = (oracle.OPT_SR if opts_gpu & 1 else 0) | (oracle.OPT_RHT if opts_gpu & 4 else 0)
    return oracle.quantize_rows_opts(u16(x), row_opts, seed), oracle.quantize_cols_opts(u16(x), col_opts, seed)


OPTS = [1, 2, 4, 2 | 4, 1 | 2, 1 | 4, 1 | 2 | 4]


@pytest.mark.parametrize("opts", OPTS)
def test_compact_both_directions(mx, opts):
    M, K = 256, 384
    x = mixed_input(M, K, seed=opts)
    q, s, qT, sT = [u8(t) for t in mx.mxfp8_quantize_2d(x.cuda(), mx.ROW | mx.COL, mx.SCALES_COMPACT,
                                                        opts=opts, seed=SEED)]
    (qo, so), (qTo, sTo) = oracle_opts(x, opts, SEED)
    assert np.array_equal(s, so) and np.array_equal(sT, sTo)
    assert np.array_equal(q, qo), f"{int((q != qo).sum())} row codes differ"
    assert np.array_equal(qT, qTo), f"{int((qT != qTo).sum())} column codes differ"


@pytest.mark.parametrize("dirs,opts", [(1, 1), (1, 3), (2, 1), (2, 5)])
def test_single_direction_equals_fused(mx, dirs, opts):
    x = mixed_input(128, 256, seed=40 + opts).cuda()
    a = mx.mxfp8_quantize_2d(x, mx.ROW | mx.COL, mx.SCALES_COMPACT, opts=opts, seed=SEED)
    b = mx.mxfp8_quantize_2d(x, dirs, mx.SCALES_COMPACT, opts=opts, seed=SEED)
    torch.cuda.synchronize()
    i = 0 if dirs == 1 else 2
    assert torch.equal(a[i], b[i]) and torch.equal(a[i + 1], b[i + 1])


@pytest.mark.parametrize("opts", [1, 4, 1 | 2 | 4])
def test_blocked_grouped(mx, opts):
    sizes = [96, 0, 160, 32]
    M, K = sum(sizes), 416   # K/32 = 13: a partial last scale tile
    x = mixed_input(M, K, seed=50 + opts)
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")
    q, s, qT, sT = [u8(t) for t in mx.mxfp8_quantize_2d(x.cuda(), mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs,
                                                        opts=opts, seed=SEED)]
    (qo, so), (qTo, sTo) = oracle_opts(x, opts, SEED)
    ends = sizes_to_ends(sizes)
    n_row = oracle.blocked_rowgroups_bytes(ends, K // 32)
    n_col = oracle.blocked_colgroups_bytes(K, ends)
    assert np.array_equal(q, qo) and np.array_equal(qT, qTo)
    assert np.array_equal(s[:n_row], oracle.blocked_rowgroups(so, ends))
    assert np.array_equal(sT[:n_col], oracle.blocked_colgroups(sTo, ends))


def special_values_input(M, K, seed):
    """mixed_input with blocks the stochastic-rounding paths treat apart: Inf / NaN (a non-finite
    block keeps its replaced codes), whole blocks of bf16 subnormals (scale byte 0, codes from the
    normal E4M3 range), signed zeros, and elements at 2^-17 .. 2^-6 after scaling (the E4M3
    subnormal range, where the exact rule decides)."""
    x = mixed_input(M, K, seed).float()
    x[0, 5], x[3, 40], x[70, 64] = float("inf"), float("nan"), -float("inf")
    x[100:132, 200] = float("nan")
    i = torch.arange(32, dtype=torch.float32)
    sub = torch.ldexp(1.0 + i / 32.0, -127.0 - (i % 7))                     # [2^-133, 2^-126): bf16 subnormals
    x[10, :32] = sub * torch.where(i % 3 == 0, -1.0, 1.0)
    x[32:64, 96] = sub
    x[11, :] = 0.0
    x[12, :32] = -0.0
    # one element at 256 * 2^e (the block amax), the others at 2^-17 .. 2^-5 of it (scaled: 2^-9 .. 2^3)
    x[13, 32:64] = torch.ldexp(torch.full((32,), 1.5), 8.0 - i)
    x[14, 64:96] = -x[13, 32:64]
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("dirs", [1, 2, 3])
def test_sr_special_values(mx, dirs):
    """Stochastic rounding alone runs a packed bf16 path with an exact pass for the E4M3 subnormal
    range: both against the oracle on special blocks, codes and scales byte for byte."""
    M, K = 256, 384
    x = special_values_input(M, K, seed=70 + dirs)
    out = mx.mxfp8_quantize_2d(x.cuda(), dirs, mx.SCALES_COMPACT, opts=1, seed=SEED)
    (qo, so), (qTo, sTo) = oracle_opts(x, 1, SEED)
    if dirs & 1:
        q, s = u8(out[0]), u8(out[1])
        assert np.array_equal(s, so)
        assert np.array_equal(q, qo), f"{int((q != qo).sum())} row codes differ"
    if dirs & 2:
        qT, sT = u8(out[2]), u8(out[3])
        assert np.array_equal(sT, sTo)
        assert np.array_equal(qT, qTo), f"{int((qT != qTo).sum())} column codes differ"


def test_seed_changes_only_what_it_keys(mx):
    x = mixed_input(64, 128, seed=60).cuda()
    a = mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT, opts=1, seed=1)
    b = mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT, opts=1, seed=2)
    c = mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT, opts=1, seed=1)
    torch.cuda.synchronize()
    assert torch.equal(a[0], c[0]) and not torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_option_errors(mx):
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    for dirs, opts in ((mx.ROW, mx.OPT_HADAMARD_COL), (mx.COL, mx.OPT_HADAMARD_ROW), (mx.ROW, 8),
                       (mx.BLOCK32X32, mx.OPT_STOCHASTIC)):
        with pytest.raises(mx.Mxfp8Error, match="LAYOUT"):
            mx.mxfp8_quantize_2d(x, dirs, mx.SCALES_COMPACT, opts=opts, seed=1)


def test_composite_with_stability_options(mx):
    sizes = [128, 64, 0, 96]
    G, N, K = len(sizes), 128, 256
    M = sum(sizes)
    A = mixed_input(M, K, seed=70)
    W = synth.randn_bf16((G, N, K), 0.02, seed=71)
    dO = synth.randn_bf16((M, N), 1e-2, seed=72)
    offs = torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")
    Ag, Wg = A.cuda().requires_grad_(True), W.cuda().requires_grad_(True)
    out = mx.to_mxfp8_then_scaled_grouped_mm(Ag, Wg, offs, stochastic_rounding=True, hadamard_wgrad=True, seed=SEED)
    out.backward(dO.cuda())
    torch.cuda.synchronize()
    ends = sizes_to_ends(sizes)
    # dgrad: dOut rounded stochastically along N
    dq, ds = oracle.quantize_rows_opts(u16(dO), oracle.OPT_SR, SEED)
    wTq, wTs = zip(*[oracle.quantize_cols(u16(W[g])) for g in range(G)])
    assert_gemm_close(f64(Ag.grad), oracle.grouped_mm_rows(dq, ds, np.stack(wTq), np.stack(wTs), ends), what="dA")
    # wgrad: both operands Hadamard-transformed along the tokens with the same seed, dOut also SR
    dTq, dTs = oracle.quantize_cols_opts(u16(dO), oracle.OPT_SR | oracle.OPT_RHT, SEED)
    aTq, aTs = oracle.quantize_cols_opts(u16(A), oracle.OPT_RHT, SEED)
    ref_dw = oracle.grouped_mm_wgrad(dTq, dTs, aTq, aTs, ends)
    assert_gemm_close(f64(Wg.grad), ref_dw, what="dW")
    # the transform is orthogonal, so the wgrad still approximates dOut^T A: against the fp64
    # product of the unquantized inputs it is about as accurate as the plain MXFP8 wgrad (a sign
    # vector that differed between the two operands would leave an error near 100%)
    exact = np.zeros_like(ref_dw)
    lo = 0
    for g, hi in enumerate(ends):
        exact[g] = f64(dO)[lo:hi].T @ f64(A)[lo:hi]
        lo = int(hi)
    Ap, Wp = A.cuda().requires_grad_(True), W.cuda().requires_grad_(True)
    mx.to_mxfp8_then_scaled_grouped_mm(Ap, Wp, offs).backward(dO.cuda())
    torch.cuda.synchronize()
    rel = lambda got: np.linalg.norm(f64(got) - exact) / np.linalg.norm(exact)
    assert rel(Wg.grad) < max(2.0 * rel(Wp.grad), 0.02), (rel(Wg.grad), rel(Wp.grad))


def test_full_size_grouped_sampled(mx):
    """The Scout activations' shape [16384, 5120] with its 8 token groups, every option at once
    (stochastic rounding, Hadamard on both copies), sampled blocks against the oracle."""
    sizes = synth.scout_group_sizes(0)
    M, K = 16384, 5120
    x = synth.log_uniform_rows(M, K, seed=3, device="cuda")
    ends = sizes_to_ends(sizes)
    starts = np.concatenate([[0], ends[:-1]])
    offs = torch.tensor(ends.astype(np.int32), device="cuda")
    opts = mx.OPT_STOCHASTIC | mx.OPT_HADAMARD_ROW | mx.OPT_HADAMARD_COL
    st = mx.new_status()
    q, s, qT, sT = mx.mxfp8_quantize_2d(x, mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs, st, opts=opts, seed=SEED)
    mx.read_status(st)
    o_opts = oracle.OPT_SR | oracle.OPT_RHT
    padded = np.concatenate([[0], np.cumsum([-(-int(m) // 128) * 128 for m in sizes])])
    group_of = lambda r: int(np.searchsorted(ends, r, side="right"))
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), ends[np.array(sizes) > 0] - 1]))
    for r in rows:
        g = group_of(int(r))
        pr = padded[g] + int(r) - starts[g]
        for b in rng.integers(0, K // 32, 3):
            qo, so = oracle.quantize_block_at(u16(x[r, 32 * b:32 * b + 32]), int(r), 32 * int(b), False, K, o_opts, SEED)
            assert np.array_equal(u8(q[r, 32 * b:32 * b + 32]), qo)
            assert int(s[oracle.blocked_offset(int(pr), int(b), K // 128)].item()) == so
    ct = int(padded[-1]) // 128
    for c in rng.integers(0, K, 12):
        g = int(rng.integers(0, len(sizes)))
        if sizes[g] == 0:
            continue
        t0 = int(starts[g]) + 32 * int(rng.integers(0, sizes[g] // 32))
        qo, so = oracle.quantize_block_at(np.ascontiguousarray(u16(x[t0:t0 + 32, c])), t0, int(c), True, K, o_opts,
                                          SEED)
        assert np.array_equal(u8(qT[c, t0:t0 + 32]), qo)
        cq = padded[g] // 32 + (t0 - starts[g]) // 32
        assert int(sT[oracle.blocked_offset(int(c), int(cq), ct)].item()) == so
