"""GPU parity of the block-scaled grouped GEMMs (fwd, dgrad, wgrad) and the
composite differentiable op against the fp64 CPU oracle.

Acceptance: |gpu - o| <= 1e-2 |o| + 1e-3 rms(o) elementwise (rms over the whole
reference tensor, or over the sample at full size).  The GPU and the oracle
each quantize the same bf16 inputs themselves (the quantization is bit-exact,
see test_gpu_quantize.py).  Special cases: identity weights (the product equals
the dequantized activations exactly), one group == dense GEMM, empty groups
(no rows; zero dW), ragged groups, ragged N and K tails.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._util import assert_gemm_close, f64, require_gpu, sizes_to_ends, sqnr_db, u8, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def offs_dev(sizes):
    return torch.tensor(sizes_to_ends(sizes).astype(np.int32), device="cuda")


def gpu_fwd(mx, A, W, sizes):
    st = mx.new_status()
    offs = offs_dev(sizes)
    aq, as_, _, _ = mx.mxfp8_quantize_2d(A.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)
    wq, ws, _, _ = mx.mxfp8_quantize_3d_experts(W.cuda(), mx.ROW, mx.SCALES_BLOCKED, st)
    out = mx.mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs, dev_status=st)
    mx.read_status(st)
    return f64(out)


def gpu_dgrad(mx, D, W, sizes):
    st = mx.new_status()
    offs = offs_dev(sizes)
    dq, ds, _, _ = mx.mxfp8_quantize_2d(D.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)
    _, _, wTq, wTs = mx.mxfp8_quantize_3d_experts(W.cuda(), mx.COL, mx.SCALES_BLOCKED, st)
    out = mx.mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs, dev_status=st)
    mx.read_status(st)
    return f64(out)


def gpu_wgrad(mx, D, A, sizes):
    st = mx.new_status()
    offs = offs_dev(sizes)
    _, _, dTq, dTs = mx.mxfp8_quantize_2d(D.cuda(), mx.COL, mx.SCALES_BLOCKED, offs, st)
    _, _, aTq, aTs = mx.mxfp8_quantize_2d(A.cuda(), mx.COL, mx.SCALES_BLOCKED, offs, st)
    out = mx.mxfp8_grouped_mm_wgrad(dTq, dTs, aTq, aTs, offs, dev_status=st)
    mx.read_status(st)
    return f64(out)


def oracle_fwd(A, W, sizes):
    aq, as_ = oracle.quantize_rows(u16(A))
    wq, ws = zip(*[oracle.quantize_rows(u16(W[g])) for g in range(W.shape[0])])
    return oracle.grouped_mm_rows(aq, as_, np.stack(wq), np.stack(ws), sizes_to_ends(sizes))


def oracle_dgrad(D, W, sizes):
    dq, ds = oracle.quantize_rows(u16(D))
    wTq, wTs = zip(*[oracle.quantize_cols(u16(W[g])) for g in range(W.shape[0])])  # [K, N] per expert
    return oracle.grouped_mm_rows(dq, ds, np.stack(wTq), np.stack(wTs), sizes_to_ends(sizes))


def oracle_wgrad(D, A, sizes):
    dTq, dTs = oracle.quantize_cols(u16(D))
    aTq, aTs = oracle.quantize_cols(u16(A))
    return oracle.grouped_mm_wgrad(dTq, dTs, aTq, aTs, sizes_to_ends(sizes))


# (sizes, N, K): several tiles, ragged group tails (fwd/dgrad accept any size),
# N and K tails that are not multiples of the 256 / 128 tile.
FWD_CASES = [
    ([128, 128], 128, 256),
    ([200, 0, 64, 333, 31], 384, 320),
    ([0, 517, 0], 256, 1056),
    ([1, 127, 129, 255], 96, 224),
    ([640], 544, 160),
]


@pytest.mark.parametrize("sizes,N,K", FWD_CASES)
def test_fwd(mx, sizes, N, K):
    M, G = sum(sizes), len(sizes)
    A = synth.randn_bf16((M, K), 1.0, seed=M + N)
    W = synth.randn_bf16((G, N, K), 0.02, seed=K + G)
    got = gpu_fwd(mx, A, W, sizes)
    ref = oracle_fwd(A, W, sizes)
    assert_gemm_close(got, ref, what="fwd")


@pytest.mark.parametrize("sizes,N,K", FWD_CASES)
def test_dgrad(mx, sizes, N, K):
    M, G = sum(sizes), len(sizes)
    D = synth.randn_bf16((M, N), 1e-3, seed=M + 2 * N)
    W = synth.randn_bf16((G, N, K), 0.02, seed=K + 3 * G)
    got = gpu_dgrad(mx, D, W, sizes)
    ref = oracle_dgrad(D, W, sizes)
    assert_gemm_close(got, ref, what="dgrad")


WGRAD_CASES = [
    ([128, 128], 128, 256),
    ([96, 0, 160, 32, 256], 160, 288),
    ([0, 544, 0], 256, 512),
    ([32], 64, 32),
    ([384, 128, 0, 32], 416, 96),
]


@pytest.mark.parametrize("sizes,N,K", WGRAD_CASES)
def test_wgrad(mx, sizes, N, K):
    M = sum(sizes)
    D = synth.randn_bf16((M, N), 1e-3, seed=M + 5 * N)
    A = synth.randn_bf16((M, K), 1.0, seed=K + 7)
    got = gpu_wgrad(mx, D, A, sizes)
    ref = oracle_wgrad(D, A, sizes)
    for g, m in enumerate(sizes):
        if m == 0:
            assert np.all(got[g] == 0.0), f"empty group {g} must give zero dW"
    assert_gemm_close(got, ref, what="wgrad")


@pytest.mark.parametrize("G", [100, 140])
def test_wgrad_many_groups(mx, G):
    """Many small token groups (multiples of 32, a fifth of them empty) through the CTA-pair wgrad:
    G <= 128 runs the schedule that ranks groups by size (ties between equal sizes included),
    G > 128 the plain round-robin one.  Every group's dW against the oracle; empty groups zero."""
    rng = np.random.default_rng(G)
    sizes = [int(x) for x in rng.integers(0, 6, G) * 32]
    for g in rng.choice(G, G // 5, replace=False):
        sizes[int(g)] = 0
    M, N, K = sum(sizes), 160, 288   # N = 160: the pair's second CTA holds 32 valid rows
    D = synth.randn_bf16((M, N), 1e-3, seed=G + 11)
    A = synth.randn_bf16((M, K), 1.0, seed=G + 13)
    got = gpu_wgrad(mx, D, A, sizes)
    ref = oracle_wgrad(D, A, sizes)
    for g, m in enumerate(sizes):
        if m == 0:
            assert np.all(got[g] == 0.0), f"empty group {g} must give zero dW"
    assert_gemm_close(got, ref, what=f"wgrad G={G}")


def test_max_groups(mx):
    """MXFP8_MAX_GROUPS (1024) groups, a quarter of them empty: the group tables of the quantize and
    GEMM kernels at full capacity.  fwd and dgrad take groups of any size; the wgrad and the
    column-wise quantization groups of multiples of 32 (the token blocks).  GEMMs within the bound
    (references by the oracle's matmul forms, pinned to its scalar loops on the CPU), quantization
    byte for byte in both blocked layouts, empty groups zero dW."""
    G, N, K = 1024, 32, 256   # K >= 256: the wgrad runs the CTA-pair kernel
    rng = np.random.default_rng(1024)
    W = synth.randn_bf16((G, N, K), 0.05, seed=1)
    sizes = [int(x) for x in rng.integers(1, 48, G)]
    sizes32 = [32] * G
    for g in rng.choice(G, G // 4, replace=False):
        sizes[int(g)] = 0
        sizes32[int(g)] = 0
    M, M32 = sum(sizes), sum(sizes32)
    A = synth.randn_bf16((M, K), 1.0, seed=2)
    D = synth.randn_bf16((M, N), 1e-2, seed=3)
    ends_any = sizes_to_ends(sizes)
    wq, ws = zip(*[oracle.quantize_rows(u16(W[g])) for g in range(G)])
    wTq, wTs = zip(*[oracle.quantize_cols(u16(W[g])) for g in range(G)])
    aq, as_ = oracle.quantize_rows(u16(A))
    dq, ds = oracle.quantize_rows(u16(D))
    ref_fwd = oracle.grouped_mm_rows_blas(aq, as_, np.stack(wq), np.stack(ws), ends_any)
    ref_dgrad = oracle.grouped_mm_rows_blas(dq, ds, np.stack(wTq), np.stack(wTs), ends_any)
    assert_gemm_close(gpu_fwd(mx, A, W, sizes), ref_fwd, what="fwd G=1024")
    assert_gemm_close(gpu_dgrad(mx, D, W, sizes), ref_dgrad, what="dgrad G=1024")
    A32 = synth.randn_bf16((M32, K), 1.0, seed=4)
    D32 = synth.randn_bf16((M32, N), 1e-2, seed=5)
    got = gpu_wgrad(mx, D32, A32, sizes32)
    for g, m in enumerate(sizes32):
        if m == 0:
            assert np.all(got[g] == 0.0), f"empty group {g} must give zero dW"
    dTq, dTs = oracle.quantize_cols(u16(D32))
    aTq, aTs = oracle.quantize_cols(u16(A32))
    ref_wgrad = oracle.grouped_mm_wgrad_blas(dTq, dTs, aTq, aTs, sizes_to_ends(sizes32))
    assert_gemm_close(got, ref_wgrad, what="wgrad G=1024")
    ends = sizes_to_ends(sizes32)
    q, s, qT, sT = [u8(t) for t in mx.mxfp8_quantize_2d(A32.cuda(), mx.ROW | mx.COL, mx.SCALES_BLOCKED,
                                                        offs_dev(sizes32))]
    qo, so = oracle.quantize_rows(u16(A32))
    qTo, sTo = oracle.quantize_cols(u16(A32))
    assert np.array_equal(q, qo) and np.array_equal(qT, qTo)
    n_row, n_col = oracle.blocked_rowgroups_bytes(ends, K // 32), oracle.blocked_colgroups_bytes(K, ends)
    assert np.array_equal(s[:n_row], oracle.blocked_rowgroups(so, ends))
    assert np.array_equal(sT[:n_col], oracle.blocked_colgroups(sTo, ends))


def test_max_groups_pair_rowgrouped(mx):
    """1024 ragged groups (a quarter empty) through the CTA-pair fwd and dgrad: N = 288 is one
    256-wide pair tile plus a 32-column tail whose B rows past N read TMA's zero fill; K = 160
    ends in a partial k-tile."""
    G, N, K = 1024, 288, 160
    rng = np.random.default_rng(2048)
    sizes = [int(x) for x in rng.integers(1, 40, G)]
    for g in rng.choice(G, G // 4, replace=False):
        sizes[int(g)] = 0
    M = sum(sizes)
    W = synth.randn_bf16((G, N, K), 0.05, seed=7)
    A = synth.randn_bf16((M, K), 1.0, seed=8)
    D = synth.randn_bf16((M, N), 1e-2, seed=9)
    ends = sizes_to_ends(sizes)
    wq, ws = zip(*[oracle.quantize_rows(u16(W[g])) for g in range(G)])
    wTq, wTs = zip(*[oracle.quantize_cols(u16(W[g])) for g in range(G)])
    aq, as_ = oracle.quantize_rows(u16(A))
    dq, ds = oracle.quantize_rows(u16(D))
    assert_gemm_close(gpu_fwd(mx, A, W, sizes), oracle.grouped_mm_rows_blas(aq, as_, np.stack(wq), np.stack(ws), ends),
                      what="pair fwd G=1024")
    assert_gemm_close(gpu_dgrad(mx, D, W, sizes),
                      oracle.grouped_mm_rows_blas(dq, ds, np.stack(wTq), np.stack(wTs), ends), what="pair dgrad G=1024")


def test_identity_weights_exact(mx):
    """W[g] = I: every weight scale is 2^-8 and every diagonal code 256, so the
    product is the dequantized activation, exact in fp32; bf16 rounding of that
    value is the only step, and it must equal the oracle's bf16 rounding."""
    K = 256
    sizes = [100, 156]
    rng = np.random.default_rng(1)
    A = torch.tensor(rng.standard_normal((256, K)) * 3, dtype=torch.float32).to(torch.bfloat16)
    W = torch.eye(K).repeat(2, 1, 1).to(torch.bfloat16)
    got = gpu_fwd(mx, A, W, sizes)
    aq, as_ = oracle.quantize_rows(u16(A))
    deq = oracle.dequant(aq, np.repeat(as_, 32, axis=1))
    want = torch.tensor(deq, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)


def test_single_group_equals_dense(mx):
    M, N, K = 384, 256, 512
    A = synth.randn_bf16((M, K), 1.0, seed=21)
    W = synth.randn_bf16((1, N, K), 0.02, seed=22)
    got = gpu_fwd(mx, A, W, [M])
    aq, as_ = oracle.quantize_rows(u16(A))
    wq, ws = oracle.quantize_rows(u16(W[0]))
    dense = oracle.dequant(aq, np.repeat(as_, 32, 1)) @ oracle.dequant(wq, np.repeat(ws, 32, 1)).T
    assert_gemm_close(got, dense, what="G=1 dense")


def test_tiny_config_composite_fwd_bwd(mx):
    """The tiny workload through the differentiable op, stage by stage against the oracle."""
    w = synth.workload("tiny", seed=0)
    A = w["A"].cuda().requires_grad_(True)
    W = w["W"].cuda().requires_grad_(True)
    offs = w["offs"].cuda()
    out = mx.to_mxfp8_then_scaled_grouped_mm(A, W, offs)
    out.backward(w["dOut"].cuda())
    torch.cuda.synchronize()
    assert_gemm_close(f64(out), oracle_fwd(w["A"], w["W"], w["sizes"]), what="composite fwd")
    assert_gemm_close(f64(A.grad), oracle_dgrad(w["dOut"], w["W"], w["sizes"]), what="composite dA")
    assert_gemm_close(f64(W.grad), oracle_wgrad(w["dOut"], w["A"], w["sizes"]), what="composite dW")
    # information only: MXFP8 vs the unquantized product
    ref = w["A"].double() @ w["W"][0].double().T
    assert sqnr_db(ref[:128].numpy(), f64(out)[:128]) > 20.0


# ---------------------------------------------------------------- full-size workloads, sampled
def _pairs(rows, cols, n, seed):
    rng = np.random.default_rng(seed)
    return rng.choice(rows, n), rng.choice(cols, n)


def _full_case(name):
    if name == "scout":
        return synth.workload("scout", seed=0, device="cuda")
    if name == "imbalanced":
        return synth.workload("imbalanced", seed=0, device="cuda")
    raise KeyError(name)


@pytest.mark.parametrize("name", ["scout", "imbalanced"])
def test_full_size_fwd_dgrad_wgrad_sampled(mx, name):
    w = _full_case(name)
    A, W, D, sizes = w["A"], w["W"], w["dOut"], w["sizes"]
    M, N, K, G = w["M"], w["N"], w["K"], w["G"]
    offs = w["offs"].cuda()
    ends = sizes_to_ends(sizes)
    starts = np.concatenate([[0], ends[:-1]])
    st = mx.new_status()
    aq, as_, aTq, aTs = mx.mxfp8_quantize_2d(A, mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs, st)
    wq, ws, wTq, wTs = mx.mxfp8_quantize_3d_experts(W, mx.ROW | mx.COL, mx.SCALES_BLOCKED, st)
    dq, ds, dTq, dTs = mx.mxfp8_quantize_2d(D, mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs, st)
    out = mx.mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs, dev_status=st)
    dA = mx.mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs, dev_status=st)
    dW = mx.mxfp8_grouped_mm_wgrad(dTq, dTs, aTq, aTs, offs, dev_status=st)
    mx.read_status(st)

    # rows: random plus the first and last row of every non-empty group
    rng = np.random.default_rng(0)
    edge = np.concatenate([starts[np.array(sizes) > 0], ends[np.array(sizes) > 0] - 1])
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), edge]))
    group_of = lambda r: int(np.searchsorted(ends, r, side="right"))
    # forward: out[m, n]
    ncols = np.unique(np.concatenate([rng.integers(0, N, 12), [0, N - 1]]))
    ref, got = [], []
    for r in rows:
        g = group_of(r)
        qa, sa = oracle.quantize_rows(u16(A[r:r + 1]))
        for n in ncols:
            qw, sw = oracle.quantize_rows(u16(W[g, n:n + 1]))
            ref.append(oracle.dot(qa[0], sa[0], qw[0], sw[0]))
        got.append(f64(out[r, torch.as_tensor(ncols, device="cuda")]))
    ref = np.array(ref)
    assert_gemm_close(np.concatenate(got), ref, what=f"{name} fwd sampled")
    # dgrad: dA[m, k] = sum_n dOut[m, n] W[g][n, k]
    kcols = np.unique(np.concatenate([rng.integers(0, K, 8), [0, K - 1]]))
    ref, got = [], []
    for r in rows:
        g = group_of(r)
        qd, sd = oracle.quantize_rows(u16(D[r:r + 1]))
        for k in kcols:
            qw, sw = oracle.quantize_vec(u16(W[g, :, k]))
            ref.append(oracle.dot(qd[0], sd[0], qw, sw))
        got.append(f64(dA[r, torch.as_tensor(kcols, device="cuda")]))
    assert_gemm_close(np.concatenate(got), np.array(ref), what=f"{name} dgrad sampled")
    # wgrad: dW[g][n, k] over the group's tokens; empty groups all zero
    for g in range(G):
        lo, hi = int(starts[g]), int(ends[g])
        if hi == lo:
            assert int(torch.count_nonzero(dW[g]).item()) == 0
            continue
        ns = rng.integers(0, N, 4)
        ks = rng.integers(0, K, 4)
        ref, gv = [], []
        for n in ns:
            qd, sd = oracle.quantize_vec(u16(D[lo:hi, n]))
            for k in ks:
                qa, sa = oracle.quantize_vec(u16(A[lo:hi, k]))
                ref.append(oracle.dot(qd, sd, qa, sa))
                gv.append(float(dW[g, n, k].item()))
        assert_gemm_close(np.array(gv), np.array(ref), rms=float(np.sqrt(np.mean(np.square(ref)))),
                          what=f"{name} wgrad group {g}")


def test_full_size_swiglu_gemm_shapes_sampled(mx):
    """The SwiGLU expert's two GEMM shapes (gate/up: N=8192, K=5120; down: N=5120,
    K=8192) at M=65600 split 39360/26240, forward, sampled."""
    sizes = synth.swiglu_group_sizes()
    M = sum(sizes)
    offs = offs_dev(sizes)
    ends = sizes_to_ends(sizes)
    rng = np.random.default_rng(1)
    for N, K, seed in ((8192, 5120, 1), (5120, 8192, 2)):
        A = synth.randn_bf16((M, K), 1.0, seed, device="cuda")
        W = synth.randn_bf16((2, N, K), 0.02, seed + 10, device="cuda")
        st = mx.new_status()
        aq, as_, _, _ = mx.mxfp8_quantize_2d(A, mx.ROW, mx.SCALES_BLOCKED, offs, st)
        wq, ws, _, _ = mx.mxfp8_quantize_3d_experts(W, mx.ROW, mx.SCALES_BLOCKED, st)
        out = mx.mxfp8_grouped_mm_fwd(aq, as_, wq, ws, offs, dev_status=st)
        mx.read_status(st)
        rows = np.unique(np.concatenate([rng.integers(0, M, 16), [0, ends[0] - 1, ends[0], M - 1]]))
        ref, got = [], []
        for r in rows:
            g = int(np.searchsorted(ends, r, side="right"))
            qa, sa = oracle.quantize_rows(u16(A[r:r + 1]))
            for n in rng.integers(0, N, 6):
                qw, sw = oracle.quantize_rows(u16(W[g, n:n + 1]))
                ref.append(oracle.dot(qa[0], sa[0], qw[0], sw[0]))
                got.append(float(out[r, n].item()))
        assert_gemm_close(np.array(got), np.array(ref), what=f"swiglu fwd N={N} K={K}")
        del A, W, aq, as_, wq, ws, out


def test_wgrad_rejects_misaligned_group_offsets(mx):
    """Token groups that are not multiples of 32 would put a TMA coordinate off its 16-byte
    alignment in the wgrad; the kernel checks the offsets before any copy, reports
    MXFP8_ERR_OFFSETS and issues nothing (host-side fault injection: the offsets are bad, no
    device fault is provoked)."""
    M, N, K = 256, 256, 256
    dTq = torch.zeros((N, M), dtype=torch.uint8, device="cuda")
    aTq = torch.zeros((K, M), dtype=torch.uint8, device="cuda")
    s1 = torch.zeros(mx.mxfp8_scale_bytes_colgroups(N, M, 2), dtype=torch.uint8, device="cuda")
    s2 = torch.zeros(mx.mxfp8_scale_bytes_colgroups(K, M, 2), dtype=torch.uint8, device="cuda")
    bad = torch.tensor([100, 256], dtype=torch.int32, device="cuda")
    st = mx.new_status()
    mx.mxfp8_grouped_mm_wgrad(dTq, s1, aTq, s2, bad, dev_status=st)
    assert int(st.item()) == 7
    # the context stays usable
    x = torch.ones((32, 32), dtype=torch.bfloat16, device="cuda")
    q, s, _, _ = mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT)
    assert int(q[0, 0].item()) == 0x78


def test_full_size_swiglu_dgrad_wgrad_sampled(mx):
    """The SwiGLU gate shapes (N=8192, K=5120, M=65600 in two groups), dgrad and wgrad, sampled."""
    sizes = synth.swiglu_group_sizes()
    M, N, K = sum(sizes), 8192, 5120
    offs = offs_dev(sizes)
    ends = sizes_to_ends(sizes)
    starts = ends - np.asarray(sizes)
    A = synth.randn_bf16((M, K), 1.0, 5, device="cuda")
    W = synth.randn_bf16((2, N, K), 0.02, 6, device="cuda")
    D = synth.randn_bf16((M, N), 1e-3, 7, device="cuda")
    st = mx.new_status()
    _, _, aTq, aTs = mx.mxfp8_quantize_2d(A, mx.COL, mx.SCALES_BLOCKED, offs, st)
    _, _, wTq, wTs = mx.mxfp8_quantize_3d_experts(W, mx.COL, mx.SCALES_BLOCKED, st)
    dq, ds, dTq, dTs = mx.mxfp8_quantize_2d(D, mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs, st)
    dA = mx.mxfp8_grouped_mm_dgrad(dq, ds, wTq, wTs, offs, dev_status=st)
    dW = mx.mxfp8_grouped_mm_wgrad(dTq, dTs, aTq, aTs, offs, dev_status=st)
    mx.read_status(st)
    rng = np.random.default_rng(3)
    ref, got = [], []
    for r in np.unique(np.concatenate([rng.integers(0, M, 10), [0, ends[0] - 1, ends[0], M - 1]])):
        g = int(np.searchsorted(ends, r, side="right"))
        qd, sd = oracle.quantize_rows(u16(D[r:r + 1]))
        for k in rng.integers(0, K, 4):
            qw, sw = oracle.quantize_vec(u16(W[g, :, k]))
            ref.append(oracle.dot(qd[0], sd[0], qw, sw))
            got.append(float(dA[r, k].item()))
    assert_gemm_close(np.array(got), np.array(ref), what="swiglu dgrad sampled")
    for g in range(2):
        lo, hi = int(starts[g]), int(ends[g])
        ref, got = [], []
        for n in rng.integers(0, N, 3):
            q1, s1 = oracle.quantize_vec(u16(D[lo:hi, n]))
            for k in rng.integers(0, K, 3):
                q2, s2 = oracle.quantize_vec(u16(A[lo:hi, k]))
                ref.append(oracle.dot(q1, s1, q2, s2))
                got.append(float(dW[g, n, k].item()))
        assert_gemm_close(np.array(got), np.array(ref), rms=float(np.sqrt(np.mean(np.square(ref)))),
                          what=f"swiglu wgrad group {g}")


def test_bounded_wait_times_out_cleanly(mx):
    """A wait on a barrier nothing arrives on returns MXFP8_ERR_TIMEOUT after its
    limit instead of hanging, and the context stays usable afterwards."""
    st = mx.new_status()
    mx.mxfp8_debug_wait_timeout(st, 50_000_000)  # 50 ms
    assert int(st.item()) == 8
    x = torch.ones((32, 32), dtype=torch.bfloat16, device="cuda")
    q, s, _, _ = mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT)
    assert int(s[0, 0].item()) == 0x77 and int(q[0, 0].item()) == 0x78


def test_dgrad2_equals_the_sum_of_two_dgrads(mx):
    """dA = dOut1 W1 + dOut2 W2 in one GEMM (the SwiGLU expert's dx = dh1 Wg + dh3 Wu) against the
    oracle's two fp64 dgrads summed, within the GEMM bound; empty and ragged groups included."""
    sizes = [96, 0, 160, 64]
    G, N, K = len(sizes), 256, 384
    M = sum(sizes)
    ends = sizes_to_ends(sizes)
    offs = offs_dev(sizes)
    D1, D2 = synth.randn_bf16((M, N), 1.0, seed=41), synth.randn_bf16((M, N), 1.0, seed=42)
    W1, W2 = synth.randn_bf16((G, N, K), 0.02, seed=43), synth.randn_bf16((G, N, K), 0.02, seed=44)
    st = mx.new_status()
    q = [mx.mxfp8_quantize_2d(D.cuda(), mx.ROW, mx.SCALES_BLOCKED, offs, st)[:2] for D in (D1, D2)]
    wt = [mx.mxfp8_quantize_3d_experts(W.cuda(), mx.COL, mx.SCALES_BLOCKED, st)[2:] for W in (W1, W2)]
    dA = mx.mxfp8_grouped_mm_dgrad2(*q[0], *wt[0], *q[1], *wt[1], offs, dev_status=st)
    mx.read_status(st)
    ref = 0
    for D, W in ((D1, W1), (D2, W2)):
        dq, ds = oracle.quantize_rows(u16(D))
        wTq, wTs = zip(*[oracle.quantize_cols(u16(W[g])) for g in range(G)])
        ref = ref + oracle.grouped_mm_rows(dq, ds, np.stack(wTq), np.stack(wTs), ends)
    assert_gemm_close(f64(dA), ref, what="dgrad2")
    with pytest.raises(ValueError):
        mx.mxfp8_grouped_mm_dgrad2(*q[0], *wt[0], q[1][0][:, :128].contiguous(), q[1][1], *wt[1], offs)


@pytest.mark.parametrize("N,K", [(256, 256), (160, 128)])
def test_wgrad_next_group_nonfinite_does_not_leak(mx, N, K):
    """A group whose size is a multiple of 32 but not of 128 ends inside a 128-token copy box; the
    box's remaining columns hold the next group's tokens.  With Inf/NaN in the next group's first
    tokens (their column blocks quantize to NaN codes), the group's own dW must stay finite and
    equal the oracle's, which sums over the group's tokens only ("grouped result equals per-group
    dense GEMMs").  K = 256: the CTA-pair kernel; K = 128: the single-CTA kernel."""
    sizes = [96, 64, 160]
    M = sum(sizes)
    D = synth.randn_bf16((M, N), 1e-3, seed=401).float()
    A = synth.randn_bf16((M, K), 1.0, seed=402).float()
    D[96, 5], D[97, :] = float("nan"), float("inf")   # first tokens of group 1
    A[96, 7], A[100, 3] = -float("inf"), float("nan")
    D, A = D.to(torch.bfloat16), A.to(torch.bfloat16)
    got = gpu_wgrad(mx, D, A, sizes)
    ref = oracle_wgrad(D, A, sizes)
    for g in (0, 2):
        assert np.all(np.isfinite(got[g])), f"group {g}: non-finite values leaked from the next group"
        assert_gemm_close(got[g], ref[g], what=f"wgrad group {g} beside a non-finite group")
    assert not np.all(np.isfinite(got[1]))  # the group that holds them does see them


def test_composite_op_rejects_bad_offsets(mx):
    """Group sizes that are not multiples of 32 cannot be quantized along the tokens for the wgrad:
    with W requiring a gradient the composite op raises instead of returning the outputs the
    kernels skipped; with only A requiring one, the same offsets run (fwd and dgrad take any
    size).  Offsets that do not end at M raise too."""
    sizes = [48, 80]
    M, N, K = sum(sizes), 128, 128
    A = synth.randn_bf16((M, K), 1.0, seed=411)
    W = synth.randn_bf16((2, N, K), 0.02, seed=412)
    offs = offs_dev(sizes)
    with pytest.raises(mx.Mxfp8Error, match="OFFSETS"):
        mx.to_mxfp8_then_scaled_grouped_mm(A.cuda().requires_grad_(True), W.cuda().requires_grad_(True), offs)
    a = A.cuda().requires_grad_(True)
    out = mx.to_mxfp8_then_scaled_grouped_mm(a, W.cuda(), offs)
    out.backward(synth.randn_bf16((M, N), 1e-3, seed=413).cuda())
    torch.cuda.synchronize()
    assert_gemm_close(f64(out), oracle_fwd(A, W, sizes), what="fwd with 48/80-token groups")
    short = torch.tensor([48, 100], dtype=torch.int32, device="cuda")
    with pytest.raises(mx.Mxfp8Error, match="OFFSETS"):
        mx.to_mxfp8_then_scaled_grouped_mm(A.cuda(), W.cuda(), short)
    # the context stays usable
    x = torch.ones((32, 32), dtype=torch.bfloat16, device="cuda")
    assert int(mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT)[0][0, 0].item()) == 0x78
