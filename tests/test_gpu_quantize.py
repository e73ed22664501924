"""GPU parity of the MXFP8 quantization kernels against the CPU oracle.

Bit-exact on every e4m3 code and every E8M0 scale byte, including the zero
padding of the blocked tensor-core layout.  Small cases compare whole tensors
(several 128x128 tiles, ragged row and column tails, empty groups); the
full-size workloads compare sampled rows and columns.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from mxfp8_precision_moe_gb300 import synth
from tests._util import require_gpu, sizes_to_ends, u8, u16

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def mx():
    require_gpu()
    import mxfp8_precision_moe_gb300 as m

    m.load()
    return m


def mixed_input(M, K, seed, outliers=True):
    """log-uniform row magnitudes, a few outliers, zero rows and bf16 subnormals."""
    x = synth.log_uniform_rows(M, K, seed).float()
    if outliers:
        g = torch.Generator().manual_seed(seed + 100)
        mask = torch.rand((M, K), generator=g) < 0.01
        x = torch.where(mask, x * 100.0, x)
    if M > 3:
        x[1] = 0.0
        x[2] = x[2] * 1e-36  # into the bf16 subnormal range
    return x.to(torch.bfloat16)


def run(mx, x, dirs, layout, offs=None):
    status = mx.new_status()
    xs = x.cuda()
    o = None if offs is None else torch.tensor(np.asarray(offs, dtype=np.int32)).cuda()
    res = mx.mxfp8_quantize_2d(xs, dirs, layout, o, status)
    mx.read_status(status)
    return [None if t is None else u8(t) for t in res]


# ---------------------------------------------------------------- hand-worked blocks
def test_hand_worked_blocks_on_gpu(mx):
    rows, expect = [], []
    with open(os.path.join(HERE, "golden", "hand_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, fill, x0, x1, s, q0, q1, qf = line.split()
            v = np.full(32, float.fromhex(fill))
            v[0], v[1] = float.fromhex(x0), float.fromhex(x1)
            rows.append(v)
            expect.append((int(s, 16), int(q0, 16), int(q1, 16), int(qf, 16), name))
    x = torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16)
    # -0.0 survives the float -> bf16 cast
    q, s, _, _ = run(mx, x, mx.ROW, mx.SCALES_COMPACT)
    for i, (se, q0, q1, qf, name) in enumerate(expect):
        assert s[i, 0] == se, f"{name}: scale {s[i, 0]:#x} != {se:#x}"
        assert q[i, 0] == q0 and q[i, 1] == q1, f"{name}: {q[i, 0]:#x} {q[i, 1]:#x}"
        assert np.all(q[i, 2:] == qf), f"{name}: fill {np.unique(q[i, 2:])}"


def test_nonfinite_block_reading_on_gpu(mx):
    # the NaN/Inf reading (pinned in test_oracle_quantize.py) on hand-made blocks, GPU == oracle
    v = np.zeros((1, 64), dtype=np.float32)
    v[0, 0], v[0, 1], v[0, 2] = np.inf, -1.0, 2.0
    v[0, 32:] = np.linspace(-3, 3, 32)
    v[0, 40] = np.nan
    x = torch.tensor(v).to(torch.bfloat16)
    q, s, _, _ = run(mx, x, mx.ROW, mx.SCALES_COMPACT)
    qo, so = oracle.quantize_rows(u16(x))
    assert np.array_equal(s, so) and np.array_equal(q, qo)


# ---------------------------------------------------------------- whole-tensor parity, small shapes
ROW_SHAPES = [(256, 256), (200, 96), (1, 32), (33, 160), (384, 1056), (130, 4128)]


@pytest.mark.parametrize("M,K", ROW_SHAPES)
def test_row_compact(mx, oracle_lib, M, K):
    x = mixed_input(M, K, seed=M * 7 + K)
    q, s, _, _ = run(mx, x, mx.ROW, mx.SCALES_COMPACT)
    qo, so = oracle_lib.quantize_rows(u16(x))
    assert np.array_equal(s, so), "scales"
    assert np.array_equal(q, qo), "codes"


@pytest.mark.parametrize("sizes,K", [([200, 0, 64, 305, 31], 320), ([128, 128], 256), ([0, 0, 77], 160),
                                     ([1, 2, 3, 500], 4160)])
def test_row_blocked_groups(mx, oracle_lib, sizes, K):
    M = sum(sizes)
    x = mixed_input(M, K, seed=sum(sizes) + K)
    ends = sizes_to_ends(sizes)
    q, s, _, _ = run(mx, x, mx.ROW, mx.SCALES_BLOCKED, ends)
    qo, so = oracle_lib.quantize_rows(u16(x))
    want = oracle_lib.blocked_rowgroups(so, ends)
    assert np.array_equal(q, qo), "codes"
    assert s.size >= want.size
    assert np.array_equal(s[: want.size], want), "blocked scales (incl. zero padding)"


COL_CASES = [(256, 256, None), (96, 96, None), (608, 224, [96, 0, 160, 32, 320]), (512, 4128, [512]),
             (1024, 192, [0, 1024, 0])]


@pytest.mark.parametrize("M,K,sizes", COL_CASES)
@pytest.mark.parametrize("layout", ["compact", "blocked"])
def test_col(mx, oracle_lib, M, K, sizes, layout):
    x = mixed_input(M, K, seed=M + 3 * K)
    ends = None if sizes is None else sizes_to_ends(sizes)
    lay = mx.SCALES_COMPACT if layout == "compact" else mx.SCALES_BLOCKED
    _, _, qT, sT = run(mx, x, mx.COL, lay, ends)
    qo, so = oracle_lib.quantize_cols(u16(x))
    assert np.array_equal(qT, qo), "codes"
    if layout == "compact":
        assert np.array_equal(sT, so)
    else:
        want = oracle_lib.blocked_colgroups(so, ends if ends is not None else [M])
        assert np.array_equal(sT[: want.size], want), "blocked column-group scales"


@pytest.mark.parametrize("layout", ["compact", "blocked"])
def test_row_col_fused_equals_oracle(mx, oracle_lib, layout):
    sizes = [96, 0, 416, 32]
    M, K = sum(sizes), 352
    x = mixed_input(M, K, seed=5)
    ends = sizes_to_ends(sizes)
    lay = mx.SCALES_COMPACT if layout == "compact" else mx.SCALES_BLOCKED
    q, s, qT, sT = run(mx, x, mx.ROW | mx.COL, lay, ends)
    qo, so = oracle_lib.quantize_rows(u16(x))
    qTo, sTo = oracle_lib.quantize_cols(u16(x))
    assert np.array_equal(q, qo) and np.array_equal(qT, qTo)
    if layout == "compact":
        assert np.array_equal(s, so) and np.array_equal(sT, sTo)
    else:
        w1 = oracle_lib.blocked_rowgroups(so, ends)
        w2 = oracle_lib.blocked_colgroups(sTo, ends)
        assert np.array_equal(s[: w1.size], w1) and np.array_equal(sT[: w2.size], w2)


@pytest.mark.parametrize("M,K", [(64, 64), (96, 160), (256, 4096)])
def test_32x32(mx, oracle_lib, M, K):
    x = mixed_input(M, K, seed=M * K)
    q, s, _, _ = run(mx, x, mx.BLOCK32X32, mx.SCALES_COMPACT)
    qo, so = oracle_lib.quantize_32x32(u16(x))
    assert np.array_equal(s, so) and np.array_equal(q, qo)
    # transpose invariance on the GPU side as well
    q2, s2, _, _ = run(mx, x.t().contiguous(), mx.BLOCK32X32, mx.SCALES_COMPACT)
    assert np.array_equal(q2, q.T) and np.array_equal(s2, s.T)


@pytest.mark.parametrize("G,N,K", [(3, 160, 96), (2, 128, 256), (1, 32, 32), (4, 256, 416)])
@pytest.mark.parametrize("layout", ["compact", "blocked"])
def test_3d_plain_and_transposed(mx, oracle_lib, G, N, K, layout):
    w = synth.randn_bf16((G, N, K), 0.02, seed=G + N + K)
    lay = mx.SCALES_COMPACT if layout == "compact" else mx.SCALES_BLOCKED
    status = mx.new_status()
    q, s, qT, sT = [u8(t) for t in mx.mxfp8_quantize_3d_experts(w.cuda(), mx.ROW | mx.COL, lay, status)]
    mx.read_status(status)
    for g in range(G):
        qo, so = oracle_lib.quantize_rows(u16(w[g]))
        qTo, sTo = oracle_lib.quantize_cols(u16(w[g]))
        assert np.array_equal(q[g], qo) and np.array_equal(qT[g], qTo)
        if layout == "compact":
            assert np.array_equal(s[g], so) and np.array_equal(sT[g], sTo)
        else:
            assert np.array_equal(s[g], oracle_lib.blocked_rowgroups(so, [N]))
            assert np.array_equal(sT[g], oracle_lib.blocked_rowgroups(sTo, [K]))


def test_single_direction_matches_fused(mx):
    sizes = [64, 192]
    x = mixed_input(256, 512, seed=9)
    ends = sizes_to_ends(sizes)
    a = run(mx, x, mx.ROW | mx.COL, mx.SCALES_BLOCKED, ends)
    r = run(mx, x, mx.ROW, mx.SCALES_BLOCKED, ends)
    c = run(mx, x, mx.COL, mx.SCALES_BLOCKED, ends)
    # blocked buffers are sized by an upper bound; only the layout's extent is defined
    n_row = (128 + 256) * 4 * 4
    n_col = 512 * (1 + 2) * 4
    assert np.array_equal(a[0], r[0]) and np.array_equal(a[1][:n_row], r[1][:n_row])
    assert np.array_equal(a[2], c[2]) and np.array_equal(a[3][:n_col], c[3][:n_col])


def test_call_from_fresh_host_thread(mx, oracle_lib):
    """A host thread that has made no CUDA call yet (like an autograd worker)."""
    import threading

    x = mixed_input(256, 128, seed=77)
    xd = x.cuda()
    torch.cuda.synchronize()
    box = {}

    def work():
        try:
            box["res"] = mx.mxfp8_quantize_2d(xd, mx.ROW | mx.COL, mx.SCALES_COMPACT)
            torch.cuda.synchronize()
        except Exception as e:  # reported in the main thread
            box["err"] = e

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert "err" not in box, box.get("err")
    qo, so = oracle_lib.quantize_rows(u16(x))
    assert np.array_equal(u8(box["res"][0]), qo) and np.array_equal(u8(box["res"][1]), so)


def test_argument_errors(mx):
    x = torch.zeros((64, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.Mxfp8Error, match="ALIGN"):
        mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_COMPACT)
    x = torch.zeros((40, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.Mxfp8Error, match="ALIGN"):
        mx.mxfp8_quantize_2d(x, mx.COL, mx.SCALES_COMPACT)


def test_offsets_check_reports_bad_offsets(mx):
    status = mx.new_status()
    bad = torch.tensor([64, 32, 128], dtype=torch.int32, device="cuda")  # not monotone
    mx.mxfp8_check_offsets(bad, 128, 32, status)
    assert int(status.item()) == 7
    status = mx.new_status()
    ok = torch.tensor([64, 64, 128], dtype=torch.int32, device="cuda")
    mx.mxfp8_check_offsets(ok, 128, 32, status)
    assert int(status.item()) == 0
    status = mx.new_status()
    mx.mxfp8_check_offsets(torch.tensor([48, 128], dtype=torch.int32, device="cuda"), 128, 32, status)
    assert int(status.item()) == 7


# ---------------------------------------------------------------- full-size workloads, sampled
def _sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, n)]))


def _check_rows_sampled(oracle_lib, x_gpu, q_gpu, s_gpu, rows, ends=None, blocked=True):
    xs = u16(x_gpu[torch.as_tensor(rows, device=x_gpu.device)])
    qo, so = oracle_lib.quantize_rows(xs)
    qg = u8(q_gpu[torch.as_tensor(rows, device=q_gpu.device)])
    assert np.array_equal(qg, qo), "sampled row codes"
    K = x_gpu.shape[1]
    kbt = (K + 127) // 128
    sb = u8(s_gpu)
    if ends is None:
        ends = np.array([x_gpu.shape[0]])
    starts = np.concatenate([[0], ends[:-1]])
    pstart = np.concatenate([[0], np.cumsum((-(-(ends - starts) // 128)) * 128)[:-1]])
    for i, r in enumerate(rows):
        g = int(np.searchsorted(ends, r, side="right"))
        pr = pstart[g] + (r - starts[g])
        got = np.array([sb[oracle_lib.blocked_offset(int(pr), kb, kbt)] for kb in range(K // 32)])
        assert np.array_equal(got, so[i]), f"row {r} scales"


def _check_cols_sampled(oracle_lib, x_gpu, qT_gpu, sT_gpu, cols, ends=None):
    M, K = x_gpu.shape
    if ends is None:
        ends = np.array([M])
    starts = np.concatenate([[0], ends[:-1]])
    ct = int(np.sum(-(-(ends - starts) // 128)))
    sb = u8(sT_gpu)
    for c in cols:
        col = u16(x_gpu[:, int(c)])
        qo, so = oracle_lib.quantize_vec(col)
        assert np.array_equal(u8(qT_gpu[int(c)]), qo), f"col {c} codes"
        qcol = 0
        for g in range(len(ends)):
            nb = (ends[g] - starts[g]) // 32
            for b in range(nb):
                got = sb[oracle_lib.blocked_offset(int(c), qcol + b, ct)]
                assert got == so[starts[g] // 32 + b], f"col {c} group {g} block {b}"
            qcol += -(-(ends[g] - starts[g]) // 128) * 4


@pytest.mark.parametrize("name", ["scout", "imbalanced", "swiglu_x"])
def test_full_size_activations_sampled(mx, oracle_lib, name):
    if name == "scout":
        sizes, M, K = synth.scout_group_sizes(0), 16384, 5120
        x = synth.randn_bf16((M, K), 1.0, 1, device="cuda")
    elif name == "imbalanced":
        sizes, M, K = synth.imbalanced_group_sizes(0), 32768, 7168
        x = synth.outlier_activations((M, K), 1, device="cuda")
    else:
        sizes, M, K = synth.swiglu_group_sizes(), 65600, 5120
        x = synth.randn_bf16((M, K), 1.0, 1, device="cuda")
    ends = sizes_to_ends(sizes)
    offs = torch.tensor(ends.astype(np.int32), device="cuda")
    status = mx.new_status()
    q, s, qT, sT = mx.mxfp8_quantize_2d(x, mx.ROW | mx.COL, mx.SCALES_BLOCKED, offs, status)
    mx.read_status(status)
    rows = np.unique(np.concatenate([_sample_rows(M, 48, 3), np.clip(ends - 1, 0, M - 1), np.clip(ends, 0, M - 1)]))
    _check_rows_sampled(oracle_lib, x, q, s, rows, ends)
    cols = _sample_rows(K, 6, 4)
    _check_cols_sampled(oracle_lib, x, qT, sT, cols, ends)


@pytest.mark.parametrize("M,K", [(131072, 8192), (8192, 5120)])
def test_full_size_sweep_sampled(mx, oracle_lib, M, K):
    x = synth.log_uniform_rows(M, K, seed=11, device="cuda")
    status = mx.new_status()
    q, s, qT, sT = mx.mxfp8_quantize_2d(x, mx.ROW | mx.COL, mx.SCALES_BLOCKED, None, status)
    mx.read_status(status)
    _check_rows_sampled(oracle_lib, x, q, s, _sample_rows(M, 48, 5))
    _check_cols_sampled(oracle_lib, x, qT, sT, _sample_rows(K, 3, 6))
    del q, s, qT, sT
    q32, s32, _, _ = mx.mxfp8_quantize_2d(x, mx.BLOCK32X32, mx.SCALES_COMPACT, None, status)
    mx.read_status(status)
    for br in _sample_rows(M // 32, 6, 7):
        blk = u16(x[br * 32:(br + 1) * 32])
        qo, so = oracle_lib.quantize_32x32(blk)
        assert np.array_equal(u8(q32[br * 32:(br + 1) * 32]), qo)
        assert np.array_equal(u8(s32[br]), so[0])


def test_full_size_single_directions_sampled(mx, oracle_lib):
    """The row-only and column-only launches the sweep times, at its largest 5120-wide shape, and the
    3D expert weights [16, 8192, 5120] quantized along K only and along N only: sampled rows and
    columns byte-exact against the oracle (codes and blocked scales)."""
    M, K = 131072, 5120
    x = synth.log_uniform_rows(M, K, seed=13, device="cuda")
    status = mx.new_status()
    q, s, _, _ = mx.mxfp8_quantize_2d(x, mx.ROW, mx.SCALES_BLOCKED, None, status)
    mx.read_status(status)
    _check_rows_sampled(oracle_lib, x, q, s, _sample_rows(M, 32, 8))
    del q, s
    _, _, qT, sT = mx.mxfp8_quantize_2d(x, mx.COL, mx.SCALES_BLOCKED, None, status)
    mx.read_status(status)
    _check_cols_sampled(oracle_lib, x, qT, sT, _sample_rows(K, 3, 9))
    del x, qT, sT
    G, N, K = 16, 8192, 5120
    w = synth.randn_bf16((G, N, K), 0.02, seed=4, device="cuda")
    q, s, _, _ = mx.mxfp8_quantize_3d_experts(w, mx.ROW, mx.SCALES_BLOCKED, status)
    mx.read_status(status)
    for g in (1, 14):
        _check_rows_sampled(oracle_lib, w[g], q[g], s[g], _sample_rows(N, 8, 20 + g))
    del q, s
    _, _, qT, sT = mx.mxfp8_quantize_3d_experts(w, mx.COL, mx.SCALES_BLOCKED, status)
    mx.read_status(status)
    for g in (2, 15):
        _check_cols_sampled(oracle_lib, w[g], qT[g], sT[g], _sample_rows(K, 2, 30 + g))


def test_full_size_3d_weights_sampled(mx, oracle_lib):
    G, N, K = 16, 8192, 5120
    w = synth.randn_bf16((G, N, K), 0.02, seed=2, device="cuda")
    status = mx.new_status()
    q, s, qT, sT = mx.mxfp8_quantize_3d_experts(w, mx.ROW | mx.COL, mx.SCALES_BLOCKED, status)
    mx.read_status(status)
    for g in (0, 7, 15):
        _check_rows_sampled(oracle_lib, w[g], q[g], s[g], _sample_rows(N, 8, g))
        _check_cols_sampled(oracle_lib, w[g], qT[g], sT[g], _sample_rows(K, 2, g + 1))
