"""Pins for the oracle's blocked scale layout and its grouped GEMMs (CPU only).

Layout: hand-computed positions (tests/golden/blocked_layout.txt), bijection,
per-group padding positions and zero padding.
GEMM: brute-force Python loops on tiny shapes, numpy matmul of the dequantized
operands (a library routine the oracle does not use), the identity-weight
special case, G=1 == dense, empty groups, and the wgrad transpose identity.
"""
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def golden_offsets():
    rows = []
    with open(os.path.join(HERE, "golden", "blocked_layout.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(tuple(int(t) for t in line.split()))
    return rows


@pytest.mark.parametrize("kbt,r,kb,off", golden_offsets())
def test_blocked_offset_hand_positions(oracle_lib, kbt, r, kb, off):
    assert oracle_lib.blocked_offset(r, kb, kbt) == off


def test_blocked_offset_bijection(oracle_lib):
    R, Kb = 384, 12
    offs = {oracle_lib.blocked_offset(r, kb, Kb // 4) for r in range(R) for kb in range(Kb)}
    assert offs == set(range(R * Kb))


def test_blocked_rowgroups_padding(oracle_lib):
    # groups of 100, 0, 200 rows; Kb = 5 -> padded to 8 columns (2 tiles)
    ends = [100, 100, 300]
    s = (np.arange(300 * 5) % 250 + 1).astype(np.uint8).reshape(300, 5)
    out = oracle_lib.blocked_rowgroups(s, ends)
    # padded rows: group0 -> 128, group1 -> 0, group2 -> 256 => 384 rows x 8 cols
    assert out.size == 384 * 8
    kbt = 2
    # group 0 row 7 -> padded row 7; group 2 row 0 (global row 100) -> padded row 128
    assert out[oracle_lib.blocked_offset(7, 3, kbt)] == s[7, 3]
    assert out[oracle_lib.blocked_offset(128, 4, kbt)] == s[100, 4]
    assert out[oracle_lib.blocked_offset(128 + 199, 0, kbt)] == s[299, 0]
    # everything not a scale is zero: count non-zero bytes == number of scales (all non-zero)
    assert np.count_nonzero(out) == 300 * 5
    for r in range(100, 128):          # group 0 padding rows
        for kb in range(8):
            assert out[oracle_lib.blocked_offset(r, kb, kbt)] == 0
    for kb in range(5, 8):             # padding columns
        assert out[oracle_lib.blocked_offset(3, kb, kbt)] == 0


def test_blocked_colgroups_padding(oracle_lib):
    # tokens: groups of 64, 0, 160 tokens (multiples of 32); 40 rows
    ends = [64, 64, 224]
    R, Mb = 40, 224 // 32
    s = (np.arange(R * Mb) % 200 + 1).astype(np.uint8).reshape(R, Mb)
    out = oracle_lib.blocked_colgroups(s, ends)
    # columns: group0 -> 4 (ceil(64/128)*4), group1 -> 0, group2 -> 8 => 12 cols; rows padded to 128
    assert out.size == 128 * 12
    kbt = 3
    assert out[oracle_lib.blocked_offset(5, 1, kbt)] == s[5, 1]          # group 0 block 1
    assert out[oracle_lib.blocked_offset(5, 4, kbt)] == s[5, 2]          # group 2 block 0 -> col 4
    assert out[oracle_lib.blocked_offset(39, 8, kbt)] == s[39, 6]        # group 2 block 4 -> col 8
    assert np.count_nonzero(out) == R * Mb


def make_case(M, N, K, sizes, seed):
    rng = np.random.default_rng(seed)
    A = bf16_bits(rng.standard_normal((M, K))).reshape(M, K)
    W = bf16_bits(rng.standard_normal((len(sizes), N, K)) * 0.02).reshape(len(sizes), N, K)
    return A, W, np.cumsum(sizes)


def deq_rows(o, q, s):
    return o.dequant(q, np.repeat(s, 32, axis=-1))


def test_grouped_fwd_bruteforce_tiny(oracle_lib):
    o = oracle_lib
    A, W, ends = make_case(12, 3, 64, [5, 0, 7], 10)
    aq, as_ = o.quantize_rows(A)
    wq, ws = zip(*[o.quantize_rows(W[g]) for g in range(3)])
    wq, ws = np.stack(wq), np.stack(ws)
    out = o.grouped_mm_rows(aq, as_, wq, ws, ends)
    tab = o.e4m3_table()
    lo = 0
    for g, hi in enumerate(ends):
        for m in range(lo, hi):
            for n in range(3):
                acc = 0.0
                for k in range(64):
                    a = tab[aq[m, k]] * 2.0 ** (int(as_[m, k // 32]) - 127)
                    b = tab[wq[g, n, k]] * 2.0 ** (int(ws[g, n, k // 32]) - 127)
                    acc += a * b
                assert out[m, n] == acc
        lo = hi


def test_grouped_fwd_equals_numpy_per_group(oracle_lib):
    o = oracle_lib
    sizes = [32, 0, 96, 17, 15]
    A, W, ends = make_case(sum(sizes), 40, 128, sizes, 11)
    aq, as_ = o.quantize_rows(A)
    wq, ws = zip(*[o.quantize_rows(W[g]) for g in range(len(sizes))])
    wq, ws = np.stack(wq), np.stack(ws)
    out = o.grouped_mm_rows(aq, as_, wq, ws, ends)
    Ad = deq_rows(o, aq, as_)
    lo = 0
    for g, hi in enumerate(ends):
        ref = Ad[lo:hi] @ deq_rows(o, wq[g], ws[g]).T
        np.testing.assert_allclose(out[lo:hi], ref, rtol=1e-12, atol=1e-300)
        lo = hi


def test_identity_weight_gives_dequantized_activations(oracle_lib):
    o = oracle_lib
    K = 64
    A = bf16_bits(np.random.default_rng(12).standard_normal((48, K)) * 5).reshape(48, K)
    W = bf16_bits(np.stack([np.eye(K), np.eye(K)])).reshape(2, K, K)
    aq, as_ = o.quantize_rows(A)
    wq, ws = zip(*[o.quantize_rows(W[g]) for g in range(2)])
    wq, ws = np.stack(wq), np.stack(ws)
    # identity rows: the block holding the diagonal has scale 0x77 (amax 1) and
    # code 0x78 there; the other block of the row is all zero (scale 0x00)
    n = np.arange(K)
    assert np.all(ws[:, n, n // 32] == 0x77) and np.all(np.diagonal(wq, axis1=1, axis2=2) == 0x78)
    assert np.count_nonzero(ws) == 2 * K and np.count_nonzero(wq) == 2 * K
    out = o.grouped_mm_rows(aq, as_, wq, ws, [16, 48])
    assert np.array_equal(out, deq_rows(o, aq, as_))


def test_single_group_equals_dense(oracle_lib):
    o = oracle_lib
    A, W, _ = make_case(40, 24, 96, [40], 13)
    aq, as_ = o.quantize_rows(A)
    wq, ws = o.quantize_rows(W[0])
    out = o.grouped_mm_rows(aq, as_, wq[None], ws[None], [40])
    np.testing.assert_allclose(out, deq_rows(o, aq, as_) @ deq_rows(o, wq, ws).T, rtol=1e-12, atol=1e-300)


def test_wgrad_matches_numpy_and_empty_group_zero(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(14)
    sizes = [64, 0, 96]
    M, N, K = sum(sizes), 24, 40
    ends = np.cumsum(sizes)
    A = bf16_bits(rng.standard_normal((M, K))).reshape(M, K)
    D = bf16_bits(rng.standard_normal((M, N)) * 1e-3).reshape(M, N)
    dq, ds = o.quantize_cols(D)       # dOut^T [N, M]
    aq, as_ = o.quantize_cols(A)      # A^T    [K, M]
    dw = o.grouped_mm_wgrad(dq, ds, aq, as_, ends)
    assert np.all(dw[1] == 0.0)
    Dd = deq_rows(o, dq, ds)          # [N, M]
    Ad = deq_rows(o, aq, as_)         # [K, M]
    lo = 0
    for g, hi in enumerate(ends):
        ref = Dd[:, lo:hi] @ Ad[:, lo:hi].T
        np.testing.assert_allclose(dw[g], ref, rtol=1e-12, atol=1e-300)
        lo = hi


def test_wgrad_bruteforce_tiny(oracle_lib):
    o = oracle_lib
    rng = np.random.default_rng(15)
    sizes = [32, 32]
    M, N, K = 64, 2, 3
    A = bf16_bits(rng.standard_normal((M, K))).reshape(M, K)
    D = bf16_bits(rng.standard_normal((M, N))).reshape(M, N)
    dq, ds = o.quantize_cols(D)
    aq, as_ = o.quantize_cols(A)
    dw = o.grouped_mm_wgrad(dq, ds, aq, as_, np.cumsum(sizes))
    tab = o.e4m3_table()
    for g in range(2):
        for n in range(N):
            for k in range(K):
                acc = 0.0
                for m in range(g * 32, g * 32 + 32):
                    acc += tab[dq[n, m]] * 2.0 ** (int(ds[n, m // 32]) - 127) * tab[aq[k, m]] * 2.0 ** (int(as_[k, m // 32]) - 127)
                assert dw[g, n, k] == acc


def test_blas_forms_equal_the_scalar_loops(oracle_lib):
    """The matmul-per-group forms used for large parity cases give the scalar loops' sums (same
    products, another summation order: fp64 agreement to ~1e-13 relative), empty groups included."""
    o = oracle_lib
    rng = np.random.default_rng(16)
    sizes = [64, 0, 33, 95, 32]
    A, W, ends = make_case(sum(sizes), 48, 160, sizes, 17)
    aq, as_ = o.quantize_rows(A)
    wq, ws = zip(*[o.quantize_rows(W[g]) for g in range(len(sizes))])
    wq, ws = np.stack(wq), np.stack(ws)
    ref = o.grouped_mm_rows(aq, as_, wq, ws, ends)
    np.testing.assert_allclose(o.grouped_mm_rows_blas(aq, as_, wq, ws, ends), ref, rtol=1e-12, atol=1e-300)
    sizes = [64, 0, 96, 32]
    M, N, K = sum(sizes), 40, 24
    D = bf16_bits(rng.standard_normal((M, N))).reshape(M, N)
    Ak = bf16_bits(rng.standard_normal((M, K)) * 3).reshape(M, K)
    dq, ds = o.quantize_cols(D)
    akq, aks = o.quantize_cols(Ak)
    ends = np.cumsum(sizes)
    ref = o.grouped_mm_wgrad(dq, ds, akq, aks, ends)
    got = o.grouped_mm_wgrad_blas(dq, ds, akq, aks, ends)
    assert np.all(got[1] == 0.0)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-300)
