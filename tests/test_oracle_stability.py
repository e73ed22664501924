"""Pins of the oracle's stability variants ("MXFP8 (Micro-scaling FP8)", "Numerical
stability": random Hadamard transforms and stochastic rounding), no GPU:
- Philox4x32-10 against the published known-answer vectors (tests/golden);
- the Hadamard signs and the stochastic-rounding bytes against values written by an independent
  pure-Python Philox4x32-10 (tests/golden/stability_words.txt, make_stability_words.py);
- stochastic rounding against hand-worked cases, against an independent fp32 bit-pattern
  algorithm (add the random byte to the top 8 of the 20 mantissa bits E4M3 drops, truncate) on
  the normal E4M3 range, and for its mean (within 1/256 of a step);
- the Hadamard transform against scipy's Hadamard matrix on inputs where fp32 is exact, its
  norm preservation, and the transpose relation between the row and column quantizations."""
import os

import numpy as np
import pytest
import scipy.linalg

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def kat_rows():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            yield [int(w, 16) for w in line.split()]


@pytest.mark.parametrize("row", list(kat_rows()))
def test_philox_known_answers(row):
    assert oracle.philox4x32_10(row[0:4], row[4:6]) == row[6:10]


STAB = os.path.join(os.path.dirname(__file__), "golden", "stability_words.txt")


def stability_rows(kind):
    for line in open(STAB):
        f = line.split()
        if f and f[0] == kind:
            yield f[1:]


def test_independent_philox_meets_the_known_answers():
    """The pure-Python generator that wrote stability_words.txt reproduces the published vectors."""
    from tests.golden import make_stability_words as ref
    for row in kat_rows():
        assert ref.philox4x32_10(row[0:4], row[4:6]) == row[6:10]


@pytest.mark.parametrize("seed,r,c,C,byte", list(stability_rows("sr")))
def test_sr_byte_golden(seed, r, c, C, byte):
    """oracle_sr_byte against bytes written by an independent Philox (tests/golden/stability_words.txt):
    byte 8 (r mod 2) + (c mod 8) of the draw for block floor(r/2) (C/8) + floor(c/8)."""
    assert oracle.sr_byte(int(seed, 16), int(r), int(c), int(C)) == int(byte, 16)


def test_golden_bytes_tell_plausible_misreadings_apart():
    """The stored bytes pin the selection: the other row of the 2 x 8 block, a big-endian byte order
    inside a word, the counter's high word dropped, or the blocks numbered column-major each give
    another byte for some golden case."""
    from tests.golden import make_stability_words as ref
    M = 0xFFFFFFFF
    misses = {"row parity": 0, "byte order": 0, "high counter word": 0, "column-major blocks": 0}
    for seed, r, c, C, byte in stability_rows("sr"):
        seed, r, c, C, byte = int(seed, 16), int(r), int(c), int(C), int(byte, 16)
        key = [seed & M, seed >> 32]
        b = ref.sr_block(r, c, C)
        out = ref.philox4x32_10([b & M, b >> 32, 0, 0], key)
        k = 8 * (r % 2) + c % 8
        assert (out[k // 4] >> (8 * (k % 4))) & 0xFF == byte
        k2 = 8 * (1 - r % 2) + c % 8
        misses["row parity"] += ((out[k2 // 4] >> (8 * (k2 % 4))) & 0xFF) != byte
        misses["byte order"] += ((out[k // 4] >> (8 * (3 - k % 4))) & 0xFF) != byte
        o2 = ref.philox4x32_10([b & M, 0, 0, 0], key)
        misses["high counter word"] += ((o2[k // 4] >> (8 * (k % 4))) & 0xFF) != byte
        bc = (c // 8) * (1 << 40) + r // 2
        o3 = ref.philox4x32_10([bc & M, bc >> 32, 0, 0], key)
        misses["column-major blocks"] += ((o3[k // 4] >> (8 * (k % 4))) & 0xFF) != byte
    assert all(v > 0 for v in misses.values()), misses


E = oracle.e4m3_table()


@pytest.mark.parametrize("y,u,code", [
    (1.0625, 128, 0x39),             # midway 1.0 / 1.125: F = 128, F + u = 256 -> up
    (1.0625, 127, 0x38),             # F + u = 255 -> down
    (-1.0625, 128, 0xB9),            # the sign is applied afterwards
    (1.5 * 2 ** -9, 128, 0x02),      # subnormal step, midway -> up
    (1.5 * 2 ** -9, 127, 0x01),
    (447.0, 8, 0x7E),                # 447 = 416 + 31/32 step: F = 248, up iff u >= 8
    (447.0, 7, 0x7D),
    (1.0 + 1 / 2048, 255, 0x39),     # 1/256 of the step: F = 1, 1 + 255 = 256 -> up only at u = 255
    (1.0 + 1 / 2048, 254, 0x38),
    (1.0 + 1 / 4096, 255, 0x38),     # below 1/256 of the step: F = 0, never up
    (460.0, 0, 0x7E),                # beyond the largest finite magnitude: 448
    (1e9, 255, 0x7E),
    (0.0, 255, 0x00),
    (-0.0, 255, 0x80),
])
def test_sr_hand_cases(y, u, code):
    assert oracle.e4m3_encode_sr(y, u) == code


def test_sr_keeps_representable_values():
    for c in range(0x7F):
        for u in (0, 0x5A, 0xFF):
            assert oracle.e4m3_encode_sr(E[c], u) == c


def test_sr_matches_fp32_bit_algorithm_on_normal_range():
    """On the normal E4M3 range (2^-6 .. 448) the reading equals an independent bit algorithm: add
    the byte into the top 8 of the 20 fp32 mantissa bits E4M3 drops, then truncate those 20 bits."""
    rng = np.random.default_rng(1)
    y = np.float32(2.0) ** rng.uniform(-6, np.log2(448), 4000).astype(np.float32)
    y = y * rng.choice([-1, 1], y.size).astype(np.float32)
    u = rng.integers(0, 256, y.size, dtype=np.uint64)
    bits = np.abs(y).view(np.uint32).astype(np.uint64)
    t = ((bits + (u << np.uint64(12))) & ~np.uint64(0xFFFFF)).astype(np.uint32)
    want = np.minimum(t.view(np.float32).astype(np.float64), 448.0) * np.sign(y)
    codes = [oracle.e4m3_encode_sr(float(a), int(b)) for a, b in zip(y, u)]
    got = np.array([E[q & 0x7F] * (-1 if q & 0x80 else 1) for q in codes])
    assert np.array_equal(got, want)


def test_sr_is_unbiased_to_within_a_256th_of_a_step():
    """Over all 256 byte values the mean is exactly lo + (F / 256) step, within step / 256 of y; over
    random bytes it is within 5 standard errors of that."""
    rng = np.random.default_rng(2)
    for y in (1.0 + 5 / 64, 3.3, 0.013, 300.0, 2.5 * 2 ** -9):
        every = np.array([E[oracle.e4m3_encode_sr(y, u)] for u in range(256)])
        lo, hi = every.min(), every.max()
        step = hi - lo
        assert set(np.unique(every)) <= {lo, hi} and step > 0
        assert abs(every.mean() - y) <= step / 256 + 1e-15
        r = rng.integers(0, 256, 20000)
        vals = every[r]
        p = (every.mean() - lo) / step
        se = step * np.sqrt(p * (1 - p) / r.size)
        assert abs(vals.mean() - every.mean()) <= 5 * se + 1e-12


@pytest.mark.parametrize("seed,signs", list(stability_rows("sign")))
def test_rht_signs_golden(seed, signs):
    """oracle_rht_signs against signs written by an independent Philox: sign i is -1 iff bit i of
    word 0 of counter (0, 0, 2, 0) is set.  The stored strings are not palindromes, so a reversed
    bit order fails, and they differ from the bits of words 1-3."""
    from tests.golden import make_stability_words as ref
    d = oracle.rht_signs(int(seed, 16))
    assert "".join("-" if v < 0 else "+" for v in d) == signs
    assert signs != signs[::-1]
    out = ref.philox4x32_10([0, 0, 2, 0], [int(seed, 16) & 0xFFFFFFFF, int(seed, 16) >> 32])
    for w in out[1:]:
        assert "".join("-" if (w >> i) & 1 else "+" for i in range(32)) != signs


def test_rht_matches_hadamard_matrix_exactly_on_integers():
    rng = np.random.default_rng(3)
    H = scipy.linalg.hadamard(32).astype(np.int64)
    c = np.float32(1.0 / np.sqrt(32.0))
    for seed in (0, 7, 2 ** 40 + 3):
        d = oracle.rht_signs(seed)
        x = rng.integers(-1000, 1000, 32).astype(np.float32)
        exact = H @ (d.astype(np.int64) * x.astype(np.int64))     # integers, exact in fp32
        want = exact.astype(np.float32) * c
        assert np.array_equal(oracle.rht32(x, d), want)


def test_rht_preserves_the_norm():
    rng = np.random.default_rng(4)
    d = oracle.rht_signs(11)
    for _ in range(20):
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        y = oracle.rht32(x, d)
        assert abs(np.linalg.norm(y.astype(np.float64)) / np.linalg.norm(x.astype(np.float64)) - 1) < 1e-5


def bf16(a):
    import torch
    from tests._util import u16
    return u16(torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16))


def test_options_reduce_and_transpose():
    rng = np.random.default_rng(5)
    x = bf16(rng.standard_normal((64, 96)) * 3)
    q, s = oracle.quantize_rows(x)
    assert all(np.array_equal(a, b) for a, b in zip(oracle.quantize_rows_opts(x, 0, 9), (q, s)))
    # the Hadamard transform alone is deterministic, so the column quantization of x is the
    # row quantization of x^T
    qT, sT = oracle.quantize_cols_opts(x, oracle.OPT_RHT, 9)
    qr, sr = oracle.quantize_rows_opts(np.ascontiguousarray(x.T), oracle.OPT_RHT, 9)
    assert np.array_equal(qT, qr) and np.array_equal(sT, sr)
    # stochastic rounding moves no code by more than one step and keeps the scales
    q2, s2 = oracle.quantize_rows_opts(x, oracle.OPT_SR, 9)
    assert np.array_equal(s2, s)
    assert np.all(np.abs(E[q2 & 0x7F] - E[q & 0x7F]) <= np.maximum(E[q & 0x7F] / 8, 2.0 ** -9) + 1e-12)


def test_block_at_matches_the_tensor_routines():
    rng = np.random.default_rng(6)
    x = bf16(rng.standard_normal((64, 96)))
    for opts in (0, oracle.OPT_SR, oracle.OPT_RHT, oracle.OPT_SR | oracle.OPT_RHT):
        q, s = oracle.quantize_rows_opts(x, opts, 77)
        qT, sT = oracle.quantize_cols_opts(x, opts, 77)
        for r, b in ((0, 0), (5, 1), (63, 2)):
            qb, sb = oracle.quantize_block_at(x[r, 32 * b:32 * b + 32], r, 32 * b, False, 96, opts, 77)
            assert np.array_equal(qb, q[r, 32 * b:32 * b + 32]) and sb == s[r, b]
        for c, b in ((0, 0), (7, 1), (95, 1)):
            qc, sc = oracle.quantize_block_at(np.ascontiguousarray(x[32 * b:32 * b + 32, c]), 32 * b, c, True, 96,
                                              opts, 77)
            assert np.array_equal(qc, qT[c, 32 * b:32 * b + 32]) and sc == sT[c, b]
