"""Pins for the oracle's quantization (CPU only).

The oracle is checked against things other than itself:
  * hand-worked blocks (tests/golden/hand_blocks.txt);
  * the scale byte from the bf16 exponent field (s = max(E - 8, 0)), a closed
    form independent of the oracle's frexp route;
  * a bit-level round-to-nearest-even E4M3 encoder written here (arithmetic
    rounding of the scaled mantissa), independent of the oracle's exhaustive
    nearest-code search, over every bf16 pattern at several scales;
  * torch's float8_e4m3fn cast (a library routine) on unsaturated values;
  * the round-trip bound |x - deq(q)| <= ulp/2 at the block scale;
  * transpose invariance of 32x32 blocks, and rows-of-X^T == columns-of-X.
"""
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def load_hand_blocks():
    rows = []
    with open(os.path.join(HERE, "golden", "hand_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, fill, x0, x1, s, q0, q1, qf = line.split()
            rows.append((name, float.fromhex(fill), float.fromhex(x0), float.fromhex(x1),
                         int(s, 16), int(q0, 16), int(q1, 16), int(qf, 16)))
    return rows


HAND = load_hand_blocks()


@pytest.mark.parametrize("row", HAND, ids=[r[0] for r in HAND])
def test_hand_worked_blocks(oracle_lib, row):
    name, fill, x0, x1, s, q0, q1, qf = row
    vals = np.full(32, fill, dtype=np.float64)
    vals[0], vals[1] = x0, x1
    bits = bf16_bits(vals)
    # the fixture values are exact in bf16
    assert all(oracle_lib.bf16_to_f64(b) == v or (v == 0 and oracle_lib.bf16_to_f64(b) == 0) for b, v in zip(bits, vals))
    q, sc = oracle_lib.quantize_vec(bits)
    assert sc[0] == s, f"{name}: scale {sc[0]:#x} != {s:#x}"
    assert q[0] == q0 and q[1] == q1, f"{name}: q0,q1 = {q[0]:#x},{q[1]:#x}"
    assert np.all(q[2:] == qf), f"{name}: fill codes {np.unique(q[2:])}"


def test_e4m3_decode_definition_points(oracle_lib):
    # Format landmarks: max 448, min normal 2^-6, min subnormal 2^-9, NaN codes.
    assert oracle_lib.e4m3_to_f64(0x7E) == 448.0
    assert oracle_lib.e4m3_to_f64(0x08) == 2.0 ** -6
    assert oracle_lib.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle_lib.e4m3_to_f64(0x07) == 7 * 2.0 ** -9
    assert oracle_lib.e4m3_to_f64(0x38) == 1.0
    assert oracle_lib.e4m3_to_f64(0xB8) == -1.0
    assert np.isnan(oracle_lib.e4m3_to_f64(0x7F)) and np.isnan(oracle_lib.e4m3_to_f64(0xFF))
    # strictly increasing over the non-negative finite codes
    tab = oracle_lib.e4m3_table()
    assert np.all(np.diff(tab[:0x7F]) > 0)


def scale_from_exponent_field(x_bits_block: np.ndarray) -> int:
    """Closed form from bf16 bits: s = max(E(amax) - 8, 0), E = biased exponent field."""
    mag = (x_bits_block & 0x7FFF).astype(np.int64)
    E = int(mag.max()) >> 7
    return max(E - 8, 0)


def rne_e4m3_bitlevel(y: np.ndarray) -> np.ndarray:
    """Independent encoder: clamp to 448, find the binade, round the scaled
    mantissa half-to-even with np.round, then assemble sign/exponent/mantissa."""
    y = np.asarray(y, dtype=np.float64)
    neg = np.signbit(y)
    a = np.minimum(np.abs(y), 448.0)
    _, p = np.frexp(a)
    E = np.maximum(p - 1, -6)              # subnormals share the min-normal binade
    step = np.ldexp(1.0, E - 3)            # 3 mantissa bits
    r = np.round(a / step)                 # half to even
    v = r * step
    code = np.zeros(a.shape, dtype=np.int64)
    sub = v < 2.0 ** -6
    code[sub] = (v[sub] / 2.0 ** -9).astype(np.int64)
    nrm = ~sub
    _, p2 = np.frexp(v[nrm])
    e2 = p2 - 1
    mant = ((v[nrm] / np.ldexp(1.0, e2) - 1.0) * 8).astype(np.int64)
    code[nrm] = ((e2 + 7) << 3) | mant
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _finite_bf16_values():
    v = torch.from_numpy(ALL_BF16.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return v[np.isfinite(v)]


@pytest.mark.parametrize("s", [0, 60, 119, 200, 246])
def test_element_encoding_bruteforce_all_bf16(oracle_lib, s):
    """Every finite bf16 value scaled by 2^(127-s): the oracle's exhaustive search
    equals the bit-level RNE encoder (and, where |y| <= 448, torch's cast)."""
    v = _finite_bf16_values()
    y = np.ldexp(v, 127 - s)
    got = np.array([oracle_lib.e4m3_encode(t) for t in y], dtype=np.uint8)
    ref = rne_e4m3_bitlevel(y)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"s={s}: {bad.size} mismatches, first y={y[bad[0]]!r} got {got[bad[0]]:#x} ref {ref[bad[0]]:#x}"
    ok = (np.abs(y) <= 448.0) & (np.abs(y) >= 2.0 ** -100)
    lib_cast = torch.from_numpy(y[ok].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(lib_cast, got[ok])


def test_scale_two_ways_random_blocks(oracle_lib):
    rng = np.random.default_rng(1)
    for trial in range(400):
        mag = 10.0 ** rng.uniform(-40, 38)
        vals = rng.standard_normal(32) * mag
        if trial % 7 == 0:
            vals[rng.integers(0, 32, 5)] = 0.0
        bits = bf16_bits(vals)
        q, s = oracle_lib.quantize_vec(bits)
        assert s[0] == scale_from_exponent_field(bits)
        x = np.array([oracle_lib.bf16_to_f64(b) for b in bits])
        assert np.array_equal(q, rne_e4m3_bitlevel(np.ldexp(x, 127 - int(s[0]))))


def test_roundtrip_error_bound(oracle_lib):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 256)) * (10.0 ** rng.uniform(-6, 6, (64, 1)))
    bits = bf16_bits(x).reshape(64, 256)
    q, s = oracle_lib.quantize_rows(bits)
    xv = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    se = np.repeat(s, 32, axis=1).astype(np.int64)
    deq = oracle_lib.dequant(q, se)
    e = se - 127
    y = np.abs(np.ldexp(xv, -e))
    unsat = y <= 448.0
    _, p = np.frexp(np.maximum(y, 2.0 ** -6))
    ulp = np.ldexp(1.0, np.maximum(p - 1, -6) - 3)
    bound = 0.5 * ulp * np.ldexp(1.0, e)
    assert np.all(np.abs(xv - deq)[unsat] <= bound[unsat])
    # saturated elements land on +-448 * 2^e and lie in (448, 512) * 2^e
    sat = ~unsat
    if sat.any():
        assert np.all(np.abs(deq[sat]) == np.ldexp(448.0, e[sat]))
        assert np.all(y[sat] < 512.0)


def test_rows_of_transpose_equal_columns(oracle_lib):
    rng = np.random.default_rng(3)
    x = bf16_bits(rng.standard_normal((96, 64)) * 3.0).reshape(96, 64)
    qT, sT = oracle_lib.quantize_cols(x)
    q2, s2 = oracle_lib.quantize_rows(np.ascontiguousarray(x.T))
    assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_32x32_transpose_invariant_and_max_of_row_scales(oracle_lib):
    rng = np.random.default_rng(4)
    x = bf16_bits(rng.standard_normal((64, 96)) * (10.0 ** rng.uniform(-3, 3, (64, 1)))).reshape(64, 96)
    q, s = oracle_lib.quantize_32x32(x)
    qt, st = oracle_lib.quantize_32x32(np.ascontiguousarray(x.T))
    assert np.array_equal(qt, q.T) and np.array_equal(st, s.T)
    # the square-block scale is the largest of its 32 row-block scales (scale is monotone in amax)
    _, sr = oracle_lib.quantize_rows(x)
    assert np.array_equal(s, sr.reshape(2, 32, 3).max(axis=1))
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    se = np.repeat(np.repeat(s, 32, 0), 32, 1).astype(np.int64)
    assert np.array_equal(q, rne_e4m3_bitlevel(np.ldexp(xv, 127 - se)))


def test_nonfinite_block_reading(oracle_lib):
    """The reading for a block holding Inf or NaN (the pages are silent): the E8M0 NaN scale 0xFF,
    which the OCP MX format defines as making every element of its block NaN, and each code the
    E4M3 NaN carrying the element's own sign.  Pinned against two things outside the oracle: the
    block dequantizes to all-NaN through the format definition, and every code equals torch's
    float8_e4m3fn cast of a NaN with the element's sign (its NaN encoding 0x7F / 0xFF); blocks
    without a non-finite value next to it are quantized as usual."""
    vals = np.zeros(32)
    vals[0], vals[1], vals[2] = np.inf, -1.0, 2.0
    q, s = oracle_lib.quantize_vec(bf16_bits(vals))
    assert s[0] == 0xFF and q[0] == 0x7F and q[1] == 0xFF and q[2] == 0x7F
    rng = np.random.default_rng(31)
    x = rng.standard_normal((8, 96)) * 10.0 ** rng.uniform(-3, 3, (8, 1))
    x[rng.random(x.shape) < 0.05] = 0.0
    x[rng.random(x.shape) < 0.05] *= -0.0
    planted = [(0, 3, np.inf), (1, 40, -np.inf), (2, 70, np.nan), (3, 0, -np.nan), (3, 31, np.inf),
               (5, 33, np.nan), (5, 34, -np.inf), (7, 95, -np.inf)]
    for r, c, v in planted:
        x[r, c] = v
    xb = bf16_bits(x.ravel()).reshape(x.shape)
    q, s = oracle_lib.quantize_rows(xb)
    xv = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).float()
    nan_signed = torch.where(torch.signbit(xv), -torch.tensor(float("nan")), torch.tensor(float("nan")))
    want_nan_codes = nan_signed.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad_blocks = {(r, c // 32) for r, c, _ in planted}
    qc, sc = oracle_lib.quantize_rows(np.where(np.isfinite(xv.numpy()), xb, np.uint16(0)).astype(np.uint16))
    for r in range(8):
        for b in range(3):
            sl = slice(32 * b, 32 * b + 32)
            if (r, b) in bad_blocks:
                assert s[r, b] == 0xFF
                assert np.all(np.isnan(oracle_lib.dequant(q[r, sl], np.full(32, s[r, b], np.uint8))))
                assert np.array_equal(q[r, sl], want_nan_codes[r, sl])
            else:
                assert s[r, b] == sc[r, b] and np.array_equal(q[r, sl], qc[r, sl])
    # the column and 32x32 forms follow the same reading
    qT, sT = oracle_lib.quantize_cols(np.ascontiguousarray(np.tile(xb, (4, 1))))
    assert sT[3, 0] == 0xFF and np.array_equal(qT[3, :32], np.tile(want_nan_codes[:, 3], 4))
