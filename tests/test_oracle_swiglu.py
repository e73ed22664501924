"""Pins of the oracle's SwiGLU stage (no GPU): the fp64 -> bf16 rounding,
h = bf16(bf16(silu(h1)) * h3) and its backward (dh1, dh3), each checked against something
other than itself (torch's fp32 -> bf16 cast, torch's fp64 silu and silu_backward, hand-worked
values)."""
import numpy as np
import pytest
import torch

import oracle
from tests._util import u16


def test_bf16_rounding_matches_torch_on_fp32_values():
    # every fp32 value is exact in fp64, so torch's single fp32 -> bf16 RNE is the reference
    rng = np.random.default_rng(0)
    pat = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = pat.view(np.float32)
    f = f[np.isfinite(f)]
    ref = u16(torch.from_numpy(f.copy()).to(torch.bfloat16))
    got = oracle.bf16_from_f64(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rounding_of_every_tie_between_neighbours():
    # midpoints between consecutive bf16 values round to the even pattern
    b = np.arange(0x0000, 0x7F7F, 97, dtype=np.uint32)
    lo = (b << 16).view(np.float32).astype(np.float64)
    hi = ((b + 1) << 16).view(np.float32).astype(np.float64)
    got = oracle.bf16_from_f64((lo + hi) / 2)
    want = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("x,want", [
    (1.0 + 2 ** -8, 0x3F80),               # tie -> even (down)
    (1.0 + 3 * 2 ** -8, 0x3F82),           # tie -> even (up)
    (1.0 + 2 ** -8 + 2 ** -40, 0x3F81),    # just above the tie: one rounding goes up (via fp32 it would tie)
    (-0.0, 0x8000),
    (2.0 ** -133, 0x0001),                 # smallest subnormal
    (2.0 ** -134, 0x0000),                 # tie between 0 and the smallest subnormal -> 0
    (3 * 2.0 ** -134, 0x0002),             # tie -> even
    (3.3895313892515355e38, 0x7F7F),       # largest finite bf16
    ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80),  # the midpoint to 2^128 -> inf (ties to the even 0x7F80)
    ((2 - 2 ** -8 - 2 ** -20) * 2.0 ** 127, 0x7F7F),  # just below it
    (float("inf"), 0x7F80),
    (-float("inf"), 0xFF80),
])
def test_bf16_rounding_hand_cases(x, want):
    assert int(oracle.bf16_from_f64(np.array([x]))[0]) == want


def test_bf16_rounding_nan():
    got = int(oracle.bf16_from_f64(np.array([float("nan")]))[0])
    assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0


def test_silu_against_torch_fp64_on_every_bf16_pattern():
    # h3 = 1.0 makes h = bf16(silu(h1)) (the product rounds to itself)
    h1 = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    ones = np.full_like(h1, 0x3F80)
    got = oracle.swiglu_bf16(h1, ones)
    with np.errstate(invalid="ignore"):
        x = torch.from_numpy((h1.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    ref = oracle.bf16_from_f64(torch.nn.functional.silu(x).numpy())
    nan = np.isnan(x.numpy())
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


def test_swiglu_hand_values():
    b = lambda v: oracle.bf16_from_f64(np.array([v], np.float64))
    sw = lambda a, c: int(oracle.swiglu_bf16(b(a), b(c))[0])
    # silu(1) = 0.7310585786... -> bf16 0.73046875; times 2 is exact
    assert sw(1.0, 2.0) == int(b(1.4609375)[0])
    # silu(v) = v exactly in fp64 for v >= 40; products in [128, 256) round to integers:
    assert sw(129.0, 1.5) == 0x4342        # 193.5 is a tie -> even 194
    assert sw(129.0, 1.0078125) == int(b(130.0)[0])   # 130.0078125 -> 130
    assert sw(200.0, 1.0078125) == int(b(202.0)[0])   # 201.5625 -> 202
    assert sw(0.0, 3.0) == 0x0000          # silu(0) = 0
    assert sw(-200.0, 3.0) == 0x8000       # silu(-200) = -0 after rounding, times 3 keeps the sign
    assert sw(5.0, 0.0) == 0x0000


def test_swiglu_gate_up_reduces_to_the_parts():
    # G=1, W = I and 2I: h1 and h3 are the dequantized x and twice it (the exact GEMM pin)
    M, D = 64, 64
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((M, D)).astype(np.float32)).to(torch.bfloat16)
    eye = torch.eye(D, dtype=torch.bfloat16)[None]
    two = (2 * torch.eye(D, dtype=torch.bfloat16))[None]
    o = oracle.swiglu_gate_up(u16(x), u16(eye), u16(two), [M])
    xq, xs = oracle.quantize_rows(u16(x))
    deq_x = oracle.dequant(xq, np.repeat(xs, 32, axis=1))
    assert np.array_equal(o["h1_f64"], deq_x) and np.array_equal(o["h3_f64"], 2 * deq_x)
    assert np.array_equal(o["h"], oracle.swiglu_bf16(o["h1"], o["h3"]))
    q, s = oracle.quantize_rows(o["h"])
    assert np.array_equal(o["h_q"], q) and np.array_equal(o["h_s"], s)
    qT, sT = oracle.quantize_cols(o["h"])
    assert np.array_equal(o["hT_q"], qT) and np.array_equal(o["hT_s"], sT)


def test_swiglu_backward_against_torch_autograd_ops():
    # fp64 torch ops restate the same derivative; the oracle rounds once per op, so on inputs
    # whose fp64 results round the same either way the patterns agree exactly
    rng = np.random.default_rng(7)
    n = 4096
    b16 = lambda a: oracle.bf16_from_f64(a)
    h1 = b16(rng.standard_normal(n) * 3)
    h3 = b16(rng.standard_normal(n))
    dh = b16(rng.standard_normal(n) * 1e-2)
    f = lambda u: torch.from_numpy((u.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    t1, t3, tg = f(h1), f(h3), f(dh)
    silu = f(b16(torch.nn.functional.silu(t1).numpy()))
    want3 = b16((tg * silu).numpy())
    dsilu = f(b16((tg * t3).numpy()))
    want1 = b16(torch.ops.aten.silu_backward(dsilu, t1).numpy())
    got1, got3 = oracle.swiglu_bwd_bf16(dh, h1, h3)
    assert np.array_equal(got3, want3)
    assert (got1 == want1).mean() > 0.999   # silu_backward's fp64 evaluation order differs from the oracle's


def test_swiglu_backward_hand_values():
    b = lambda v: oracle.bf16_from_f64(np.array([v], np.float64))
    one = lambda dh, a, u: [int(x[0]) for x in oracle.swiglu_bwd_bf16(b(dh), b(a), b(u))]
    # h1 = 0: sig = 1/2, silu = 0, silu' = 1/2 -> dh1 = bf16(dh * h3) / 2, dh3 = 0
    assert one(1.0, 0.0, 3.0) == [int(b(1.5)[0]), 0x0000]
    # large h1: silu(h1) = h1, silu' = 1 -> dh1 = dh * h3, dh3 = dh * h1
    assert one(0.5, 100.0, 2.0) == [int(b(1.0)[0]), int(b(50.0)[0])]
    # very negative h1: silu and its derivative vanish
    d1, d3 = one(1.0, -200.0, 3.0)
    assert (d1 & 0x7FFF) == 0 and (d3 & 0x7FFF) == 0
