#!/usr/bin/env python
"""Writes tests/golden/stability_words.txt: the random signs of the Hadamard transform and the
stochastic-rounding bytes that the readings of "MXFP8 (Micro-scaling FP8)", "Numerical
stability" draw from Philox4x32-10.

The generator here is a pure-Python Philox4x32-10 written from its definition in Salmon,
Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011): a 4 x 32-bit
counter and a 2 x 32-bit key, ten rounds; each round multiplies counter words 0 and 2 by the
round constants 0xD2511F53 and 0xCD9E8D57 into 64-bit products, and the new counter is
(hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)); the key is bumped by the
Weyl constants 0x9E3779B9 and 0xBB67AE85 after every round.  It shares no code with the C
oracle or the CUDA kernels, and it is checked against the published known-answer vectors
(philox4x32_10_kat.txt) before any value is written.

How each stored value is selected from the generator (the readings being pinned):
  signs  seed -> 32 characters; character i is '-' iff bit i (bit 0 = least significant) of
         output word 0 of Philox4x32-10 with counter (0, 0, 2, 0) and key
         (seed mod 2^32, seed >> 32) is set, else '+'.
  sr     (seed, r, c, C) -> the random byte of element (r, c) of an input with C columns:
         byte 8 * (r mod 2) + (c mod 8) of the 16-byte output (output word k holds bytes
         4k .. 4k+3, least significant first) for counter (b mod 2^32, floor(b / 2^32), 0, 0),
         b = floor(r / 2) * (C / 8) + floor(c / 8), and the same key.

    python tests/golden/make_stability_words.py      # rewrites the golden file
"""
from __future__ import annotations

import os

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "stability_words.txt")
KAT = os.path.join(HERE, "philox4x32_10_kat.txt")

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    c0, c1, c2, c3 = (int(v) & MASK for v in ctr)
    k0, k1 = (int(v) & MASK for v in key)
    for _ in range(10):
        p0 = M0 * c0
        p1 = M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & MASK, p1 & MASK, ((p0 >> 32) ^ c3 ^ k1) & MASK, p0 & MASK
        k0 = (k0 + W0) & MASK
        k1 = (k1 + W1) & MASK
    return [c0, c1, c2, c3]


def kat_rows():
    with open(KAT) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                yield [int(w, 16) for w in line.split()]


def check_kat():
    n = 0
    for row in kat_rows():
        assert philox4x32_10(row[0:4], row[4:6]) == row[6:10], "pure-Python Philox4x32-10 fails a known answer"
        n += 1
    assert n >= 3


def key_of(seed: int):
    return [seed & MASK, (seed >> 32) & MASK]


def signs(seed: int) -> str:
    w0 = philox4x32_10([0, 0, 2, 0], key_of(seed))[0]
    return "".join("-" if (w0 >> i) & 1 else "+" for i in range(32))


def sr_block(r: int, c: int, C: int) -> int:
    return (r // 2) * (C // 8) + c // 8


def sr_byte(seed: int, r: int, c: int, C: int) -> int:
    b = sr_block(r, c, C)
    out = philox4x32_10([b & MASK, (b >> 32) & MASK, 0, 0], key_of(seed))
    k = 8 * (r % 2) + c % 8
    return (out[k // 4] >> (8 * (k % 4))) & 0xFF


SIGN_SEEDS = [0, 1, 0x5EED, 0x0123456789ABCDEF, (1 << 40) + 3]
SR_CASES = [  # (seed, r, c, C): both row parities, all byte positions of a word, blocks past 2^32
    (0, 0, 0, 8), (0, 0, 5, 8), (0, 1, 2, 8), (0, 1, 7, 8),
    (0x5EED, 12345, 4321, 5120), (0x5EED, 12344, 4321, 5120), (0x5EED, 12345, 4326, 5120),
    (0x0123456789ABCDEF, 65599, 8191, 8192), (0x0123456789ABCDEF, 2, 9, 32),
    (0x0123456789ABCDEF, (1 << 23) + 3, 1030, 8192), (0x0123456789ABCDEF, (3 << 24) + 2, 17, 8192),
    ((1 << 63) + 11, 40001, 6, 5120), (42, 16383, 5119, 5120),
]


def main():
    check_kat()
    lines = [
        "# Random words of the stability-variant readings, written by make_stability_words.py from a",
        "# pure-Python Philox4x32-10 (Salmon et al., SC 2011) checked against philox4x32_10_kat.txt.",
        "# sign <seed hex> <32 signs>: sign i is '-' iff bit i of output word 0 of Philox4x32-10 with",
        "#      counter (0, 0, 2, 0), key (seed mod 2^32, seed >> 32) is set ('+' otherwise).",
        "# sr <seed hex> <r> <c> <C> <byte hex>: byte 8(r mod 2) + (c mod 8) of the Philox4x32-10 output",
        "#      (word k = bytes 4k..4k+3, least significant first) for counter (b mod 2^32, floor(b/2^32), 0, 0),",
        "#      b = floor(r/2)(C/8) + floor(c/8), and the same key.",
    ]
    for s in SIGN_SEEDS:
        lines.append(f"sign {s:x} {signs(s)}")
    for s, r, c, C in SR_CASES:
        lines.append(f"sr {s:x} {r} {c} {C} {sr_byte(s, r, c, C):02x}")
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(OUT)


if __name__ == "__main__":
    main()
