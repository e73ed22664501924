#!/usr/bin/env python
"""Writes tests/golden/stability_words.txt: the random signs of the Hadamard transform and the
stochastic-rounding words that the readings of "MXFP8 (Micro-scaling FP8)", "Numerical
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
  sr     (seed, n, dir) -> output word (n mod 4) of Philox4x32-10 with counter
         (floor(n / 4) mod 2^32, floor(n / 2^34), dir, 0) and the same key.

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


def sr_word(seed: int, n: int, direction: int) -> int:
    out = philox4x32_10([(n >> 2) & MASK, (n >> 34) & MASK, direction, 0], key_of(seed))
    return out[n & 3]


SIGN_SEEDS = [0, 1, 0x5EED, 0x0123456789ABCDEF, (1 << 40) + 3]
SR_CASES = [
    (0, 0, 0), (0, 1, 1), (0, 2, 0), (0, 3, 1),
    (0x5EED, 12345, 0), (0x5EED, 12345, 1),
    (0x0123456789ABCDEF, 7, 0), (0x0123456789ABCDEF, (1 << 32) + 6, 1),
    (0x0123456789ABCDEF, (1 << 34) + 5, 0), (0x0123456789ABCDEF, (1 << 34) + 5, 1),
    ((1 << 63) + 11, (3 << 34) + (1 << 33) + 2, 1), (42, 16384 * 5120 - 1, 0),
]


def main():
    check_kat()
    lines = [
        "# Random words of the stability-variant readings, written by make_stability_words.py from a",
        "# pure-Python Philox4x32-10 (Salmon et al., SC 2011) checked against philox4x32_10_kat.txt.",
        "# sign <seed hex> <32 signs>: sign i is '-' iff bit i of output word 0 of Philox4x32-10 with",
        "#      counter (0, 0, 2, 0), key (seed mod 2^32, seed >> 32) is set ('+' otherwise).",
        "# sr <seed hex> <n hex> <dir> <word hex>: output word (n mod 4) of Philox4x32-10 with counter",
        "#      (floor(n/4) mod 2^32, floor(n/2^34), dir, 0) and the same key.",
    ]
    for s in SIGN_SEEDS:
        lines.append(f"sign {s:x} {signs(s)}")
    for s, n, d in SR_CASES:
        lines.append(f"sr {s:x} {n:x} {d} {sr_word(s, n, d):08x}")
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(OUT)


if __name__ == "__main__":
    main()
