/*
 * mxfp8_oracle.c -- plain, slow, obviously-correct CPU oracle for MXFP8
 * dynamic quantization and the block-scaled grouped GEMM of MoE routed experts.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package
 * entry file and the CPU-baseline leg of bench.py load this library.  It shares
 * no code, header, table or constant generator with the CUDA path.
 *
 * What it computes (sources):
 *  - "MXFP8 (Micro-scaling FP8)" (sysdesign-wiki), section "Definition": one
 *    shared scale per small block of values; section "Low-precision Flash
 *    Attention": scales are generated along each GEMM's K dimension, and the
 *    [32, 32] square-block variant (item 3) is transpose invariant.
 *  - "MXFP8 training for MoEs" (theaicatchup), the paragraph on
 *    _to_mxfp8_then_scaled_grouped_mm: activations and weights are quantized
 *    dynamically, a scaled grouped GEMM runs, the output is in the original
 *    precision, and the op is differentiable (backprop mirrors the forward).
 *  - "[mxfp8 moe training] wrap 3d quantize tensor in custom ops" (pytorch/ao
 *    PR 3004): 3D expert-weight quantization, plain and column-wise.
 *  - The pages give no scale rule, rounding mode or encoding.  The oracle uses
 *    the OCP Microscaling Formats (MX) v1.0 rule: shared exponent
 *    floor(log2(amax)) - emax_elem with emax_elem = 8 for E4M3, clamped to the
 *    E8M0 range; an all-zero block takes the smallest scale 2^-127; elements are
 *    x * 2^-e rounded to nearest-even E4M3 and saturated at +-448.
 *
 * Deliberately different algorithms from the GPU path:
 *  - the shared exponent comes from frexp() on the fp64 amax (not from bf16
 *    exponent bits);
 *  - E4M3 encoding is an exhaustive nearest search over all finite codes with
 *    ties broken towards the even code (not a hardware cvt);
 *  - the GEMM is an fp64 dot product of dequantized values, per group, in
 *    natural k order.
 *
 * Pinned (tests/test_oracle_*.py): hand-worked blocks, a bit-level RNE written
 * independently in the tests, torch's float8_e4m3fn cast on unsaturated values,
 * round-trip error bounds, transpose invariance, blocked-layout bijection and
 * hand-computed positions, brute-force tiny GEMMs, the identity-weight case.
 * NaN/Inf input blocks: the OCP NaN scale (every element dequantizes to NaN)
 * and torch's float8_e4m3fn cast of a NaN with each element's sign.
 * SwiGLU stage: bf16 rounding pinned against torch's fp32->bf16 cast, hand
 * ties and a double-rounding case; silu against torch's fp64 silu.
 * Stability variants: Philox4x32-10 against its published known-answer
 * vectors; the Hadamard signs and the stochastic-rounding bytes (which output
 * byte, which counter) against values written by an independent pure-Python
 * Philox4x32-10 (tests/golden/stability_words.txt); stochastic rounding by hand
 * cases, an independent fp32 bit algorithm, exactness on the grid and its mean; the Hadamard butterflies against
 * scipy's Hadamard matrix on inputs where fp32 is exact, and orthogonality.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define BLK 32            /* elements per MX block */
#define E4M3_MAX 448.0    /* largest finite E4M3 magnitude */
#define E8M0_NAN 0xFF

/* ------------------------------------------------------------------ */
/* Scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> exact fp64 value (bf16 is the top half of an fp32). */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 (bias 7, no infinities, S.1111.111 = NaN) code -> fp64 value,
 * straight from the format definition: normal (1 + m/8) * 2^(E-7),
 * subnormal (m/8) * 2^(1-7). */
double oracle_e4m3_to_f64(uint8_t q) {
    int sign = (q >> 7) & 1;
    int ex = (q >> 3) & 0xF;
    int man = q & 7;
    double v;
    if (ex == 0xF && man == 7) return NAN;
    if (ex == 0)
        v = ldexp((double)man / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sign ? -v : v;
}

/* E8M0 scale byte -> 2^(s-127). */
double oracle_e8m0_to_f64(uint8_t s) {
    if (s == E8M0_NAN) return NAN;
    return ldexp(1.0, (int)s - 127);
}

/* Nearest finite E4M3 code to y by exhaustive search over the 127 non-negative
 * finite magnitudes (codes 0x00..0x7E); ties go to the code with an even
 * mantissa LSB; the sign is applied afterwards (so -tiny -> 0x80).
 * satfinite: a magnitude beyond 448 is first clamped to 448 (the nearest finite
 * code of any such value; clamping keeps the fp64 distances exact for huge y).
 * NaN input -> 0x7F with the sign kept. */
uint8_t oracle_e4m3_encode(double y) {
    int neg = signbit(y) ? 1 : 0;
    if (isnan(y)) return (uint8_t)(0x7F | (neg << 7));
    double a = fabs(y);
    if (a > E4M3_MAX) a = E4M3_MAX;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(best | (neg << 7));
}

/* Shared E8M0 scale byte of a block whose largest magnitude is amax (fp64):
 * e = floor(log2(amax)) - 8 via frexp (amax = f * 2^p, f in [0.5,1) so
 * floor(log2 amax) = p - 1), clamped to [-127, 127]; s = e + 127.
 * amax == 0 -> s = 0 (2^-127).  Non-finite amax -> 0xFF (NaN scale). */
uint8_t oracle_e8m0_from_amax(double amax) {
    if (isnan(amax) || isinf(amax)) return E8M0_NAN;
    if (amax == 0.0) return 0;
    int p;
    frexp(amax, &p);
    int e = (p - 1) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* ------------------------------------------------------------------ */
/* Block quantization                                                  */
/* ------------------------------------------------------------------ */

static uint8_t quantize_block_f64_rw(const double* v, int64_t n, uint8_t* q, int64_t qstride, const uint32_t* rw);

/* Quantize n values (already widened to fp64) sharing one scale.
 * Writes n codes to q (stride qstride) and returns the scale byte. */
static uint8_t quantize_block_f64(const double* v, int64_t n, uint8_t* q, int64_t qstride) {
    return quantize_block_f64_rw(v, n, q, qstride, NULL);
}

uint8_t oracle_e4m3_encode_sr(double y, uint32_t r);

/* As above; with rw != NULL each element is rounded stochastically with its
 * random word rw[i] (oracle_e4m3_encode_sr) instead of to nearest even. */
static uint8_t quantize_block_f64_rw(const double* v, int64_t n, uint8_t* q, int64_t qstride, const uint32_t* rw) {
    double amax = 0.0;
    int nonfinite = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (!isfinite(v[i])) nonfinite = 1;
        else if (fabs(v[i]) > amax) amax = fabs(v[i]);
    }
    if (nonfinite) {
        /* Reading for non-finite input (the pages are silent): NaN scale and
         * NaN codes with the element's sign. */
        for (int64_t i = 0; i < n; ++i) q[i * qstride] = (uint8_t)(0x7F | (signbit(v[i]) ? 0x80 : 0));
        return E8M0_NAN;
    }
    uint8_t s = oracle_e8m0_from_amax(amax);
    int e = (int)s - 127;
    for (int64_t i = 0; i < n; ++i)
        q[i * qstride] = rw ? oracle_e4m3_encode_sr(ldexp(v[i], -e), rw[i]) : oracle_e4m3_encode(ldexp(v[i], -e));
    return s;
}

/* Quantize a strided bf16 vector of length n (n % 32 == 0) in blocks of 32
 * consecutive elements: q[i] for element i, s[b] for block b. */
void oracle_quantize_vec(const uint16_t* x, int64_t n, int64_t xstride, uint8_t* q, uint8_t* s) {
    double v[BLK];
    for (int64_t b = 0; b < n / BLK; ++b) {
        for (int i = 0; i < BLK; ++i) v[i] = oracle_bf16_to_f64(x[(b * BLK + i) * xstride]);
        s[b] = quantize_block_f64(v, BLK, q + b * BLK, 1);
    }
}

/* Row-wise quantization of x[R, C] (blocks of 32 along C, i.e. along the
 * GEMM's K for an operand stored K-contiguous): q[R, C], compact s[R, C/32]. */
void oracle_quantize_rows(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, uint8_t* s) {
    for (int64_t r = 0; r < R; ++r)
        oracle_quantize_vec(x + r * C, C, 1, q + r * C, s + r * (C / BLK));
}

/* Column-wise quantization of x[R, C] (blocks of 32 consecutive rows of one
 * column), stored transposed: qT[C, R], compact sT[C, R/32]. */
void oracle_quantize_cols(const uint16_t* x, int64_t R, int64_t C, uint8_t* qT, uint8_t* sT) {
    for (int64_t c = 0; c < C; ++c)
        oracle_quantize_vec(x + c, R, C, qT + c * R, sT + c * (R / BLK));
}

/* 32x32 square-block quantization of x[R, C] (R, C % 32 == 0): one scale per
 * 32x32 tile, q[R, C] in place of x, compact s[R/32, C/32]. */
void oracle_quantize_32x32(const uint16_t* x, int64_t R, int64_t C, uint8_t* q, uint8_t* s) {
    double v[BLK * BLK];
    uint8_t qt[BLK * BLK];
    for (int64_t br = 0; br < R / BLK; ++br)
        for (int64_t bc = 0; bc < C / BLK; ++bc) {
            for (int i = 0; i < BLK; ++i)
                for (int j = 0; j < BLK; ++j)
                    v[i * BLK + j] = oracle_bf16_to_f64(x[(br * BLK + i) * C + bc * BLK + j]);
            s[br * (C / BLK) + bc] = quantize_block_f64(v, BLK * BLK, qt, 1);
            for (int i = 0; i < BLK; ++i)
                for (int j = 0; j < BLK; ++j)
                    q[(br * BLK + i) * C + bc * BLK + j] = qt[i * BLK + j];
        }
}

/* ------------------------------------------------------------------ */
/* Blocked (tensor-core) scale layout                                  */
/* ------------------------------------------------------------------ */
/* The scale matrix (rows x kb columns, kb = one 32-element block) is cut
 * into tiles of 128 rows x 4 block-columns, stored one after another with
 * the column tiles of a row tile adjacent.  Inside a 512-byte tile the row r
 * (0..127) is split as r = 32*i + j (i = r/32, j = r%32), and the byte for
 * (i, j, c) with c = kb%4 sits at j*16 + i*4 + c: row j of a 32x16-byte
 * matrix whose 16 bytes are the four 32-row quarters side by side.
 * Written here as an explicit tile walk, the GPU uses its own formula. */
int64_t oracle_blocked_offset(int64_t r, int64_t kb, int64_t kb_tiles) {
    int64_t tile_r = r / 128, in_r = r % 128;
    int64_t tile_c = kb / 4, in_c = kb % 4;
    int64_t tile_base = (tile_r * kb_tiles + tile_c) * 512;
    int64_t quarter = in_r / 32, lane = in_r % 32;
    return tile_base + lane * 16 + quarter * 4 + in_c;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Blocked layout with groups along the ROWS (fwd / dgrad A operand, and 3D
 * weights with G experts of equal size): group g owns rows [lo_g, hi_g) of the
 * compact scale matrix s[R, Kb]; in the blocked buffer each group starts on a
 * fresh 128-row tile: padded row base P_g = sum_{h<g} ceil(M_h/128)*128.
 * Kb is padded to a multiple of 4.  Every byte not holding a scale is 0.
 * ends[g] = cumulative end row of group g.  Returns the bytes written. */
int64_t oracle_blocked_rowgroups(const uint8_t* s, int64_t R, int64_t Kb, const int64_t* ends, int64_t G,
                                 uint8_t* out) {
    int64_t kb_tiles = ceil_div(Kb, 4);
    int64_t prow = 0;
    for (int64_t g = 0; g < G; ++g) prow += ceil_div(ends[g] - (g ? ends[g - 1] : 0), 128) * 128;
    int64_t total = prow * kb_tiles * 4;
    memset(out, 0, (size_t)total);
    int64_t base = 0;
    for (int64_t g = 0; g < G; ++g) {
        int64_t lo = g ? ends[g - 1] : 0, hi = ends[g];
        for (int64_t r = lo; r < hi; ++r)
            for (int64_t kb = 0; kb < Kb; ++kb)
                out[oracle_blocked_offset(base + (r - lo), kb, kb_tiles)] = s[r * Kb + kb];
        base += ceil_div(hi - lo, 128) * 128;
    }
    (void)R;
    return total;
}

/* Blocked layout with groups along the block-COLUMNS (wgrad operands, whose
 * contraction runs over the tokens of one group): s[R, Mb] with Mb = M/32;
 * group g owns block-columns [lo_g/32, hi_g/32) and starts on a fresh 4-column
 * tile: padded column base Q_g = sum_{h<g} ceil(M_h/128)*4.  Rows padded to a
 * multiple of 128.  ends[] are token offsets (multiples of 32).  Returns the
 * bytes written. */
int64_t oracle_blocked_colgroups(const uint8_t* s, int64_t R, int64_t Mb, const int64_t* ends, int64_t G,
                                 uint8_t* out) {
    int64_t qcols = 0;
    for (int64_t g = 0; g < G; ++g) qcols += ceil_div(ends[g] - (g ? ends[g - 1] : 0), 128) * 4;
    int64_t kb_tiles = qcols / 4;
    int64_t total = ceil_div(R, 128) * 128 * qcols;
    memset(out, 0, (size_t)total);
    int64_t base = 0;
    for (int64_t g = 0; g < G; ++g) {
        int64_t lo = (g ? ends[g - 1] : 0) / BLK, hi = ends[g] / BLK;
        for (int64_t r = 0; r < R; ++r)
            for (int64_t b = lo; b < hi; ++b)
                out[oracle_blocked_offset(r, base + (b - lo), kb_tiles)] = s[r * Mb + b];
        base += ceil_div((hi - lo) * BLK, 128) * 4;
    }
    return total;
}

/* ------------------------------------------------------------------ */
/* GEMMs (fp64, per group)                                             */
/* ------------------------------------------------------------------ */

/* deq(q, s) = E4M3(q) * 2^(s-127). */
static double deq(uint8_t q, uint8_t s) { return oracle_e4m3_to_f64(q) * oracle_e8m0_to_f64(s); }

/* One output element: sum_k deq(a[k], sa[k/32]) * deq(b[k], sb[k/32]),
 * fp64, k in natural order.  a, b are K-contiguous codes with compact scales. */
double oracle_dot(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb, int64_t K) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += deq(a[k], sa[k / BLK]) * deq(b[k], sb[k / BLK]);
    return acc;
}

/* Forward / dgrad form: rows of the token operand A (codes aq[M, K], compact
 * scales as[M, K/32]) in group g are contracted with expert g's matrix
 * bq[g] ([Nb, K], scales bs[g] [Nb, K/32]):  out[m, n] = sum_k A[m,k] B_g[n,k].
 * ends[g] = cumulative end row of group g.  out is fp64 [M, Nb].
 *   fwd:   A = activations [M,K],   B_g = W[g]   [N,K]
 *   dgrad: A = dOut        [M,N],   B_g = W[g]^T [K,N] */
void oracle_grouped_mm_rows(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs,
                            const int64_t* ends, int64_t G, int64_t M, int64_t Nb, int64_t K, double* out) {
    int64_t Kb = K / BLK;
    for (int64_t g = 0; g < G; ++g) {
        int64_t lo = g ? ends[g - 1] : 0, hi = ends[g];
        const uint8_t* bqg = bq + g * Nb * K;
        const uint8_t* bsg = bs + g * Nb * Kb;
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t m = lo; m < hi; ++m)
            for (int64_t n = 0; n < Nb; ++n)
                out[m * Nb + n] = oracle_dot(aq + m * K, as + m * Kb, bqg + n * K, bsg + n * Kb, K);
    }
    (void)M;
}

/* Wgrad form: for each group g, out[g][n, k] = sum_{m in g} dOut[m,n] A[m,k],
 * from the column-quantized operands dOut^T (codes dq[N, M], compact scales
 * ds[N, M/32]) and A^T (codes aq[K, M], scales as[K, M/32]); the contraction
 * runs over the group's tokens only.  An empty group gives all zeros. */
void oracle_grouped_mm_wgrad(const uint8_t* dq, const uint8_t* ds, const uint8_t* aq, const uint8_t* as,
                             const int64_t* ends, int64_t G, int64_t M, int64_t N, int64_t K, double* out) {
    int64_t Mb = M / BLK;
    for (int64_t g = 0; g < G; ++g) {
        int64_t lo = g ? ends[g - 1] : 0, hi = ends[g];
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t k = 0; k < K; ++k)
                out[(g * N + n) * K + k] =
                    oracle_dot(dq + n * M + lo, ds + n * Mb + lo / BLK, aq + k * M + lo, as + k * Mb + lo / BLK, hi - lo);
    }
}

/* ------------------------------------------------------------------ */
/* Stability variants: stochastic rounding, random Hadamard transform  */
/* ------------------------------------------------------------------ */
/* "MXFP8 (Micro-scaling FP8)", "Numerical stability": random Hadamard
 * transforms spread outliers before quantization, and stochastic rounding
 * removes the bias of deterministic rounding.  The pages define neither; the
 * readings below are written identically (but independently) on the GPU. */

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011): ten rounds of two 32x32->64-bit products with
 * the multipliers 0xD2511F53 and 0xCD9E8D57, the key bumped by 0x9E3779B9 and
 * 0xBB67AE85 between rounds.  Pinned by the published known-answer vectors. */
void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1, n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The random byte of element (r, c) of an input with C columns (C % 8 == 0):
 * byte 8 * (r mod 2) + (c mod 8) of the 16-byte Philox4x32-10 output (word k
 * holds bytes 4k .. 4k+3, least significant first) for counter (b mod 2^32,
 * b / 2^32, 0, 0), b = floor(r / 2) * (C / 8) + floor(c / 8), and key (seed
 * low 32 bits, seed high 32 bits).  One draw serves a 2 x 8 block; the
 * row-wise and the column-wise copy of an element use the same byte. */
uint8_t oracle_sr_byte(uint64_t seed, uint64_t r, uint64_t c, uint64_t C) {
    uint64_t b = (r / 2) * (C / 8) + c / 8;
    uint32_t ctr[4] = {(uint32_t)b, (uint32_t)(b >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    oracle_philox4x32_10(ctr, key, o);
    unsigned k = 8u * (unsigned)(r % 2) + (unsigned)(c % 8);
    return (uint8_t)((o[k / 4] >> (8 * (k % 4))) & 0xFFu);
}

/* Stochastic rounding of y to E4M3 (satfinite).  For |y| between the
 * consecutive finite magnitudes lo <= |y| < hi, let F = floor((|y| - lo) /
 * (hi - lo) * 256), the position inside the step in units of 1/256 of it.  The
 * magnitude rounds up to hi iff F + u >= 256, so with u a uniform byte it rounds
 * up with probability F / 256.  |y| >= 448 gives 448; the sign is applied
 * afterwards; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode_sr(double y, uint32_t u) {
    int neg = signbit(y) ? 1 : 0;
    if (isnan(y)) return (uint8_t)(0x7F | (neg << 7));
    double a = fabs(y);
    int code;
    if (a >= E4M3_MAX) {
        code = 0x7E;
    } else {
        int lo = 0;
        for (int c = 0; c <= 0x7E; ++c)
            if (oracle_e4m3_to_f64((uint8_t)c) <= a) lo = c;
        double vlo = oracle_e4m3_to_f64((uint8_t)lo), vhi = oracle_e4m3_to_f64((uint8_t)(lo + 1));
        double F = floor((a - vlo) / (vhi - vlo) * 256.0);
        code = (F + (double)(u & 0xFFu) >= 256.0) ? lo + 1 : lo;
    }
    return (uint8_t)(code | (neg << 7));
}

/* The 32 signs D of the Hadamard transform: bit i of word 0 of Philox4x32-10
 * with counter (0, 0, 2, 0) and the seed as key; a set bit means -1. */
void oracle_rht_signs(uint64_t seed, int8_t* d) {
    uint32_t ctr[4] = {0u, 0u, 2u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    oracle_philox4x32_10(ctr, key, o);
    for (int i = 0; i < BLK; ++i) d[i] = ((o[0] >> i) & 1u) ? -1 : 1;
}

/* y = c * H * (D x) for one block of 32, in fp32: the signs flip, then the
 * Sylvester-ordered Hadamard matrix (H[i][j] = (-1)^popcount(i & j)) is applied
 * as butterflies (a, b) -> (a + b, a - b) over the pairs (i, i + h) for
 * h = 1, 2, 4, 8, 16 in that order, each sum rounded to fp32; finally every
 * element is multiplied by c = fp32(1/sqrt(32)).  H D / sqrt(32) is orthogonal,
 * so two operands transformed alike along a GEMM's K keep their product. */
void oracle_rht32(const float* x, const int8_t* d, float* y) {
    float t[BLK];
    for (int i = 0; i < BLK; ++i) t[i] = d[i] < 0 ? -x[i] : x[i];
    for (int h = 1; h < BLK; h <<= 1)
        for (int i = 0; i < BLK; ++i)
            if ((i & h) == 0) {
                float a = t[i], b = t[i + h];
                t[i] = a + b;
                t[i + h] = a - b;
            }
    const float c = (float)(1.0 / sqrt(32.0));
    for (int i = 0; i < BLK; ++i) y[i] = t[i] * c;
}

/* One block of 32 bf16 values (element i at x[i * xstride], at row r0 + i * dr,
 * column c0 + i * dc of an input with C columns) quantized with options:
 * bit 0 = stochastic rounding (oracle_sr_byte), bit 1 = Hadamard transform first. */
static uint8_t quantize_block_opts(const uint16_t* x, int64_t xstride, uint64_t r0, uint64_t c0, uint64_t dr,
                                   uint64_t dc, uint64_t C, unsigned opts, uint64_t seed, uint8_t* q, int64_t qstride) {
    double v[BLK];
    uint32_t rw[BLK];
    if (opts & 2u) {
        float xf[BLK], yf[BLK];
        int8_t d[BLK];
        oracle_rht_signs(seed, d);
        for (int i = 0; i < BLK; ++i) xf[i] = (float)oracle_bf16_to_f64(x[i * xstride]);
        oracle_rht32(xf, d, yf);
        for (int i = 0; i < BLK; ++i) v[i] = (double)yf[i];
    } else {
        for (int i = 0; i < BLK; ++i) v[i] = oracle_bf16_to_f64(x[i * xstride]);
    }
    if (opts & 1u)
        for (int i = 0; i < BLK; ++i) rw[i] = oracle_sr_byte(seed, r0 + (uint64_t)i * dr, c0 + (uint64_t)i * dc, C);
    return quantize_block_f64_rw(v, BLK, q, qstride, (opts & 1u) ? rw : NULL);
}

/* One block of 32 contiguous bf16 values whose element i sits at row r0 + i * dr, column
 * c0 + i * dc of an input with C columns (a row block: dr = 0, dc = 1; a column block:
 * dr = 1, dc = 0), quantized with options: 32 codes into q32, returns the scale byte (for
 * checking single blocks of a large tensor). */
uint8_t oracle_quantize_block_at(const uint16_t* x32, uint64_t r0, uint64_t c0, uint64_t dr, uint64_t dc, uint64_t C,
                                 unsigned opts, uint64_t seed, uint8_t* q32) {
    return quantize_block_opts(x32, 1, r0, c0, dr, dc, C, opts, seed, q32, 1);
}

/* Row-wise quantization of x[R, C] with options (see quantize_block_opts). */
void oracle_quantize_rows_opts(const uint16_t* x, int64_t R, int64_t C, unsigned opts, uint64_t seed, uint8_t* q,
                               uint8_t* s) {
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < C / BLK; ++b)
            s[r * (C / BLK) + b] = quantize_block_opts(x + r * C + b * BLK, 1, (uint64_t)r, (uint64_t)(b * BLK), 0, 1,
                                                       (uint64_t)C, opts, seed, q + r * C + b * BLK, 1);
}

/* Column-wise quantization of x[R, C] with options, stored transposed. */
void oracle_quantize_cols_opts(const uint16_t* x, int64_t R, int64_t C, unsigned opts, uint64_t seed, uint8_t* qT,
                               uint8_t* sT) {
    for (int64_t c = 0; c < C; ++c)
        for (int64_t b = 0; b < R / BLK; ++b)
            sT[c * (R / BLK) + b] = quantize_block_opts(x + b * BLK * C + c, C, (uint64_t)(b * BLK), (uint64_t)c, 1, 0,
                                                        (uint64_t)C, opts, seed, qT + c * R + b * BLK, 1);
}

/* ------------------------------------------------------------------ */
/* SwiGLU stage of a routed expert (bf16 rounding points)              */
/* ------------------------------------------------------------------ */
/* "feat(moe): add MoK MXFP8 expert support" (gate / up / down routed-expert
 * weights) and "MXFP8 (Micro-scaling FP8)", "Neutralizing quantization
 * overhead" (quantization fused into the kernel that produces the activation).
 * The pages give no formula for the expert's activation; the reading is the
 * SwiGLU of an elementwise bf16 evaluation:
 *   h1 = bf16(x Wg^T), h3 = bf16(x Wu^T), s = bf16(silu(h1)), h = bf16(s * h3),
 * with silu(v) = v / (1 + e^-v).  Every bf16() is round-to-nearest-even of the
 * exact value (computed here in fp64). */

/* fp64 -> bf16 bit pattern, nearest with ties to the even pattern, directly
 * from the fp64 value (never through fp32: that would round twice).  Magnitudes
 * at or past the midpoint between the largest finite bf16 and 2^128 give inf;
 * NaN gives the quiet NaN 0x7FC0 with the sign. */
uint16_t oracle_bf16_from_f64(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int E;
    frexp(a, &E);                       /* a = m * 2^E, m in [0.5, 1) */
    int qexp = E - 8;                   /* 8 significant bits: quantum 2^(E-8) */
    if (qexp < -133) qexp = -133;       /* subnormal quantum 2^-133 */
    double n = ldexp(a, -qexp);         /* exact: power-of-two scaling */
    double lo = floor(n), frac = n - lo;
    double r = lo;
    if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0)) r = lo + 1.0;
    double v = ldexp(r, qexp);
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;                 /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

void oracle_bf16_from_f64_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_f64(x[i]);
}

/* h = bf16( bf16(silu(h1)) * h3 ) elementwise over bf16 bit patterns. */
void oracle_swiglu_bf16(const uint16_t* h1, const uint16_t* h3, int64_t n, uint16_t* h) {
    for (int64_t i = 0; i < n; ++i) {
        double a = oracle_bf16_to_f64(h1[i]);
        double s = oracle_bf16_to_f64(oracle_bf16_from_f64(a / (1.0 + exp(-a))));
        h[i] = oracle_bf16_from_f64(s * oracle_bf16_to_f64(h3[i]));  /* 8 x 8 significant bits: exact in fp64 */
    }
}

/* Backward of h = silu(h1) * h3 with the rounding points of the bf16 autograd ops, all
 * values bf16 patterns, arithmetic in fp64 with one rounding per op:
 *   dh3 = bf16(dh * bf16(silu(h1)))
 *   dh1 = bf16(bf16(dh * h3) * sig * (1 + h1 * (1 - sig))),  sig = 1 / (1 + e^-h1)
 * (the derivative of silu(x) = x * sig(x) is sig * (1 + x * (1 - sig))). */
void oracle_swiglu_bwd_bf16(const uint16_t* dh, const uint16_t* h1, const uint16_t* h3, int64_t n, uint16_t* dh1,
                            uint16_t* dh3) {
    for (int64_t i = 0; i < n; ++i) {
        double g = oracle_bf16_to_f64(dh[i]), a = oracle_bf16_to_f64(h1[i]), u = oracle_bf16_to_f64(h3[i]);
        double sig = 1.0 / (1.0 + exp(-a));
        double silu = oracle_bf16_to_f64(oracle_bf16_from_f64(a * sig));
        dh3[i] = oracle_bf16_from_f64(g * silu);
        double dsilu = oracle_bf16_to_f64(oracle_bf16_from_f64(g * u));
        dh1[i] = oracle_bf16_from_f64(dsilu * sig * (1.0 + a * (1.0 - sig)));
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Thread count of the OpenMP loops above (the per-group GEMMs); no effect without OpenMP.  Lets
 * a caller time the same oracle single-threaded and over all host cores. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
