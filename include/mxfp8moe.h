/*
 * mxfp8moe.h -- C ABI of the GB300 (sm_103a) MXFP8 routed-expert hot path:
 * dynamic MXFP8 quantization plus block-scaled grouped GEMMs (forward, dgrad,
 * wgrad) over a token-offsets array, the computation behind
 * _to_mxfp8_then_scaled_grouped_mm.
 *
 * Sources (web pages; the paragraph or section named):
 *  [P1] "MXFP8 training for MoEs" (theaicatchup.com): the engine paragraph on
 *       _to_mxfp8_then_scaled_grouped_mm -- activations and weights are quantized
 *       dynamically to MXFP8, a scaled grouped GEMM runs, the output comes back
 *       in the original precision, the op is differentiable; "Why Does MXFP8
 *       Speed Up MoE Training": routed experts are grouped GEMMs over many small
 *       matrices and backprop mirrors the forward.
 *  [P2] "[mxfp8 moe training] wrap 3d quantize tensor in custom ops and
 *       integrate it" (pytorch/ao PR 3004): 3D expert-weight quantization, the
 *       column-wise 3D kernel, the per-group blocked scale format.
 *  [P3] "MXFP8 (Micro-scaling FP8)" (sysdesign-wiki): "Definition" (one shared
 *       scale per small block); "Low-precision Flash Attention" (scales along
 *       each GEMM's K; scale bits by bit manipulation; [32, 32] blocks).
 *  [P4] "feat(moe): add MoK MXFP8 expert support" (NVIDIA-NeMo/Automodel PR
 *       3606): each expert weight is carried as (weight_fp8, weight_scale,
 *       weight_t_fp8, weight_t_scale).
 * The pages fix neither the scale rule nor the encodings; this library uses
 * the OCP Microscaling (MX) v1.0 rule: per block of 32 elements,
 * e = floor(log2(amax)) - 8 clamped to [-127, 127], scale byte s = e + 127
 * (E8M0, value 2^(s-127)), an all-zero block gets s = 0, and each element is
 * x * 2^-e rounded to nearest-even E4M3 and saturated to +-448.  A block
 * holding Inf or NaN gets s = 0xFF and every code 0x7F with the element's sign.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory, keeps no state between calls (apart from a per-device
 *    architecture check), never synchronizes, and enqueues its work on `stream`.
 *  - Row-major, contiguous.  bf16 = IEEE bfloat16, e4m3 = one byte per element,
 *    E8M0 scales = one byte per 32-element block.
 *  - Group offsets `offs` (int32, device, length G) are cumulative END rows:
 *    group g holds rows [offs[g-1], offs[g]) with offs[-1] = 0, offs[G-1] = M.
 *    An empty group repeats the previous offset.  Kernels clamp the offsets into
 *    [0, M] so no access leaves the buffers even for bad offsets; bad offsets
 *    are reported through `dev_status` by mxfp8_check_offsets().
 *  - Argument errors are returned synchronously before any launch.  Errors the
 *    device finds are written to `*dev_status` (int32, device, nullable; the
 *    first error sticks; the caller zeroes it and reads it after the stream
 *    synchronizes).  No kernel traps.
 *  - Outputs are fully overwritten, including zero dW for empty groups and the
 *    zero padding bytes of blocked scales.
 *
 * Scale layouts:
 *  - MXFP8_SCALES_COMPACT: S[R][C/32] row-major, for an operand of R rows of C
 *    elements quantized along C.
 *  - MXFP8_SCALES_BLOCKED: the tensor-core layout (NVIDIA's documented 1D block
 *    scaling factor layout for block-scaled MMA).  The scale matrix is cut into
 *    tiles of 128 rows x 4 block-columns (512 bytes); tiles are stored with the
 *    column tiles of one row band adjacent; inside a tile, row r = 32*i + j and
 *    block-column c go to byte j*16 + i*4 + c.  Bytes that hold no scale are 0.
 *      * row groups (operands quantized along K whose rows are grouped tokens or
 *        experts): each group starts on a fresh 128-row tile, so group g's
 *        rows begin at padded row P_g = sum_{h<g} ceil(M_h/128)*128;
 *        column tiles per row band Ct = ceil(C/128).
 *      * column groups (column-wise quantized operands of the wgrad, whose
 *        32-blocks run along the tokens): rows padded to ceil(R/128)*128; group g
 *        starts on a fresh column tile, at padded block-column
 *        Q_g = sum_{h<g} ceil(M_h/128)*4; Ct = sum_g ceil(M_g/128).
 *      * 3D expert weights: each expert is its own matrix in that layout, expert
 *        g at byte offset g * (per-expert blocked bytes).
 *    A buffer sized with the upper bounds below may be larger than the layout's
 *    extent; bytes past the extent are not written.
 */
#ifndef MXFP8MOE_H
#define MXFP8MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mxfp8_stream_t; /* same object as cudaStream_t; NULL = legacy default stream */

typedef enum {
    MXFP8_OK = 0,
    MXFP8_ERR_NULL = 1,      /* a required pointer is NULL */
    MXFP8_ERR_SHAPE = 2,     /* a size is negative, zero where not allowed, or too large */
    MXFP8_ERR_ALIGN = 3,     /* K or N not a multiple of 32, M not a multiple of 32 where required,
                                or a pointer not 16-byte aligned */
    MXFP8_ERR_LAYOUT = 4,    /* unknown direction / scale-layout combination */
    MXFP8_ERR_ARCH = 5,      /* the current device is not sm_103 */
    MXFP8_ERR_LAUNCH = 6,    /* a CUDA launch or query failed */
    MXFP8_ERR_OFFSETS = 7,   /* device-detected: offsets not monotone, not ending at M, or a group
                                size not a multiple of the required alignment */
    MXFP8_ERR_TIMEOUT = 8,   /* device-detected: a bounded wait inside a kernel ran out */
    MXFP8_ERR_DRIVER = 9     /* TMA descriptor encoding failed */
} mxfp8_status_t;

/* Quantization directions (bit mask). */
enum {
    MXFP8_ROW = 1,        /* blocks of 32 along the last dim (K of x[M,K]) -> q[M,K] */
    MXFP8_COL = 2,        /* blocks of 32 along the first dim, stored transposed -> qT[K,M] */
    MXFP8_BLOCK32X32 = 4  /* one scale per 32x32 tile -> q[M,K], compact scales [M/32, K/32] */
};

enum { MXFP8_SCALES_COMPACT = 0, MXFP8_SCALES_BLOCKED = 1 };

/* Options of mxfp8_quantize_2d_opts (bit mask). */
enum {
    MXFP8_OPT_STOCHASTIC = 1,     /* stochastic rounding of every code (both copies) */
    MXFP8_OPT_HADAMARD_ROW = 2,   /* random Hadamard transform of each 32-block of the row-wise copy */
    MXFP8_OPT_HADAMARD_COL = 4    /* random Hadamard transform of each 32-block of the column-wise copy */
};

/* Largest number of groups / experts a call accepts. */
#define MXFP8_MAX_GROUPS 1024

/* ----------------------------------------------------------------------------
 * mxfp8_quantize_2d -- dynamic MXFP8 quantization of a bf16 matrix x[M, K].
 * [P1] engine paragraph (dynamic quantization of activations before the scaled
 * grouped GEMM); [P3] "Low-precision Flash Attention" (scales along each GEMM's
 * K, so the backward's transposed operands get their own, column-wise scales;
 * [32, 32] square blocks, item 3).
 *
 *   dirs = MXFP8_ROW, MXFP8_COL, MXFP8_ROW|MXFP8_COL (one read of x, both
 *          outputs) or MXFP8_BLOCK32X32 (alone).
 *   ROW:  q_row [M, K] e4m3; s_row compact [M, K/32] or blocked with row groups
 *         from `offs` (offs NULL or G <= 1: one group of M rows).
 *   COL:  q_col [K, M] e4m3 (M contiguous); s_col compact [K, M/32] or blocked
 *         with column groups from `offs`.  Requires M % 32 == 0 and every group
 *         size % 32 == 0 (device-checked by mxfp8_check_offsets).
 *   BLOCK32X32: q_row [M, K]; s_row compact [M/32, K/32] (scale_layout must be
 *         MXFP8_SCALES_COMPACT); M % 32 == 0.
 *   K % 32 == 0 always.  Unused outputs may be NULL.
 *   Returns MXFP8_ERR_ALIGN / _SHAPE / _NULL / _LAYOUT synchronously.
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_quantize_2d(const void* x_bf16, int64_t M, int64_t K, unsigned dirs, int scale_layout,
                                 const int32_t* offs, int32_t G, void* q_row, void* s_row, void* q_col,
                                 void* s_col, int32_t* dev_status, mxfp8_stream_t stream);

/* ----------------------------------------------------------------------------
 * mxfp8_quantize_2d_opts -- mxfp8_quantize_2d with the stability variants of
 * [P3] "Numerical stability" (random Hadamard transforms spread outliers before
 * quantization; stochastic rounding removes the bias of deterministic rounding).
 * The pages define neither; this library's readings:
 *   random words: element (r, c) of x (index n = r*K + c) of the row-wise copy
 *     (dir 0) or the column-wise copy (dir 1) takes word n % 4 of Philox4x32-10
 *     (Salmon et al., SC 2011) with counter (n / 4 mod 2^32, n / 2^34, dir, 0)
 *     and key (seed mod 2^32, seed / 2^32).
 *   MXFP8_OPT_STOCHASTIC: the scale rule is unchanged; each scaled element y is
 *     rounded between the neighbouring finite E4M3 magnitudes lo <= |y| < hi:
 *     up iff F + (word >> 12) >= 2^20, F = floor((|y| - lo) / (hi - lo) * 2^20);
 *     |y| >= 448 gives 448.  So y rounds up with probability F / 2^20.
 *   MXFP8_OPT_HADAMARD_ROW / _COL: every 32-block along the copy's axis becomes
 *     y = c * H * (D x) in fp32 before quantization: D = diag(signs), sign i
 *     negative iff bit i of word 0 of Philox4x32-10(counter (0, 0, 2, 0), key as
 *     above) is set; H the Sylvester-ordered 32x32 Hadamard matrix applied as
 *     butterflies (a, b) -> (a + b, a - b) over the pairs (i, i + h) for
 *     h = 1, 2, 4, 8, 16 in that order, each rounded to fp32; c = fp32(1/sqrt(32)).
 *     H D / sqrt(32) is orthogonal: two operands transformed with the same seed
 *     along a GEMM's contraction keep their product (e.g. dOut and A along the
 *     tokens for the wgrad).  Scales then come from the fp32 amax by the same
 *     rule; a block with a non-finite value gets codes 0x7F of unspecified sign.
 *   dirs: MXFP8_ROW, MXFP8_COL or both (no BLOCK32X32); each HADAMARD bit needs
 *     its copy.  opts = 0 is exactly mxfp8_quantize_2d.  Other arguments,
 *     layouts and errors as for mxfp8_quantize_2d; unknown option bits:
 *     MXFP8_ERR_LAYOUT.
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_quantize_2d_opts(const void* x_bf16, int64_t M, int64_t K, unsigned dirs, int scale_layout,
                                      const int32_t* offs, int32_t G, unsigned opts, uint64_t seed, void* q_row,
                                      void* s_row, void* q_col, void* s_col, int32_t* dev_status,
                                      mxfp8_stream_t stream);

/* ----------------------------------------------------------------------------
 * mxfp8_quantize_3d_experts -- quantize expert weights w[G, N, K] (bf16).
 * [P2] (3D quantize custom op; column-wise 3D kernel); [P4] (weight_fp8,
 * weight_scale, weight_t_fp8, weight_t_scale quadruple).
 *
 *   dirs & MXFP8_ROW ("plain", along K, for the forward):
 *        q [G, N, K], s per expert [N, K/32] (compact) or blocked.
 *   dirs & MXFP8_COL ("transposed", along N, for dgrad):
 *        qT [G, K, N] (N contiguous), sT per expert [K, N/32] compact or blocked.
 *   Both bits: one read of w.  N % 32 == 0, K % 32 == 0.
 *   dirs | MXFP8_BLOCK32X32 (with ROW and/or COL): [32, 32] square blocks
 *        ([P3] "Low-precision Flash Attention", item 3: one scale per 32x32
 *        block makes the quantization transpose invariant, so one quantization
 *        serves the forward and the dgrad).  One scale per 32x32 block of each
 *        expert; qT holds exactly the codes of q, transposed.  s and sT repeat the
 *        block's scale on each of its 32 rows (columns), in the compact or blocked
 *        layout above, so the grouped GEMMs take them unchanged.
 *   Per-expert scale strides: compact N*K/32 (s) and K*N/32 (sT); blocked
 *   ceil(N/128)*128*ceil(K/128)*4 (s) and ceil(K/128)*128*ceil(N/128)*4 (sT).
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_quantize_3d_experts(const void* w_bf16, int32_t G, int64_t N, int64_t K, unsigned dirs,
                                         int scale_layout, void* q, void* s, void* qT, void* sT,
                                         int32_t* dev_status, mxfp8_stream_t stream);

/* ----------------------------------------------------------------------------
 * Block-scaled grouped GEMMs.  All operands are e4m3 codes with BLOCKED E8M0
 * scales along the contraction dim; fp32 accumulation in tensor memory; bf16
 * output rounded to nearest-even.  [P1] engine paragraph and "Why Does MXFP8
 * Speed Up MoE Training" (grouped GEMMs for routed experts; backprop mirrors
 * the forward); [P3] "Low-precision Flash Attention" (scales along each GEMM's K).
 *
 * mxfp8_grouped_mm_fwd:   out[m, n] = sum_k A[m,k] * W[g][n,k],  m in group g
 *   a_q [M, K], a_s blocked row groups (offs), w_q [G, N, K], w_s blocked per
 *   expert (N rows, K/32 cols); out [M, N] bf16.
 * mxfp8_grouped_mm_dgrad: dA[m, k] = sum_n dOut[m,n] * W[g][n,k]
 *   dout_q [M, N] (quantized along N), dout_s blocked row groups; wt_q [G, K, N]
 *   (3D transposed quantization), wt_s blocked per expert (K rows, N/32 cols);
 *   da [M, K] bf16.
 * mxfp8_grouped_mm_wgrad: dW[g][n, k] = sum_{m in g} dOut[m,n] * A[m,k]
 *   doutT_q [N, M], doutT_s blocked column groups (rows N); aT_q [K, M],
 *   aT_s blocked column groups (rows K) -- both from mxfp8_quantize_2d(COL);
 *   dw [G, N, K] bf16; an empty group gives dW[g] = 0.  M % 32 == 0 and
 *   every group size % 32 == 0.
 * Shapes: K % 32 == 0, N % 32 == 0, 1 <= G <= MXFP8_MAX_GROUPS; every pointer
 * 16-byte aligned.  M may be 0 (nothing but the wgrad zero fill runs).
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_grouped_mm_fwd(const void* a_q, const void* a_s, const void* w_q, const void* w_s,
                                    const int32_t* offs, int32_t G, int64_t M, int64_t N, int64_t K, void* out_bf16,
                                    int32_t* dev_status, mxfp8_stream_t stream);
mxfp8_status_t mxfp8_grouped_mm_dgrad(const void* dout_q, const void* dout_s, const void* wt_q, const void* wt_s,
                                      const int32_t* offs, int32_t G, int64_t M, int64_t N, int64_t K,
                                      void* da_bf16, int32_t* dev_status, mxfp8_stream_t stream);
/* mxfp8_grouped_mm_dgrad2: the sum of two dgrads over the same groups, in one GEMM whose contraction
 *   runs first over (dout1, wt1) and then over (dout2, wt2) into one fp32 accumulator, rounded to bf16
 *   once: dA[m, k] = sum_n dOut1[m,n] W1[g][n,k] + sum_n dOut2[m,n] W2[g][n,k].  Both pairs have the
 *   shapes and layouts of mxfp8_grouped_mm_dgrad.  The SwiGLU expert's input gradient
 *   dx = dh1 Wg + dh3 Wu is one call (the gate/up branches of "feat(moe): add MoK MXFP8 expert
 *   support").
 */
mxfp8_status_t mxfp8_grouped_mm_dgrad2(const void* dout1_q, const void* dout1_s, const void* wt1_q, const void* wt1_s,
                                       const void* dout2_q, const void* dout2_s, const void* wt2_q, const void* wt2_s,
                                       const int32_t* offs, int32_t G, int64_t M, int64_t N, int64_t K, void* da_bf16,
                                       int32_t* dev_status, mxfp8_stream_t stream);
mxfp8_status_t mxfp8_grouped_mm_wgrad(const void* doutT_q, const void* doutT_s, const void* aT_q,
                                      const void* aT_s, const int32_t* offs, int32_t G, int64_t M, int64_t N,
                                      int64_t K, void* dw_bf16, int32_t* dev_status, mxfp8_stream_t stream);

/* ----------------------------------------------------------------------------
 * mxfp8_grouped_mm_swiglu_fwd -- the gate and up GEMMs of a SwiGLU routed expert
 * with the SwiGLU and its MXFP8 quantization fused into their epilogue.
 * [P3] "Neutralizing quantization overhead" (fuse the quantization of
 * activations into the kernel that produces them); [P4] (gate/up/down routed
 * expert weights).  For rows m of group g:
 *   h1[m, n] = bf16( sum_d X[m,d] Wg[g][n,d] ),  h3[m, n] = bf16( sum_d X[m,d] Wu[g][n,d] )
 *   h[m, n]  = bf16( bf16(silu(h1[m,n])) * h3[m,n] ),  silu(x) = x / (1 + e^-x) in fp32
 * (the rounding points of an elementwise bf16 SwiGLU), then h is quantized:
 *   h_q [M, H] + h_s: along H (the down GEMM's contraction), blocked row groups
 *       (sized by mxfp8_scale_bytes(M, H, G, MXFP8_SCALES_BLOCKED));
 *   hT_q [H, M] + hT_s: along the tokens (the down GEMM's wgrad operand), blocked
 *       column groups (sized by mxfp8_scale_bytes_colgroups(H, M, G)).  Optional:
 *       both NULL to skip; when given, M % 32 == 0 and every group size % 32 == 0
 *       (device-checked: MXFP8_ERR_OFFSETS, nothing written).
 *   These are the bytes mxfp8_quantize_2d(h, MXFP8_ROW | MXFP8_COL, BLOCKED, offs)
 *   writes for h.
 * Inputs: x_q [M, D] + x_s (blocked row groups, as for the forward GEMM);
 *   wg_q, wu_q [G, H, D] + wg_s, wu_s (blocked per expert, as
 *   mxfp8_quantize_3d_experts(MXFP8_ROW) writes them).  h1, h3: [M, H] bf16
 *   outputs (kept for the SwiGLU backward).
 * Shapes: H % 32 == 0, D % 32 == 0, 1 <= G <= MXFP8_MAX_GROUPS; every pointer
 * 16-byte aligned; all buffers caller-owned device memory; M may be 0.
 * Errors: MXFP8_ERR_NULL / _SHAPE / _ALIGN / _ARCH synchronously.
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_grouped_mm_swiglu_fwd(const void* x_q, const void* x_s, const void* wg_q, const void* wg_s,
                                           const void* wu_q, const void* wu_s, const int32_t* offs, int32_t G,
                                           int64_t M, int64_t H, int64_t D, void* h1_bf16, void* h3_bf16, void* h_q,
                                           void* h_s, void* hT_q, void* hT_s, int32_t* dev_status,
                                           mxfp8_stream_t stream);

/* ----------------------------------------------------------------------------
 * mxfp8_swiglu_bwd_quantize -- the SwiGLU backward of a routed expert with the
 * MXFP8 quantization of its two outputs fused in.  [P3] "Neutralizing
 * quantization overhead" (fuse quantization into the producing kernel); [P4]
 * (gate/up/down routed-expert weights).  For h = silu(h1) * h3 and its
 * gradient dh, elementwise at the rounding points of the bf16 autograd ops:
 *   dh3 = bf16(dh * bf16(silu(h1)))
 *   dh1 = bf16(bf16(dh * h3) * sig * (1 + h1 * (1 - sig))),  sig = 1 / (1 + e^-h1)
 * in fp32, then each of dh1, dh3 quantized as mxfp8_quantize_2d(MXFP8_ROW |
 * MXFP8_COL, MXFP8_SCALES_BLOCKED, offs) does: codes [M, H] + blocked row-group
 * scales (the gate/up dgrads) and codes [H, M] + blocked token-group scales
 * (their wgrads).
 * Inputs dh, h1, h3: [M, H] bf16.  M % 32 == 0, H % 32 == 0, every group size
 * % 32 == 0 (as for the column-wise quantization); scale buffers sized by
 * mxfp8_scale_bytes(M, H, G, MXFP8_SCALES_BLOCKED) and
 * mxfp8_scale_bytes_colgroups(H, M, G); all pointers caller-owned device memory,
 * 16-byte aligned.  Errors: MXFP8_ERR_NULL / _SHAPE / _ALIGN / _ARCH.
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_swiglu_bwd_quantize(const void* dh_bf16, const void* h1_bf16, const void* h3_bf16, int64_t M,
                                         int64_t H, const int32_t* offs, int32_t G, void* dh1_q, void* dh1_s,
                                         void* dh1T_q, void* dh1T_s, void* dh3_q, void* dh3_s, void* dh3T_q,
                                         void* dh3T_s, int32_t* dev_status, mxfp8_stream_t stream);

/* ----------------------------------------------------------------------------
 * Sizes and checks.
 * mxfp8_scale_bytes: bytes to allocate for the scales of an operand with `rows`
 *   rows of K elements (K % 32 == 0) quantized along K, its rows split into G
 *   groups (G <= 1: ungrouped).  Compact: rows*K/32.  Blocked: an upper bound
 *   that holds for any split, (ceil(rows/128) + G) * 128 * ceil(K/128) * 4.
 * mxfp8_scale_bytes_colgroups: blocked scales of a column-wise quantized
 *   operand qT[R, M] whose M tokens form G groups:
 *   ceil(R/128) * 128 * (ceil(M/128) + G) * 4 (an upper bound for any split).
 * mxfp8_check_offsets: enqueue a check of offs (monotone, offs[G-1] == M, every
 *   group size % align == 0); writes MXFP8_ERR_OFFSETS to *dev_status on failure.
 * ------------------------------------------------------------------------- */
size_t mxfp8_scale_bytes(int64_t rows, int64_t K, int32_t G, int scale_layout);
size_t mxfp8_scale_bytes_colgroups(int64_t R, int64_t M, int32_t G);
mxfp8_status_t mxfp8_check_offsets(const int32_t* offs, int32_t G, int64_t M, int32_t align, int32_t* dev_status,
                                   mxfp8_stream_t stream);
const char* mxfp8_status_string(mxfp8_status_t status);

/* ----------------------------------------------------------------------------
 * mxfp8_debug_wait_timeout -- self-test of the bounded waits every pipelined
 *   kernel uses: one thread waits on a barrier that nothing arrives on, gives
 *   up after limit_ns (1 ns .. 10 s) and writes MXFP8_ERR_TIMEOUT to
 *   *dev_status (device, required).  No counterpart on the pages; it exists so
 *   the timeout path can be exercised without a fault or a hang.
 * ------------------------------------------------------------------------- */
mxfp8_status_t mxfp8_debug_wait_timeout(int32_t* dev_status, uint64_t limit_ns, mxfp8_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MXFP8MOE_H */
