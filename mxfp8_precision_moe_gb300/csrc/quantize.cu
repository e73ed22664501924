// quantize.cu -- dynamic MXFP8 quantization kernels for sm_103a.
//
// One tile kernel serves every direction the routed-expert path needs
// ("MXFP8 training for MoEs", engine paragraph: activations and weights are
// quantized on the fly; "MXFP8 (Micro-scaling FP8)", "Low-precision Flash
// Attention": scales along each GEMM's K, transposed operands for the backward,
// [32, 32] square blocks; pytorch/ao PR 3004: 3D expert weights, plain and
// column-wise):
//   ROW       blocks of 32 along the row           -> q[R, C]
//   COL       blocks of 32 down a column, transposed -> qT[C, R]
//   ROW|COL   both from one read of x
//   BLK32     one scale per 32x32 tile             -> q[R, C]
// 3D expert weights run the same kernel with the expert as a batch index.
//
// Work decomposition: a CTA of 8 warps owns a 128 x 128 tile of x; each warp a
// 32-row x 64-column sub-tile; lane (i = lane/8, j = lane%8) holds rows 8i..8i+7
// and columns 8j..8j+7 of it in registers (8 x 16-byte loads; every warp load
// instruction reads four fully used 128-byte row segments).  Row blocks of 32
// span 4 lanes (2 shuffles), column blocks of 32 span the 4 lanes i = 0..3
// (2 shuffles); amax is max.NaN.xorsign.abs.bf16x2 on the raw bf16 pairs, two
// scale bytes come from the exponent fields with one packed max and subtract,
// each element is scaled by 2^(127-s) with one mixed-precision bf16 fma (exact)
// and pairs are converted with cvt.rn.satfinite.e4m3x2.  Code stores are 8-byte
// vectors; a row's scale bytes of a warp leave as one 16/32-bit store.  The grid
// is persistent (a multiple of the SM count), striding over tiles.

#include <type_traits>

#include "common.cuh"
#include "host_common.h"

namespace mx {

constexpr uint64_t kQTimeoutNs = 2000000000ull;  // bounded waits: 2 s

struct QParams {
    const uint16_t* x;   // [batch][R][C] bf16 bits
    int64_t R, C;        // per-batch matrix
    int32_t batch;
    uint8_t* q_row;      // [batch][R][C]
    uint8_t* s_row;      // row scales (compact [R][C/32] or blocked), per batch stride s_row_bstride
    int64_t s_row_bstride;
    uint8_t* q_col;      // [batch][C][R]
    uint8_t* s_col;      // col scales (compact [C][R/32] or blocked), per batch stride s_col_bstride
    int64_t s_col_bstride;
    int blocked;
    const int32_t* offs;  // row groups (2D only; nullptr = one group)
    int32_t G;
    int32_t* dev_status;
    int64_t tiles_r, tiles_c, ntiles;
    unsigned opts;       // MXFP8_OPT_* (the stability-variant kernels only)
    uint64_t seed;
    // the fused SwiGLU backward only: x = dh, x2 = h1, x3 = h3; dh1 goes to q_row .. s_col, dh3 to the
    // second output set
    const uint16_t* x2;
    const uint16_t* x3;
    uint8_t* q_row2;
    uint8_t* s_row2;
    uint8_t* q_col2;
    uint8_t* s_col2;
};

// Kernel modes: plain MX quantization; the Hadamard variants (fp32 values), without and with
// stochastic rounding; the fused SwiGLU backward (three inputs dh, h1, h3; two quantized outputs);
// stochastic rounding alone (the plain kernel's bf16 data path with stochastic codes).
enum QuantMode : int { kModePlain = 0, kModeExt = 1, kModeSwiBwd = 2, kModeSR = 3, kModeExtSR = 4 };

// Warp 0 builds, for G groups over R rows, the clamped monotone end rows and
// the padded start rows P[g] = sum_{h<g} ceil(size_h/128)*128 (also the scale
// column base of a column-grouped layout, in units of 32 rows: P[g]/32).
// Returns the padded total through *total.
__device__ void build_group_table(const int32_t* offs, int G, int64_t R, int32_t* ends_s, int32_t* pstart_s,
                                  int32_t* total) {
    const int lane = threadIdx.x & 31;
    const int per = (G + 31) / 32;
    const int g0 = lane * per, g1 = min(G, g0 + per);
    const int32_t Rc = (int32_t)R;
    // pass 1: running max of clamped offsets (makes them monotone)
    int32_t mx = 0;
    for (int g = g0; g < g1; ++g) mx = max(mx, min(max(offs[g], 0), Rc));
    int32_t incl = mx;
    for (int d = 1; d < 32; d <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl = max(incl, o);
    }
    int32_t run = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) run = 0;
    // pass 2: ends, padded sizes, exclusive scan of padded sizes
    int32_t prev = run, psum = 0;
    for (int g = g0; g < g1; ++g) {
        int32_t e = max(prev, min(max(offs[g], 0), Rc));
        ends_s[g] = e;
        psum += ((e - prev + 127) / 128) * 128;
        prev = e;
    }
    int32_t sincl = psum;
    for (int d = 1; d < 32; d <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, sincl, d);
        if (lane >= d) sincl += o;
    }
    int32_t sexcl = sincl - psum;
    prev = run;
    for (int g = g0; g < g1; ++g) {
        pstart_s[g] = sexcl;
        int32_t e = ends_s[g];
        sexcl += ((e - prev + 127) / 128) * 128;
        prev = e;
    }
    if (lane == 31) *total = sincl;
}

// Group of row r (ends_s monotone): first g with r < ends_s[g]; G if none.
__device__ __forceinline__ int find_group(const int32_t* ends_s, int G, int64_t r) {
    int lo = 0, hi = G;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (r < ends_s[mid]) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// ---- stability variants ("MXFP8 (Micro-scaling FP8)", "Numerical stability": random Hadamard
// transforms before quantization, stochastic rounding)

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// bf16 x bf16 -> bf16 for both halves (round to nearest even; exact for x times a power of two).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max(a, b) of non-negative fp32 values, NaN if either is NaN (ordered as the bit patterns are).
__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Stochastic rounding on fp32 patterns.  E4M3 steps by 2^-9 below 2^-6 and keeps 3 mantissa bits above
// it; fp32 steps by 2^-149 below 2^-126 and keeps 23 bits above it.  So the fp32 pattern of
// z = |y| 2^-120, rounded toward zero, holds in bits 20.. the E4M3 code of |y| truncated (subnormal
// or normal alike) and in bits 12-19 F = floor(256 (|y| - lo) / (hi - lo)).  Adding u << 12 carries
// into bit 20 exactly when F + u >= 256; clearing bits 0-19 leaves the chosen E4M3 magnitude times
// 2^-120 (with y's sign, which the add never reaches), and scaling back by 2^120 gives a value that
// the round-to-nearest conversion returns unchanged, or saturates to 448 at and above 448.
// One half of a bf16 pair times 2^-120 as an fp32, rounded toward zero.
template <int H>
__device__ __forceinline__ float bf16_times_2m120(uint32_t yy) {
    float d;
    if constexpr (H == 0)
        asm("{\n\t.reg .b16 a0, a1, c;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b16 c, 0x0380;\n\t"
            "fma.rz.f32.bf16 %0, a0, c, 0f80000000;\n\t}" : "=f"(d) : "r"(yy));
    else
        asm("{\n\t.reg .b16 a0, a1, c;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b16 c, 0x0380;\n\t"
            "fma.rz.f32.bf16 %0, a1, c, 0f80000000;\n\t}" : "=f"(d) : "r"(yy));
    return d;
}
__device__ __forceinline__ float f32_times_2m120(float y) {
    float d;
    asm("mul.rz.f32 %0, %1, 0f03800000;" : "=f"(d) : "f"(y));
    return d;
}
// z = y 2^-120 (toward zero) and byte b of the random word w -> the E4M3 value stochastic rounding
// picks, as an fp32.  (One asm block: the byte is moved to bits 12-19 and added in place, so that the
// two copies' uses of a byte stay separate expressions, not one value held from copy to copy.)
__device__ __forceinline__ float sr_pick_value(float z, uint32_t w, int b) {
    float d;
    asm("{\n\t.reg .b32 t;\n\tprmt.b32 t, %2, 0, %3;\n\tshl.b32 t, t, 4;\n\tadd.u32 t, t, %1;\n\t"
        "and.b32 t, t, 0xFFF00000;\n\tmul.rn.f32 %0, t, 0f7B800000;\n\t}"
        : "=f"(d) : "r"(__float_as_uint(z)), "r"(w), "r"(0x4404u | ((uint32_t)b << 4)));
    return d;
}
// The stochastic codes (bytes 0 and 1) of a scaled bf16 pair yy (exact: x times a power of two); the
// random byte of half h is byte b_h of word w_h.
__device__ __forceinline__ uint32_t sr_pair_bf16x2(uint32_t yy, uint32_t w0, int b0, uint32_t w1, int b1) {
    return cvt_e4m3x2(sr_pick_value(bf16_times_2m120<0>(yy), w0, b0), sr_pick_value(bf16_times_2m120<1>(yy), w1, b1));
}

// E8M0 scale byte from the magnitude bits of an fp32 amax (same rule as for bf16: max(E - 8, 0)).
__device__ __forceinline__ uint32_t e8m0_from_f32bits(uint32_t a) {
    const uint32_t E = a >> 23;
    if (E == 0xFFu) return 0xFFu;
    return E > 8u ? E - 8u : 0u;
}

constexpr float kRhtScale = 0x1.6a09e6p-3f;  // fp32(1 / sqrt(32))

// Scale bytes of two blocks at once from their packed bf16 magnitude amaxes (one per 16-bit half):
// s = max(E - 8, 0) per half, E the exponent field.  E = 255 (Inf/NaN) comes out as 247 here, a value
// no finite amax gives; adding kNonfiniteAdd and testing kNonfiniteBits finds it, and
// fix_nonfinite_pair() turns it into 0xFF.
__device__ __forceinline__ uint32_t e8m0_pair(uint32_t m) {
    return vmax_u16x2((m >> 7) & 0x00FF00FFu, 0x00080008u) - 0x00080008u;
}
// Bit 8 of a half is set iff that half of s + 9 reached 256, i.e. s == 247 (halves never carry).
constexpr uint32_t kNonfiniteAdd = 0x00090009u, kNonfiniteBits = 0x01000100u;
__device__ __forceinline__ uint32_t fix_nonfinite_pair(uint32_t s) {
    const uint32_t lo = s & 0xFFFFu, hi = s >> 16;
    return (lo == 247u ? 0xFFu : lo) | ((hi == 247u ? 0xFFu : hi) << 16);
}
__device__ __forceinline__ uint32_t pair_half(uint32_t s, int h) { return h ? s >> 16 : s & 0xFFFFu; }
// Both inverse scales of a pair (halves <= 247) as bf16 bit patterns: (254 - s) << 7 in each half.
__device__ __forceinline__ uint32_t inv_scale_pair_bf16(uint32_t s) { return (0x00FE00FEu - s) << 7; }

// max(|a|, |b|) per bf16 half (NaN wins); the sign bits of the result are garbage (xor of the
// inputs' signs) and are ignored by e8m0_pair.
__device__ __forceinline__ uint32_t amax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t shfl_xor_amax(uint32_t v, int m) {
    return amax_bf16x2(v, __shfl_xor_sync(0xffffffffu, v, m));
}

// The bf16 in half HW of w times the bf16 power of two in half HF of f2, as an exact fp32: one
// mixed-precision fma with a -0 addend (keeps the sign of a zero product).
template <int HW, int HF>
__device__ __forceinline__ float scale_bf16(uint32_t w, uint32_t f2) {
    float d;
    if constexpr (HW == 0 && HF == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, 0f80000000;\n\t}" : "=f"(d) : "r"(w), "r"(f2));
    else if constexpr (HW == 1 && HF == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b0, 0f80000000;\n\t}" : "=f"(d) : "r"(w), "r"(f2));
    else if constexpr (HW == 0 && HF == 1)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b1, 0f80000000;\n\t}" : "=f"(d) : "r"(w), "r"(f2));
    else
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b1, 0f80000000;\n\t}" : "=f"(d) : "r"(w), "r"(f2));
    return d;
}
// Eight bf16 (4 packed words) times the scale in half HF of f2 -> eight E4M3 codes.
template <int HF>
__device__ __forceinline__ uint2 quant8_bf16(const uint32_t (&w)[4], uint32_t f2) {
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = cvt_e4m3x2(scale_bf16<0, HF>(w[k], f2), scale_bf16<1, HF>(w[k], f2));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Sign bits of eight bf16 moved to bit 7 of each byte; used to give the codes
// of a non-finite block (all 0x7F after the NaN multiply) the element signs.
__device__ __forceinline__ uint2 signs8(const uint32_t (&w)[4]) {
    uint2 r;
    auto two = [](uint32_t v) -> uint32_t { return ((v >> 8) & 0x80u) | ((v >> 16) & 0x8000u); };
    r.x = two(w[0]) | (two(w[1]) << 16);
    r.y = two(w[2]) | (two(w[3]) << 16);
    return r;
}

constexpr int kQStages = 3;                    // SMEM ring depth (tiles in flight per CTA)
constexpr int kQTileBytes = 128 * 128 * 2;     // one 128 x 128 bf16 tile
constexpr int kQThreads = 288;                 // 8 consumer warps + 1 TMA producer warp
constexpr int kQSmem = kQStages * kQTileBytes + 128;
constexpr int kQConsumerThreads = 256;         // 8 consumer warps, no producer warp

// kModeExt / kModeExtSR: the Hadamard variants of ROW / COL / ROW|COL (runtime options p.opts, seed
// p.seed), without / with stochastic rounding; fp32 working values in the transformed copies.
// kModeSR: stochastic rounding alone, on the bf16 data path.
// kModeSwiBwd (ROW|COL only): 256 threads, no TMA ring: each warp loads its patches of dh, h1 and h3
// straight from global memory (three inputs a stage would leave room for too few warps to hide the
// arithmetic's latency), computes dh1 and dh3 and quantizes each both ways.
// The stochastic-rounding kernels have no producer warp: warp 0's lane 0 issues the ring's loads (the
// first kQStages tiles up front, then each stage again once all 8 warps are done with it), so that 2
// CTAs of 8 warps leave each thread 128 registers instead of 96 (their random words spilled at 96).
// The Hadamard kernel without stochastic rounding fits in 96 and keeps the producer warp: there a
// refill waits for the slowest warp's whole tile, which costs more than the registers give.
template <int kMode>
constexpr bool kFoldedProducer = kMode == kModeSR || kMode == kModeExtSR;
template <int kMode>
constexpr int kQThreadsOf = (kMode == kModeSwiBwd || kFoldedProducer<kMode>) ? kQConsumerThreads : kQThreads;

// kHad (the Hadamard kernels only): bit 0 = transform the row-wise copy, bit 1 = the column-wise copy,
// fixed per instance so that each holds only the paths its options take.
template <unsigned DIRS, int kMode = kModePlain, unsigned kHad = 0>
__global__ void __launch_bounds__(kQThreadsOf<kMode>, 2)
    quant_tile_kernel(const __grid_constant__ CUtensorMap xmap, QParams p) {
    constexpr bool kExt = kMode == kModeExt || kMode == kModeExtSR;
    constexpr bool kSwiBwd = kMode == kModeSwiBwd;
    constexpr int kStages = kQStages;
    constexpr uint32_t kStageBytes = kQTileBytes;
    constexpr bool kRow = (DIRS & MXFP8_ROW) != 0;
    constexpr bool kCol = (DIRS & MXFP8_COL) != 0;
    constexpr bool kB32 = (DIRS & MXFP8_BLOCK32X32) != 0;
    // 32x32 blocks alone: row-major codes + compact [R/32][C/32] scales.  32x32 blocks with ROW and/or
    // COL: the plain and/or transposed codes of the same 32x32 quantization, the block scale written
    // for every row (column) of the block in the row (column) layouts.
    constexpr bool kB32Only = DIRS == MXFP8_BLOCK32X32;
    constexpr bool kRowOut = kRow || kB32Only;
    extern __shared__ uint8_t qsmem_raw[];
    __shared__ int32_t ends_s[kMaxGroups];
    __shared__ int32_t pstart_s[kMaxGroups];
    __shared__ int32_t ptotal_s;
    __shared__ __align__(8) uint64_t full[kQStages];
    __shared__ __align__(8) uint64_t empty[kQStages];
    __shared__ int abort_s;
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 127) & ~uintptr_t(127));

    const bool grouped = p.offs != nullptr && p.G > 1;
    if (grouped && p.blocked && threadIdx.x < 32) build_group_table(p.offs, p.G, p.R, ends_s, pstart_s, &ptotal_s);
    constexpr bool kFolded = kFoldedProducer<kMode>;
    if (threadIdx.x == (kFolded ? 0 : 256)) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 8);
        }
        abort_s = 0;
        fence_barrier_init();
        prefetch_tmap(&xmap);
    }
    __syncthreads();
    volatile int* abort_flag = &abort_s;
    const int64_t R = p.R, C = p.C;
    const int64_t Cb = C / kBlk;
    const int64_t ct_row = (C + 127) / 128;                                  // row-scale column tiles
    const int64_t ct_col = grouped ? (int64_t)ptotal_s / 128 : (R + 127) / 128;  // col-scale column tiles
    // tile indices fit in 32 bits (checked on the host): 32-bit divisions, not 64-bit ones, per tile
    const uint32_t per_b = (uint32_t)(p.tiles_r * p.tiles_c), tiles_c = (uint32_t)p.tiles_c;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the folded producer (warp 0, lane 0): tile t of this CTA into stage `stage`
    uint32_t issued = 0, issued_phase = 0;  // stages with a load issued, and the phase it completes
    auto issue_tile = [&](int64_t t, int stage, uint32_t phase) {
        const uint32_t tt = (uint32_t)t, b = tt / per_b, rem = tt - b * per_b;
        const uint32_t tr = rem / tiles_c, tc = rem - tr * tiles_c;
        mbar_arrive_expect_tx(&full[stage], kStageBytes);
        tma_load_3d(tiles + stage * kStageBytes, &xmap, (int32_t)(tc * 128), (int32_t)(tr * 128), (int32_t)b,
                    &full[stage]);
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
    };
    if constexpr (kFolded) {
        if (warp == 0 && lane == 0)
            for (int s = 0; s < kStages; ++s) {
                const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
                if (t < p.ntiles) issue_tile(t, s, 0u);
            }
    }
    if (warp == 8) {
        // ------------------------------------------------ TMA producer: whole 128x128 tiles, OOB zero-filled
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_phase = 0;
            for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
                if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, kQTimeoutNs, abort_flag, p.dev_status)) {
                    for (int s = 0; s < kStages; ++s)
                        if (issued & (1u << s)) {
                            volatile int no_abort = 0;
                            mbar_wait_bounded(&full[s], (last_phase >> s) & 1u, kQTimeoutNs, &no_abort, nullptr);
                        }
                    break;
                }
                const uint32_t tt = (uint32_t)t, b = tt / per_b, rem = tt - b * per_b;
                const uint32_t tr = rem / tiles_c, tc = rem - tr * tiles_c;
                mbar_arrive_expect_tx(&full[stage], kStageBytes);
                tma_load_3d(tiles + stage * kStageBytes, &xmap, (int32_t)(tc * 128), (int32_t)(tr * 128), (int32_t)b,
                            &full[stage]);
                issued |= 1u << stage;
                last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        }
        return;
    }

    // ---- zero padding of the blocked layouts (bytes no tile writes).  Done before the tile loop, so it
    // overlaps the producer filling the ring, in small units spread over all CTAs:
    //   row layout:    (batch, group, 32-row chunk) of the group's padding rows, every column tile;
    //   column layout: (batch, group, 128-row slice) of the group's padding block-columns, and
    //                  (batch) the padding rows C .. ceil(C/128)*128, every column tile.
    auto zero_padding = [&](uint8_t* s_row, uint8_t* s_col) {
        const int G_eff = grouped ? p.G : 1;
        const int64_t rslices = (C + 127) / 128;
        const int64_t units_row = kRow ? (int64_t)p.batch * G_eff * 4 : 0;
        const int64_t units_colg = kCol ? (int64_t)p.batch * G_eff * rslices : 0;
        const int64_t units_colr = kCol ? (int64_t)p.batch : 0;
        const int tid = threadIdx.x;  // 256 consumer threads
        for (int64_t u = blockIdx.x; u < units_row + units_colg + units_colr; u += gridDim.x) {
            if (u < units_row) {
                const int64_t bb = u / (G_eff * 4);
                const int g = (int)((u / 4) % G_eff), chunk = (int)(u % 4);
                const int64_t start = grouped ? (g ? ends_s[g - 1] : 0) : 0;
                const int64_t size = grouped ? ends_s[g] - start : R;
                const int64_t P = grouped ? pstart_s[g] : 0;
                const int64_t r0 = size + chunk * 32, r1 = min64(r0 + 32, ((size + 127) / 128) * 128);
                uint8_t* sb = s_row + bb * p.s_row_bstride;
                for (int64_t i = tid; i < (r1 - r0) * ct_row; i += 256) {
                    const int64_t pr = P + r0 + i / ct_row, t = i % ct_row;
                    *reinterpret_cast<uint32_t*>(sb + ((pr >> 7) * ct_row + t) * 512 + (pr & 31) * 16 +
                                                 ((pr >> 5) & 3) * 4) = 0u;
                }
            } else if (u < units_row + units_colg) {
                const int64_t u2 = u - units_row;
                const int64_t bb = u2 / (G_eff * rslices);
                const int g = (int)((u2 / rslices) % G_eff);
                const int64_t rs = u2 % rslices;
                const int64_t start = grouped ? (g ? ends_s[g - 1] : 0) : 0;
                const int64_t size = grouped ? ends_s[g] - start : R;
                const int64_t Q = grouped ? pstart_s[g] / kBlk : 0;
                const int64_t c0 = Q + size / kBlk, c1 = Q + ((size + 127) / 128) * 4;
                const int64_t rlo = rs * 128, rn = min64(128, C - rlo);
                uint8_t* sb = s_col + bb * p.s_col_bstride;
                for (int64_t i = tid; i < rn * (c1 - c0); i += 256) {
                    const int64_t r = rlo + i / (c1 - c0), c = c0 + i % (c1 - c0);
                    sb[blocked_off(r, c, ct_col)] = 0;
                }
            } else {
                const int64_t bb = u - units_row - units_colg;
                const int64_t rows_p = ((C + 127) / 128) * 128;
                uint8_t* sb = s_col + bb * p.s_col_bstride;
                for (int64_t i = tid; i < (rows_p - C) * ct_col; i += 256) {
                    const int64_t r = C + i / ct_col, t = i % ct_col;
                    *reinterpret_cast<uint32_t*>(sb + ((r >> 7) * ct_col + t) * 512 + (r & 31) * 16 +
                                                 ((r >> 5) & 3) * 4) = 0u;
                }
            }
        }
    };
    if (p.blocked && (kRow || kCol)) {
        zero_padding(p.s_row, p.s_col);
        if constexpr (kSwiBwd) zero_padding(p.s_row2, p.s_col2);
    }

    const int wi = warp >> 1, wj = warp & 1;
    const int li = lane >> 3, lj = lane & 7;
    int stage = 0;
    uint32_t phase = 0;

    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const uint32_t tt = (uint32_t)t, b32 = tt / per_b, rem = tt - b32 * per_b;
        const uint32_t tr = rem / tiles_c, tc = rem - tr * tiles_c;
        const int64_t b = b32;
        const int64_t row0 = (int64_t)tr * 128 + wi * 32, col0 = (int64_t)tc * 128 + wj * 64;
        // this warp's 32 x 64 sub-tile: lane rows 8li..8li+7, columns 8lj..8lj+7 (16 bytes each)
        const uint8_t* src = nullptr;
        uint32_t v[8][4];
        int cur_stage = 0;
        uint32_t cur_phase = 0;
        if constexpr (!kSwiBwd) {
            if (!mbar_wait_bounded(&full[stage], phase, kQTimeoutNs, abort_flag, p.dev_status)) break;
            src = tiles + stage * kStageBytes + (32 * wi + 8 * li) * 256 + (64 * wj + 8 * lj) * 2;
            if constexpr (kMode == kModePlain || kMode == kModeSR) {
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const uint4 u = *reinterpret_cast<const uint4*>(src + rr * 256);
                    v[rr][0] = u.x; v[rr][1] = u.y; v[rr][2] = u.z; v[rr][3] = u.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                if constexpr (kFolded) {
                    // refill: once all 8 warps have read this stage, the tile kStages rounds ahead
                    const int64_t tn = t + (int64_t)kStages * gridDim.x;
                    if (warp == 0 && lane == 0 && tn < p.ntiles &&
                        mbar_wait_bounded(&empty[stage], phase, kQTimeoutNs, abort_flag, p.dev_status))
                        issue_tile(tn, stage, phase ^ 1u);
                }
            }
            cur_stage = stage;
            cur_phase = phase;
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        // the Hadamard variants read their values from the stage while they work and free it after
        // (and warp 0 then refills it, once all 8 warps are done with it)
        auto release_stage = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[cur_stage]);
            if constexpr (kFolded) {
                const int64_t tn = t + (int64_t)kStages * gridDim.x;
                if (warp == 0 && lane == 0 && tn < p.ntiles &&
                    mbar_wait_bounded(&empty[cur_stage], cur_phase, kQTimeoutNs, abort_flag, p.dev_status))
                    issue_tile(tn, cur_stage, cur_phase ^ 1u);
            }
        };
        if (row0 >= R || col0 >= C) {  // warp-uniform
            if constexpr (kExt) release_stage();
            continue;
        }

        const int64_t c8 = col0 + 8 * lj;  // first column of this lane
        const bool cval = c8 < C;          // C % 32 == 0: 8-column chunks are all-in or all-out
        int wg0 = 0, wg1 = 0;              // groups of the warp's first and last row (warp-uniform)
        if (grouped && p.blocked) {
            wg0 = find_group(ends_s, p.G, row0);
            const int64_t rl = min64(row0 + 31, R - 1);
            wg1 = (wg0 < p.G && rl < ends_s[wg0]) ? wg0 : find_group(ends_s, p.G, rl);
        }

        // Row-wise scales of the warp's 32 rows x 2 block-columns.  P0 / P1: this lane's scale bytes of
        // rows 0-3 / 4-7 of its 8-row patch (the same in the 4 lanes of a 32-column block).  Lane l
        // writes row row0 + l, both block-columns with one 16-bit store, or 32-bit with two zero bytes
        // when the rest of the layout's 4-byte word lies past C.  The whole warp calls it.
        auto store_row_scales = [&](uint8_t* s_row, uint32_t P0, uint32_t P1) {
            const int src = lane & ~7;  // lanes of rows 8i..8i+7: block 0 at 8i, block 1 at 8i + 4
            const uint32_t x0 = __shfl_sync(0xffffffffu, P0, src), x1 = __shfl_sync(0xffffffffu, P1, src);
            const uint32_t y0 = __shfl_sync(0xffffffffu, P0, src + 4), y1 = __shfl_sync(0xffffffffu, P1, src + 4);
            const int64_t cb = col0 / kBlk;
            const bool two = col0 + kBlk < C;
            const uint32_t b0 = __byte_perm(x0, x1, lane & 7) & 0xFFu;
            const uint32_t b1 = two ? __byte_perm(y0, y1, lane & 7) & 0xFFu : 0u;
            const int64_t row = row0 + lane;
            if (row >= R) return;
            uint8_t* sb = s_row + b * p.s_row_bstride;
            if (!p.blocked) {
                sb[row * Cb + cb] = (uint8_t)b0;
                if (two) sb[row * Cb + cb + 1] = (uint8_t)b1;
                return;
            }
            int64_t pr = row;
            if (grouped) {
                int g = wg0;
                if (wg0 != wg1) g = find_group(ends_s, p.G, row);
                if (g >= p.G) return;
                pr = pstart_s[g] + (row - (g ? ends_s[g - 1] : 0));
            }
            uint8_t* w = sb + ((pr >> 7) * ct_row + (cb >> 2)) * 512 + (pr & 31) * 16 + ((pr >> 5) & 3) * 4 + (cb & 3);
            if ((cb & 3) == 0 && col0 + 2 * kBlk >= C) *reinterpret_cast<uint32_t*>(w) = b0 | (b1 << 8);
            else *reinterpret_cast<uint16_t*>(w) = (uint16_t)(b0 | (b1 << 8));
        };
        // Column-wise scales of the warp's 64 columns (one 32-row block).  s2c[k]: scale bytes of this
        // lane's columns 2k (low half) and 2k+1 (high half); lane (li, lj) writes columns
        // 8lj + 2li and 8lj + 2li + 1, 16 bytes apart in the blocked layout.
        auto store_col_scales = [&](uint8_t* s_col, const uint32_t (&s2c)[4]) {
            if (!cval) return;
            const uint32_t my = li == 0 ? s2c[0] : li == 1 ? s2c[1] : li == 2 ? s2c[2] : s2c[3];
            uint8_t* sb = s_col + b * p.s_col_bstride;
            const int64_t rb = row0 / kBlk;
            const int64_t c = c8 + 2 * li;
            if (!p.blocked) {
                sb[c * (R / kBlk) + rb] = (uint8_t)my;
                sb[(c + 1) * (R / kBlk) + rb] = (uint8_t)(my >> 16);
                return;
            }
            int64_t pc = rb;
            if (grouped) {
                if (wg0 >= p.G) return;
                pc = pstart_s[wg0] / kBlk + (row0 - (wg0 ? ends_s[wg0 - 1] : 0)) / kBlk;
            }
            uint8_t* w = sb + ((c >> 7) * ct_col + (pc >> 2)) * 512 + (c & 31) * 16 + ((c >> 5) & 3) * 4 + (pc & 3);
            w[0] = (uint8_t)my;
            w[16] = (uint8_t)(my >> 16);
        };


        // Stochastic rounding: the random bytes of this lane's 8 x 8 patch, drawn once for both copies.
        // Element (r, c) takes byte 8 (r mod 2) + (c mod 8) (word k = bytes 4k .. 4k+3, least significant
        // first) of Philox4x32-10 with key = seed and counter (b mod 2^32, b / 2^32, 0, 0),
        // b = floor(r / 2) (C / 8) + floor(c / 8): draw d covers the patch's rows 2d, 2d + 1 (words x, y:
        // row 2d, columns 0-3 / 4-7; words z, w: row 2d + 1).
        uint4 rnd[4];
        if constexpr (kMode == kModeSR || kMode == kModeExtSR) {
            const uint64_t cq = (uint64_t)C >> 3;
            const uint64_t b0 = (uint64_t)((row0 + 8 * li) >> 1) * cq + (uint64_t)(c8 >> 3);
#pragma unroll
            for (int d = 0; d < 4; ++d) {
                const uint64_t bd = b0 + (uint64_t)d * cq;
                rnd[d] = philox4x32_10(make_uint4((uint32_t)bd, (uint32_t)(bd >> 32), 0u, 0u), (uint32_t)p.seed,
                                       (uint32_t)(p.seed >> 32));
            }
        }
        // the plain MX quantization of one 8 x 8 patch per lane (bf16 pairs v) into one output set
        // the row-wise half of it (sblk: the 32x32 block scale when 32x32 blocks are asked for)
        auto quant_rows = [&](const uint32_t (&v)[8][4], uint32_t sblk, uint8_t* q_row, uint8_t* s_row, bool srq) {
            if constexpr (kRowOut) {
                // s2[k]: scale bytes of rows 2k (low half) and 2k+1 (high half); 247 marks Inf/NaN
                uint32_t s2[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (kB32) {
                        s2[k] = min(sblk, 247u) * 0x00010001u;
                    } else {
                        // (amax of row 2k, amax of row 2k+1) over this lane's 8 columns, then its 4 lanes
                        const uint32_t a = amax_bf16x2(amax_bf16x2(v[2 * k][0], v[2 * k][1]), amax_bf16x2(v[2 * k][2], v[2 * k][3]));
                        const uint32_t c = amax_bf16x2(amax_bf16x2(v[2 * k + 1][0], v[2 * k + 1][1]),
                                                       amax_bf16x2(v[2 * k + 1][2], v[2 * k + 1][3]));
                        uint32_t m = amax_bf16x2(__byte_perm(a, c, 0x5410), __byte_perm(a, c, 0x7632));
                        m = shfl_xor_amax(m, 1);
                        m = shfl_xor_amax(m, 2);
                        s2[k] = e8m0_pair(m);
                    }
                }
                uint32_t nf = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) nf |= s2[k] + kNonfiniteAdd;
                const bool any_nonfinite = __any_sync(0xffffffffu, (nf & kNonfiniteBits) != 0u);
                uint8_t* qb = q_row + b * R * C;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t f2 = inv_scale_pair_bf16(s2[k]);
                    uint2 q[2];
                    if (kMode == kModeSR || (kMode == kModeExtSR && srq)) {
                        // rows 2k (scale in the low half of f2) and 2k + 1 (high half): draw k
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t fs = h ? (f2 & 0xFFFF0000u) | (f2 >> 16) : (f2 & 0xFFFFu) | (f2 << 16);
                            const uint32_t w0 = h ? rnd[k].z : rnd[k].x, w1 = h ? rnd[k].w : rnd[k].y;  // columns 0-3 / 4-7
                            uint32_t c[4];
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t w = kk < 2 ? w0 : w1;  // columns 2kk, 2kk + 1: bytes 2 (kk % 2), + 1
                                c[kk] = sr_pair_bf16x2(mul_bf16x2(v[2 * k + h][kk], fs), w, 2 * (kk & 1), w,
                                                       2 * (kk & 1) + 1);
                            }
                            q[h] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
                        }
                    } else {
                        q[0] = quant8_bf16<0>(v[2 * k], f2);
                        q[1] = quant8_bf16<1>(v[2 * k + 1], f2);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int rr = 2 * k + h;
                        const int64_t row = row0 + 8 * li + rr;
                        if (any_nonfinite && pair_half(s2[k], h) == 247u) {
                            const uint2 sg = signs8(v[rr]);
                            q[h].x = 0x7F7F7F7Fu | sg.x;
                            q[h].y = 0x7F7F7F7Fu | sg.y;
                        }
                        if (cval && row < R) *reinterpret_cast<uint2*>(qb + row * C + c8) = q[h];
                    }
                }
                if (any_nonfinite) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) s2[k] = fix_nonfinite_pair(s2[k]);
                }
                if constexpr (kB32Only) {
                    // one compact scale per 32x32 block
                    if (cval && li == 0 && (lj & 3) == 0) s_row[b * p.s_row_bstride + (row0 / kBlk) * Cb + c8 / kBlk] = (uint8_t)sblk;
                } else {
                    store_row_scales(s_row, __byte_perm(s2[0], s2[1], 0x6420), __byte_perm(s2[2], s2[3], 0x6420));
                }
            }
        };
        // the column-wise half of it
        auto quant_cols = [&](const uint32_t (&v)[8][4], uint32_t sblk, uint8_t* q_col, uint8_t* s_col, bool srq) {
            if constexpr (kCol) {
                // s2c[k]: scale bytes of this lane's columns 2k (low half) and 2k+1 (high half)
                uint32_t s2c[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (kB32) {
                        s2c[k] = min(sblk, 247u) * 0x00010001u;
                    } else {
                        // column amax over 32 rows: 8 here (packed pairs of columns), then lanes li = 0..3
                        uint32_t m = amax_bf16x2(amax_bf16x2(amax_bf16x2(v[0][k], v[1][k]), amax_bf16x2(v[2][k], v[3][k])),
                                                 amax_bf16x2(amax_bf16x2(v[4][k], v[5][k]), amax_bf16x2(v[6][k], v[7][k])));
                        m = shfl_xor_amax(m, 8);
                        m = shfl_xor_amax(m, 16);
                        s2c[k] = e8m0_pair(m);
                    }
                }
                uint32_t nf = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) nf |= s2c[k] + kNonfiniteAdd;
                const bool any_nonfinite = __any_sync(0xffffffffu, (nf & kNonfiniteBits) != 0u);
                uint8_t* qb = q_col + b * R * C;
                // codes of column 2k + h: elements (rr, half h of word k) times half h of the scale pair
                auto col_codes = [&](auto hc, int k, uint32_t f2) -> uint2 {
                    constexpr int h = decltype(hc)::value;
                    uint32_t w[4];
                    if (kMode == kModeSR || (kMode == kModeExtSR && srq)) {
                        // column j = 2k + h; rows rr, rr + 1 share draw rr / 2 (words j / 4 and 2 + j / 4,
                        // byte j % 4 of each)
                        const uint32_t fs = h ? (f2 & 0xFFFF0000u) | (f2 >> 16) : (f2 & 0xFFFFu) | (f2 << 16);
                        constexpr uint32_t kPickH = h ? 0x7632u : 0x5410u;  // half h of two words -> one pair
                        const int j = 2 * k + h, wsel = j >> 2, b = j & 3;
#pragma unroll
                        for (int rr = 0; rr < 8; rr += 2) {
                            const uint4 r4 = rnd[rr >> 1];
                            const uint32_t wa = wsel ? r4.y : r4.x, wb = wsel ? r4.w : r4.z;
                            uint32_t xx;
                            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(xx) : "r"(v[rr][k]), "r"(v[rr + 1][k]), "r"(kPickH));
                            w[rr >> 1] = sr_pair_bf16x2(mul_bf16x2(xx, fs), wa, b, wb, b);
                        }
                    } else {
#pragma unroll
                        for (int rr = 0; rr < 8; rr += 2)
                            w[rr >> 1] = cvt_e4m3x2(scale_bf16<h, h>(v[rr][k], f2), scale_bf16<h, h>(v[rr + 1][k], f2));
                    }
                    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
                };
                if (cval) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t f2 = inv_scale_pair_bf16(s2c[k]);
                        uint2 q[2] = {col_codes(std::integral_constant<int, 0>{}, k, f2),
                                      col_codes(std::integral_constant<int, 1>{}, k, f2)};
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (any_nonfinite && pair_half(s2c[k], h) == 247u) {
                                uint32_t sg[4];
#pragma unroll
                                for (int rr = 0; rr < 8; rr += 2) {
                                    const uint32_t a = h ? (v[rr][k] >> 31) : ((v[rr][k] >> 15) & 1u);
                                    const uint32_t c = h ? (v[rr + 1][k] >> 31) : ((v[rr + 1][k] >> 15) & 1u);
                                    sg[rr >> 1] = (a << 7) | (c << 15);
                                }
                                q[h].x = 0x7F7F7F7Fu | sg[0] | (sg[1] << 16);
                                q[h].y = 0x7F7F7F7Fu | sg[2] | (sg[3] << 16);
                            }
                            if (cval) *reinterpret_cast<uint2*>(qb + (c8 + 2 * k + h) * R + row0 + 8 * li) = q[h];
                        }
                    }
                }
                if (any_nonfinite) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) s2c[k] = fix_nonfinite_pair(s2c[k]);
                }
                store_col_scales(s_col, s2c);
            }
        };
        auto quant_rowcol = [&](const uint32_t (&v)[8][4], uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                uint8_t* s_col) {
            // amaxes are taken on the raw bf16 pairs (max of magnitudes; the sign bits they carry are
            // ignored when the scale byte is read off the exponent field)
            uint32_t sblk = 0;  // the 32x32 block's scale
            if constexpr (kB32) {
                // one amax over the 32x32 block: 8 rows here, 4 lanes across (lj bits 0-1), 4 down (li)
                uint32_t m = 0;
#pragma unroll
                for (int rr = 0; rr < 8; ++rr)
#pragma unroll
                    for (int k = 0; k < 4; ++k) m = amax_bf16x2(m, v[rr][k]);
                m = shfl_xor_amax(m, 1);
                m = shfl_xor_amax(m, 2);
                m = shfl_xor_amax(m, 8);
                m = shfl_xor_amax(m, 16);
                sblk = e8m0_from_absbits(max(m & 0x7FFFu, (m >> 16) & 0x7FFFu));
            }

            quant_rows(v, sblk, q_row, s_row, kMode == kModeSR);
            quant_cols(v, sblk, q_col, s_col, kMode == kModeSR);
        };

        if constexpr (kExt) {
            // Stability variants: optionally a Hadamard transform of every block of 32 along the copy's
            // axis, y = c * H * (D x) (signs D, butterflies h = 1, 2, 4 inside the lane, h = 8, 16 across
            // lanes, in that order, in fp32); codes by round-to-nearest-even or by stochastic rounding
            // with one random byte per element.  A copy with neither option takes the plain bf16 path.
            // The fp32 copies take the block's amax before the factor c (the scale byte is read off
            // fp32(amax * c), which equals the amax of the values fp32(c h): rounding is monotonic) and
            // multiply each value once by c * 2^(127 - s), which gives fp32(c h) times that power of two
            // exactly wherever the result is an fp32 normal; below that every code is a signed zero
            // either way.  Signs are applied to the bf16 patterns; the cross-lane butterflies are one fma
            // with -1 or 1 (exact in the product, one rounding as the sum or difference).  Rows (row
            // copy) and columns (column copy) are processed 4 at a time to keep the fp32 values in
            // registers.
            constexpr bool sr = kMode == kModeExtSR;
            constexpr bool had_r = (kHad & 1u) != 0, had_c = (kHad & 2u) != 0;
            const uint32_t dsign = philox4x32_10(make_uint4(0u, 0u, 2u, 0u), (uint32_t)p.seed,
                                                 (uint32_t)(p.seed >> 32)).x;
            // two codes from two scaled fp32 values and (stochastic rounding) their random bytes: byte b0
            // of word w0, byte b1 of word w1
            auto code2 = [&](float z0, float z1, uint32_t w0, int b0, uint32_t w1, int b1) -> uint32_t {
                return sr ? cvt_e4m3x2(sr_pick_value(f32_times_2m120(z0), w0, b0), sr_pick_value(f32_times_2m120(z1), w1, b1))
                          : cvt_e4m3x2(z0, z1);
            };
            // the lane's 8 x 8 bf16 patch from the stage, for the plain path
            auto load_patch = [&](uint32_t (&v)[8][4]) {
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const uint4 u = *reinterpret_cast<const uint4*>(src + rr * 256);
                    v[rr][0] = u.x; v[rr][1] = u.y; v[rr][2] = u.z; v[rr][3] = u.w;
                }
            };
            if constexpr (kRow) {
                if constexpr (!had_r) {
                    uint32_t v[8][4];
                    load_patch(v);
                    quant_rows(v, 0u, p.q_row, p.s_row, sr);
                } else {
                    uint32_t s8[8];
                    uint8_t* qb = p.q_row + b * R * C;
                    const float cc = had_r ? kRhtScale : 1.0f;
                    // sign masks of the row transform: columns 2k (bit 15) and 2k + 1 (bit 31) of the lane,
                    // at block positions 8 (lj mod 4) + 2k, + 1
                    uint32_t sm[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t d2 = had_r ? dsign >> (8 * (lj & 3) + 2 * k) : 0u;
                        sm[k] = ((d2 & 1u) << 15) | ((d2 & 2u) << 30);
                    }
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        float y[4][8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 u = *reinterpret_cast<const uint4*>(src + (4 * hr + i) * 256);
                            const uint32_t w[4] = {u.x ^ sm[0], u.y ^ sm[1], u.z ^ sm[2], u.w ^ sm[3]};
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                y[i][2 * k] = bf16lo(w[k]);
                                y[i][2 * k + 1] = bf16hi(w[k]);
                            }
                        }
                        if constexpr (had_r) {
#pragma unroll
                            for (int h = 1; h < 8; h <<= 1)
#pragma unroll
                                for (int i = 0; i < 4; ++i)
#pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        if ((c & h) == 0) {
                                            const float a = y[i][c], bb = y[i][c + h];
                                            y[i][c] = a + bb;
                                            y[i][c + h] = a - bb;
                                        }
#pragma unroll
                            for (int m = 1; m <= 2; m <<= 1) {
                                const float sg = (lane & m) ? -1.0f : 1.0f;  // upper lane: partner - own
#pragma unroll
                                for (int i = 0; i < 4; ++i)
#pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        y[i][c] = __fmaf_rn(y[i][c], sg, __shfl_xor_sync(0xffffffffu, y[i][c], m));
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float m = 0.0f;
#pragma unroll
                            for (int c = 0; c < 8; ++c) m = max_nan_f32(m, fabsf(y[i][c]));
                            m = max_nan_f32(m, __shfl_xor_sync(0xffffffffu, m, 1));
                            m = max_nan_f32(m, __shfl_xor_sync(0xffffffffu, m, 2));
                            s8[4 * hr + i] = e8m0_from_f32bits(__float_as_uint(__fmul_rn(m, cc)));
                        }
                        // rows 4hr .. 4hr+3 of the patch: draws 2hr and 2hr + 1 (rows 2d: words x, y; rows 2d+1: z, w)
                        const uint4 dr[2] = {rnd[2 * hr], rnd[2 * hr + 1]};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t sc = s8[4 * hr + i];
                            const int64_t row = row0 + 8 * li + 4 * hr + i;
                            const float f = __fmul_rn(cc, inv_scale_from_e8m0(sc));
                            const uint32_t wa = (i & 1) ? dr[i >> 1].z : dr[i >> 1].x;  // columns 0-3
                            const uint32_t wb = (i & 1) ? dr[i >> 1].w : dr[i >> 1].y;  // columns 4-7
                            uint2 q;
                            q.x = code2(y[i][0] * f, y[i][1] * f, wa, 0, wa, 1) | (code2(y[i][2] * f, y[i][3] * f, wa, 2, wa, 3) << 16);
                            q.y = code2(y[i][4] * f, y[i][5] * f, wb, 0, wb, 1) | (code2(y[i][6] * f, y[i][7] * f, wb, 2, wb, 3) << 16);
                            if (sc == 0xFFu) {
                                uint32_t sg[2] = {0u, 0u};
#pragma unroll
                                for (int c = 0; c < 8; ++c) sg[c >> 2] |= ((__float_as_uint(y[i][c]) >> 24) & 0x80u) << (8 * (c & 3));
                                q.x = 0x7F7F7F7Fu | sg[0];
                                q.y = 0x7F7F7F7Fu | sg[1];
                            }
                            if (cval && row < R) *reinterpret_cast<uint2*>(qb + row * C + c8) = q;
                        }
                    }
                    store_row_scales(p.s_row, s8[0] | (s8[1] << 8) | (s8[2] << 16) | (s8[3] << 24),
                                     s8[4] | (s8[5] << 8) | (s8[6] << 16) | (s8[7] << 24));
                }
            }
            if constexpr (kCol) {
                if constexpr (!had_c) {
                    uint32_t v[8][4];
                    load_patch(v);
                    quant_cols(v, 0u, p.q_col, p.s_col, sr);
                } else {
                    uint32_t sc[8];
                    uint8_t* qb = p.q_col + b * R * C;
                    const float cc = had_c ? kRhtScale : 1.0f;
                    const uint32_t dl = had_c ? dsign >> (8 * li) : 0u;  // signs of the lane's rows: block positions 8 li + rr
#pragma unroll
                    for (int hc = 0; hc < 2; ++hc) {
                        float y[8][4];  // columns 4hc .. 4hc+3 of the lane
#pragma unroll
                        for (int rr = 0; rr < 8; ++rr) {
                            uint2 u = *reinterpret_cast<const uint2*>(src + rr * 256 + 8 * hc);
                            const uint32_t m = ((dl >> rr) & 1u) * 0x80008000u;
                            u.x ^= m;
                            u.y ^= m;
                            y[rr][0] = bf16lo(u.x);
                            y[rr][1] = bf16hi(u.x);
                            y[rr][2] = bf16lo(u.y);
                            y[rr][3] = bf16hi(u.y);
                        }
                        if constexpr (had_c) {
#pragma unroll
                            for (int h = 1; h < 8; h <<= 1)
#pragma unroll
                                for (int rr = 0; rr < 8; ++rr)
                                    if ((rr & h) == 0)
#pragma unroll
                                        for (int j = 0; j < 4; ++j) {
                                            const float a = y[rr][j], bb = y[rr + h][j];
                                            y[rr][j] = a + bb;
                                            y[rr + h][j] = a - bb;
                                        }
#pragma unroll
                            for (int m = 8; m <= 16; m <<= 1) {
                                const float sg = (lane & m) ? -1.0f : 1.0f;  // upper lane: partner - own
#pragma unroll
                                for (int rr = 0; rr < 8; ++rr)
#pragma unroll
                                    for (int j = 0; j < 4; ++j)
                                        y[rr][j] = __fmaf_rn(y[rr][j], sg, __shfl_xor_sync(0xffffffffu, y[rr][j], m));
                            }
                        }
                        float f[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float m = 0.0f;
#pragma unroll
                            for (int rr = 0; rr < 8; ++rr) m = max_nan_f32(m, fabsf(y[rr][j]));
                            m = max_nan_f32(m, __shfl_xor_sync(0xffffffffu, m, 8));
                            m = max_nan_f32(m, __shfl_xor_sync(0xffffffffu, m, 16));
                            sc[4 * hc + j] = e8m0_from_f32bits(__float_as_uint(__fmul_rn(m, cc)));
                            f[j] = __fmul_rn(cc, inv_scale_from_e8m0(sc[4 * hc + j]));
                        }
                        // codes of the 4 columns, two rows at a time (the words of a row cover its 4 columns)
                        uint32_t qc[4][2] = {{0u, 0u}, {0u, 0u}, {0u, 0u}, {0u, 0u}};
#pragma unroll
                        for (int rr = 0; rr < 8; rr += 2) {
                            // rows rr, rr + 1 of the patch: draw rr / 2, words hc (row rr) and 2 + hc (row rr + 1),
                            // byte j for column 4hc + j
                            const uint4 r4 = rnd[rr >> 1];
                            const uint32_t wa = hc ? r4.y : r4.x, wb = hc ? r4.w : r4.z;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                qc[j][rr >> 2] |= code2(y[rr][j] * f[j], y[rr + 1][j] * f[j], wa, j, wb, j) << (8 * (rr & 3));
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint2 q = make_uint2(qc[j][0], qc[j][1]);
                            if (sc[4 * hc + j] == 0xFFu) {
                                uint32_t sg[2] = {0u, 0u};
#pragma unroll
                                for (int rr = 0; rr < 8; ++rr)
                                    sg[rr >> 2] |= ((__float_as_uint(y[rr][j]) >> 24) & 0x80u) << (8 * (rr & 3));
                                q.x = 0x7F7F7F7Fu | sg[0];
                                q.y = 0x7F7F7F7Fu | sg[1];
                            }
                            if (cval) *reinterpret_cast<uint2*>(qb + (c8 + 4 * hc + j) * R + row0 + 8 * li) = q;
                        }
                    }
                    const uint32_t s2c[4] = {sc[0] | (sc[1] << 16), sc[2] | (sc[3] << 16), sc[4] | (sc[5] << 16),
                                             sc[6] | (sc[7] << 16)};
                    store_col_scales(p.s_col, s2c);
                }
            }
            release_stage();
            continue;
        }

        if constexpr (kSwiBwd) {
            // fused SwiGLU backward: dh1 and dh3 of h = silu(h1) * h3 at the rounding points of the
            // bf16 autograd ops (silu(h1), dh*h3, their products each rounded to bf16), fp32 inside.
            // Rows past the matrix read as zeros (what the TMA path's fill gives).
            uint32_t a[8][4], u3[8][4];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int64_t row = row0 + 8 * li + rr;
                uint4 g = make_uint4(0, 0, 0, 0), x1 = g, x3 = g;
                if (row < R && cval) {
                    const int64_t off = row * C + c8;
                    g = __ldg(reinterpret_cast<const uint4*>(p.x + off));
                    x1 = __ldg(reinterpret_cast<const uint4*>(p.x2 + off));
                    x3 = __ldg(reinterpret_cast<const uint4*>(p.x3 + off));
                }
                v[rr][0] = g.x; v[rr][1] = g.y; v[rr][2] = g.z; v[rr][3] = g.w;
                a[rr][0] = x1.x; a[rr][1] = x1.y; a[rr][2] = x1.z; a[rr][3] = x1.w;
                u3[rr][0] = x3.x; u3[rr][1] = x3.y; u3[rr][2] = x3.z; u3[rr][3] = x3.w;
            }
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t d1, d3;
                    swiglu_bwd_pair(v[rr][k], a[rr][k], u3[rr][k], d1, d3);
                    a[rr][k] = d1;
                    u3[rr][k] = d3;
                }
            quant_rowcol(a, p.q_row, p.s_row, p.q_col, p.s_col);
            quant_rowcol(u3, p.q_row2, p.s_row2, p.q_col2, p.s_col2);
        } else {
            quant_rowcol(v, p.q_row, p.s_row, p.q_col, p.s_col);
        }
    }
    if constexpr (kFolded) {
        // Warp 0 waited for every tile it issued unless a wait ran out: then let every load this CTA
        // issued land before its shared memory is released (bounded waits, no abort check).
        if (warp == 0 && lane == 0 && *abort_flag) {
            for (int s = 0; s < kStages; ++s)
                if (issued & (1u << s)) {
                    volatile int no_abort = 0;
                    mbar_wait_bounded(&full[s], (issued_phase >> s) & 1u, kQTimeoutNs, &no_abort, nullptr);
                }
        }
    }
}

__global__ void check_offsets_kernel(const int32_t* offs, int32_t G, int64_t M, int32_t align, int32_t* dev_status) {
    bool bad = false;
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int64_t prev = g ? offs[g - 1] : 0;
        const int64_t cur = offs[g];
        if (cur < prev || cur > M || prev < 0) bad = true;
        if (align > 1 && ((cur - prev) % align) != 0) bad = true;
        if (g == G - 1 && cur != M) bad = true;
    }
    if (bad) report(dev_status, MXFP8_ERR_OFFSETS);
}

// ---------------------------------------------------------------- host side
// base (x or another input of x's shape) viewed as [batch][R][C] bf16 with 128 x 128 boxes, no
// swizzle, zero fill outside.
static bool make_x_map(CUtensorMap* m, const QParams& p, const uint16_t* base) {
    host::EncodeTiledFn fn = host::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)p.C, (cuuint64_t)p.R, (cuuint64_t)p.batch};
    cuuint64_t strides[2] = {(cuuint64_t)(p.C * 2), (cuuint64_t)(p.R * p.C * 2)};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <unsigned DIRS, int kMode = kModePlain, unsigned kHad = 0>
static mxfp8_status_t launch_dirs(const CUtensorMap& m, const QParams& p, int64_t grid, cudaStream_t st) {
    constexpr bool direct = kMode == kModeSwiBwd;  // no TMA ring: no dynamic shared memory, no producer warp
    constexpr int smem = direct ? 0 : kQSmem;
    static std::atomic<int> attr_set[host::kMaxDevices];
    if (!host::ensure_smem(reinterpret_cast<const void*>(quant_tile_kernel<DIRS, kMode, kHad>), smem, attr_set))
        return MXFP8_ERR_LAUNCH;
    quant_tile_kernel<DIRS, kMode, kHad><<<(unsigned)grid, kQThreadsOf<kMode>, smem, st>>>(m, p);
    return host::last_launch_status();
}

static mxfp8_status_t launch_tiles(unsigned dirs, const QParams& p, cudaStream_t st) {
    if (p.ntiles == 0) return MXFP8_OK;
    CUtensorMap m;
    if (!make_x_map(&m, p, p.x)) return MXFP8_ERR_DRIVER;
    const int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)host::num_sms() * 2);
    switch (dirs) {
        case MXFP8_ROW: return launch_dirs<MXFP8_ROW>(m, p, grid, st);
        case MXFP8_COL: return launch_dirs<MXFP8_COL>(m, p, grid, st);
        case MXFP8_ROW | MXFP8_COL: return launch_dirs<MXFP8_ROW | MXFP8_COL>(m, p, grid, st);
        case MXFP8_BLOCK32X32: return launch_dirs<MXFP8_BLOCK32X32>(m, p, grid, st);
        case MXFP8_BLOCK32X32 | MXFP8_ROW: return launch_dirs<MXFP8_BLOCK32X32 | MXFP8_ROW>(m, p, grid, st);
        case MXFP8_BLOCK32X32 | MXFP8_COL: return launch_dirs<MXFP8_BLOCK32X32 | MXFP8_COL>(m, p, grid, st);
        case MXFP8_BLOCK32X32 | MXFP8_ROW | MXFP8_COL:
            return launch_dirs<MXFP8_BLOCK32X32 | MXFP8_ROW | MXFP8_COL>(m, p, grid, st);
        default: return MXFP8_ERR_LAYOUT;
    }
}

// The stability variants: stochastic rounding alone on the plain kernel's bf16 path; any Hadamard
// option on the fp32 kernel, built apart with and without stochastic rounding.
// The Hadamard kernels, one instance per direction set and transform set (kHad: bit 0 = the row-wise
// copy, bit 1 = the column-wise copy; the host checks that each transformed copy is asked for).
template <int kMode>
static mxfp8_status_t launch_had(unsigned dirs, unsigned had, const CUtensorMap& m, const QParams& p, int64_t grid,
                                 cudaStream_t st) {
    constexpr unsigned RC = MXFP8_ROW | MXFP8_COL;
    switch (dirs | (had << 4)) {
        case MXFP8_ROW | (1u << 4): return launch_dirs<MXFP8_ROW, kMode, 1>(m, p, grid, st);
        case MXFP8_COL | (2u << 4): return launch_dirs<MXFP8_COL, kMode, 2>(m, p, grid, st);
        case RC | (1u << 4): return launch_dirs<RC, kMode, 1>(m, p, grid, st);
        case RC | (2u << 4): return launch_dirs<RC, kMode, 2>(m, p, grid, st);
        case RC | (3u << 4): return launch_dirs<RC, kMode, 3>(m, p, grid, st);
        default: return MXFP8_ERR_LAYOUT;
    }
}

static mxfp8_status_t launch_tiles_ext(unsigned dirs, const QParams& p, cudaStream_t st) {
    if (p.ntiles == 0) return MXFP8_OK;
    CUtensorMap m;
    if (!make_x_map(&m, p, p.x)) return MXFP8_ERR_DRIVER;
    const int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)host::num_sms() * 2);
    if (p.opts == MXFP8_OPT_STOCHASTIC) {
        switch (dirs) {
            case MXFP8_ROW: return launch_dirs<MXFP8_ROW, kModeSR>(m, p, grid, st);
            case MXFP8_COL: return launch_dirs<MXFP8_COL, kModeSR>(m, p, grid, st);
            case MXFP8_ROW | MXFP8_COL: return launch_dirs<MXFP8_ROW | MXFP8_COL, kModeSR>(m, p, grid, st);
            default: return MXFP8_ERR_LAYOUT;
        }
    }
    const unsigned had = ((p.opts & MXFP8_OPT_HADAMARD_ROW) ? 1u : 0u) | ((p.opts & MXFP8_OPT_HADAMARD_COL) ? 2u : 0u);
    return (p.opts & MXFP8_OPT_STOCHASTIC) ? launch_had<kModeExtSR>(dirs, had, m, p, grid, st)
                                           : launch_had<kModeExt>(dirs, had, m, p, grid, st);
}

// The fused SwiGLU backward: p.x = dh, p.x2 = h1, p.x3 = h3 (direct loads; the tensor map is unused).
static mxfp8_status_t launch_swiglu_bwd(const QParams& p, cudaStream_t st) {
    if (p.ntiles == 0) return MXFP8_OK;
    CUtensorMap m;
    if (!make_x_map(&m, p, p.x)) return MXFP8_ERR_DRIVER;
    const int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)host::num_sms() * 2);
    return launch_dirs<MXFP8_ROW | MXFP8_COL, kModeSwiBwd>(m, p, grid, st);
}

static mxfp8_status_t quantize_2d(const void* x_bf16, int64_t M, int64_t K, unsigned dirs, int scale_layout,
                                  const int32_t* offs, int32_t G, unsigned opts, uint64_t seed, void* q_row,
                                  void* s_row, void* q_col, void* s_col, int32_t* dev_status, cudaStream_t st) {
    if (M < 0 || K <= 0 || G < 0 || G > MXFP8_MAX_GROUPS || M > INT32_MAX) return MXFP8_ERR_SHAPE;
    if (K % 32) return MXFP8_ERR_ALIGN;
    if (scale_layout != MXFP8_SCALES_COMPACT && scale_layout != MXFP8_SCALES_BLOCKED) return MXFP8_ERR_LAYOUT;
    const bool row = dirs & MXFP8_ROW, col = dirs & MXFP8_COL, b32 = dirs & MXFP8_BLOCK32X32;
    if (dirs == 0 || (dirs & ~7u) || (b32 && (row || col))) return MXFP8_ERR_LAYOUT;
    if (b32 && scale_layout != MXFP8_SCALES_COMPACT) return MXFP8_ERR_LAYOUT;
    if ((opts & ~7u) || (opts && b32) || ((opts & MXFP8_OPT_HADAMARD_ROW) && !row) ||
        ((opts & MXFP8_OPT_HADAMARD_COL) && !col))
        return MXFP8_ERR_LAYOUT;
    if (!x_bf16) return MXFP8_ERR_NULL;
    if ((row || b32) && (!q_row || !s_row)) return MXFP8_ERR_NULL;
    if (col && (!q_col || !s_col)) return MXFP8_ERR_NULL;
    if ((col || b32) && (M % 32)) return MXFP8_ERR_ALIGN;
    if (!host::aligned16(x_bf16) || !host::aligned16(q_row) || !host::aligned16(q_col) || !host::aligned16(s_row) ||
        !host::aligned16(s_col))
        return MXFP8_ERR_ALIGN;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    if (M == 0) return MXFP8_OK;
    const bool blocked = scale_layout == MXFP8_SCALES_BLOCKED;
    QParams p{};
    p.x = static_cast<const uint16_t*>(x_bf16);
    p.R = M; p.C = K; p.batch = 1;
    p.q_row = static_cast<uint8_t*>(q_row); p.s_row = static_cast<uint8_t*>(s_row);
    p.q_col = static_cast<uint8_t*>(q_col); p.s_col = static_cast<uint8_t*>(s_col);
    p.blocked = blocked ? 1 : 0;
    p.offs = offs; p.G = offs ? G : 0;
    p.dev_status = dev_status;
    p.tiles_r = (M + 127) / 128; p.tiles_c = (K + 127) / 128; p.ntiles = p.tiles_r * p.tiles_c;
    p.opts = opts;
    p.seed = seed;
    if (p.ntiles >= INT32_MAX) return MXFP8_ERR_SHAPE;
    return opts ? launch_tiles_ext(dirs, p, st) : launch_tiles(dirs, p, st);
}

}  // namespace mx

using namespace mx;

extern "C" mxfp8_status_t mxfp8_quantize_2d(const void* x_bf16, int64_t M, int64_t K, unsigned dirs,
                                            int scale_layout, const int32_t* offs, int32_t G, void* q_row,
                                            void* s_row, void* q_col, void* s_col, int32_t* dev_status,
                                            mxfp8_stream_t stream) {
    return mx::quantize_2d(x_bf16, M, K, dirs, scale_layout, offs, G, 0u, 0u, q_row, s_row, q_col, s_col, dev_status,
                           reinterpret_cast<cudaStream_t>(stream));
}

extern "C" mxfp8_status_t mxfp8_quantize_2d_opts(const void* x_bf16, int64_t M, int64_t K, unsigned dirs,
                                                 int scale_layout, const int32_t* offs, int32_t G, unsigned opts,
                                                 uint64_t seed, void* q_row, void* s_row, void* q_col, void* s_col,
                                                 int32_t* dev_status, mxfp8_stream_t stream) {
    return mx::quantize_2d(x_bf16, M, K, dirs, scale_layout, offs, G, opts, seed, q_row, s_row, q_col, s_col,
                           dev_status, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" mxfp8_status_t mxfp8_quantize_3d_experts(const void* w_bf16, int32_t G, int64_t N, int64_t K, unsigned dirs,
                                                    int scale_layout, void* q, void* s, void* qT, void* sT,
                                                    int32_t* dev_status, mxfp8_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (G < 1 || G > MXFP8_MAX_GROUPS || N <= 0 || K <= 0) return MXFP8_ERR_SHAPE;
    if (N % 32 || K % 32) return MXFP8_ERR_ALIGN;
    if (scale_layout != MXFP8_SCALES_COMPACT && scale_layout != MXFP8_SCALES_BLOCKED) return MXFP8_ERR_LAYOUT;
    const bool row = dirs & MXFP8_ROW, col = dirs & MXFP8_COL;
    if ((dirs & ~7u) || !(row || col)) return MXFP8_ERR_LAYOUT;  // BLOCK32X32 only together with ROW and/or COL
    if (!w_bf16) return MXFP8_ERR_NULL;
    if (row && (!q || !s)) return MXFP8_ERR_NULL;
    if (col && (!qT || !sT)) return MXFP8_ERR_NULL;
    if (!host::aligned16(w_bf16) || !host::aligned16(q) || !host::aligned16(s) || !host::aligned16(qT) ||
        !host::aligned16(sT))
        return MXFP8_ERR_ALIGN;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    const bool blocked = scale_layout == MXFP8_SCALES_BLOCKED;
    QParams p{};
    p.x = static_cast<const uint16_t*>(w_bf16);
    p.R = N; p.C = K; p.batch = G;
    p.q_row = static_cast<uint8_t*>(q); p.s_row = static_cast<uint8_t*>(s);
    p.q_col = static_cast<uint8_t*>(qT); p.s_col = static_cast<uint8_t*>(sT);
    p.s_row_bstride = blocked ? ((N + 127) / 128) * 128 * ((K + 127) / 128) * 4 : N * (K / 32);
    p.s_col_bstride = blocked ? ((K + 127) / 128) * 128 * ((N + 127) / 128) * 4 : K * (N / 32);
    p.blocked = blocked ? 1 : 0;
    p.offs = nullptr; p.G = 0;
    p.dev_status = dev_status;
    p.tiles_r = (N + 127) / 128; p.tiles_c = (K + 127) / 128; p.ntiles = p.tiles_r * p.tiles_c * G;
    if (p.ntiles >= INT32_MAX) return MXFP8_ERR_SHAPE;
    if (mxfp8_status_t r = launch_tiles(dirs, p, st); r != MXFP8_OK) return r;
    return MXFP8_OK;
}

extern "C" mxfp8_status_t mxfp8_check_offsets(const int32_t* offs, int32_t G, int64_t M, int32_t align,
                                              int32_t* dev_status, mxfp8_stream_t stream) {
    if (!offs || !dev_status) return MXFP8_ERR_NULL;
    if (G < 1 || G > MXFP8_MAX_GROUPS || M < 0) return MXFP8_ERR_SHAPE;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    check_offsets_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(offs, G, M, align, dev_status);
    return host::last_launch_status();
}

extern "C" mxfp8_status_t mxfp8_swiglu_bwd_quantize(const void* dh_bf16, const void* h1_bf16, const void* h3_bf16,
                                                    int64_t M, int64_t H, const int32_t* offs, int32_t G,
                                                    void* dh1_q, void* dh1_s, void* dh1T_q, void* dh1T_s, void* dh3_q,
                                                    void* dh3_s, void* dh3T_q, void* dh3T_s, int32_t* dev_status,
                                                    mxfp8_stream_t stream) {
    if (!dh_bf16 || !h1_bf16 || !h3_bf16 || !offs || !dh1_q || !dh1_s || !dh1T_q || !dh1T_s || !dh3_q || !dh3_s ||
        !dh3T_q || !dh3T_s)
        return MXFP8_ERR_NULL;
    if (M < 0 || H <= 0 || G < 1 || G > MXFP8_MAX_GROUPS || M > INT32_MAX) return MXFP8_ERR_SHAPE;
    if (H % 32 || M % 32) return MXFP8_ERR_ALIGN;
    const void* ptrs[] = {dh_bf16, h1_bf16, h3_bf16, dh1_q, dh1_s, dh1T_q, dh1T_s, dh3_q, dh3_s, dh3T_q, dh3T_s};
    for (const void* q : ptrs)
        if (!host::aligned16(q)) return MXFP8_ERR_ALIGN;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    if (M == 0) return MXFP8_OK;
    QParams p{};
    p.x = static_cast<const uint16_t*>(dh_bf16);
    p.R = M; p.C = H; p.batch = 1;
    p.q_row = static_cast<uint8_t*>(dh1_q); p.s_row = static_cast<uint8_t*>(dh1_s);
    p.q_col = static_cast<uint8_t*>(dh1T_q); p.s_col = static_cast<uint8_t*>(dh1T_s);
    p.q_row2 = static_cast<uint8_t*>(dh3_q); p.s_row2 = static_cast<uint8_t*>(dh3_s);
    p.q_col2 = static_cast<uint8_t*>(dh3T_q); p.s_col2 = static_cast<uint8_t*>(dh3T_s);
    p.blocked = 1;
    p.offs = offs; p.G = G;
    p.dev_status = dev_status;
    p.tiles_r = (M + 127) / 128; p.tiles_c = (H + 127) / 128; p.ntiles = p.tiles_r * p.tiles_c;
    if (p.ntiles >= INT32_MAX) return MXFP8_ERR_SHAPE;
    p.x2 = static_cast<const uint16_t*>(h1_bf16);
    p.x3 = static_cast<const uint16_t*>(h3_bf16);
    return launch_swiglu_bwd(p, reinterpret_cast<cudaStream_t>(stream));
}
