// grouped_mm.cu -- block-scaled MXFP8 grouped GEMMs (forward, dgrad, wgrad)
// for sm_103a on the 5th-generation tensor cores.
//
// What is computed ("MXFP8 training for MoEs", engine paragraph and "Why Does
// MXFP8 Speed Up MoE Training": routed experts run as grouped GEMMs over
// tokens sorted by expert, forward and a mirrored backward; "MXFP8
// (Micro-scaling FP8)", "Low-precision Flash Attention": scales run along each
// GEMM's K):
//   fwd    out[m, n]   = sum_k  A[m,k]    W[g][n,k]      (rows of group g)
//   dgrad  dA[m, k]    = sum_n  dOut[m,n] W[g][n,k]      (W quantized along N)
//   wgrad  dW[g][n, k] = sum_{m in g} dOut[m,n] A[m,k]    (both quantized along tokens)
// All three are one "TN" contraction of two K-major e4m3 operands with E8M0
// scales per 32 K-elements in the blocked tensor-core layout; they differ only
// in how tiles map to groups:
//   ROWGROUPED (fwd, dgrad): the token operand's rows are split by group; each
//     group's rows are tiled by 128 and contracted with that expert's matrix.
//   KGROUPED (wgrad): every group owns a full output matrix; its contraction
//     runs over the group's own tokens only (empty group -> zeros).  A group's
//     last 128-token box may reach into the next group; only the 32-token
//     blocks inside the group are multiplied, so another group's values
//     (NaN included) never enter its sum.
//
// Two kernels: the CTA-pair kernel (below) runs every GEMM whose output is at least 256 wide,
// including the SwiGLU gate/up and the two-operand dgrad variants; the single-CTA kernel runs
// the narrower ones (tiles of 128 x 128).
//
// Single-CTA kernel structure (one CTA per SM, persistent over a static tile order):
//   warp 0      TMA producer: 128B-swizzled A/B tiles (128 x 128 B and BN x 128 B)
//               and the matching 512-byte scale tiles into a ring of SMEM stages.
//   warp 1      MMA issuer: four tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each,
//               scale byte k of the 32-bit TMEM scale word) per stage into an fp32
//               accumulator in tensor memory; tcgen05.commit frees stages.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each warp its 32-lane
//               quarter), fp32 -> bf16 round-to-nearest-even, masked 16-byte
//               stores of the rows and columns that belong to the tile's group.
//   warp 6      scale copies: as soon as a stage lands, tcgen05.cp moves its scale
//               tiles into that stage's tensor-memory columns and signals the MMA
//               issuer; off the issuer's thread, the copies do not hold its MMAs back.
// Every mbarrier wait is bounded (MXFP8_ERR_TIMEOUT + orderly exit).

#include "common.cuh"
#include "host_common.h"

namespace mx {

constexpr int BM = 128;  // tile rows = tensor-memory lanes
constexpr int BK = 128;  // contraction bytes (= e4m3 elements) per stage: one 128-byte swizzle row
constexpr int kThreads = 224;  // producer, MMA issuer, 4 epilogue warps, scale-copy warp
constexpr int kSfWarp = 6;     // the warp that copies each stage's scale tiles into tensor memory
constexpr int kBand = 16;  // m-tiles per raster band (tiles of a band share B tiles in L2)

enum GemmMode : int { ROWGROUPED = 0, KGROUPED = 1 };

template <int BN>
struct Cfg {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kAcc = BN == 256 ? 1 : 2;
    static constexpr int kABytes = BM * BK;
    static constexpr int kBBytes = BN * BK;
    static constexpr int kSfaBytes = 512;
    static constexpr int kSfbBytes = (BN / 128) * 512;
    static constexpr int kTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kSfCols = 4 + BN / 32;           // tensor-memory columns of one stage's scales
    static constexpr int kSfCol0 = BN * kAcc;             // first scale column
    static constexpr int kTmemCols = 512;
    static_assert(kSfCol0 + kStages * kSfCols <= kTmemCols, "tensor memory overflow");
    static constexpr int kOffB = kStages * kABytes;
    static constexpr int kOffSfa = kOffB + kStages * kBBytes;
    static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
    static constexpr int kOffStage = kOffSfb + kStages * kSfbBytes;  // epilogue staging: 4 warps x 32 rows x 128 B
    static constexpr int kStageBytes = 4 * 32 * 128;
    static constexpr int kOffBar = kOffStage + kStageBytes;
    static constexpr int kBarBytes = (3 * kStages + 2 * kAcc + 2) * 8 + 16;
    static constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + alignment slack
};

struct GemmParams {
    const uint8_t* sfa;       // blocked scales of the A operand
    const uint8_t* sfb;       // blocked scales of the B operand
    int64_t sfa_ct;           // ROWGROUPED: column tiles per 128-row band of A scales
    int64_t sfb_ct;           // ROWGROUPED: same for B scales
    int64_t sfb_estride;      // ROWGROUPED: bytes of B scales per expert
    int64_t na;               // KGROUPED: rows of A (= N); ROWGROUPED: unused
    int64_t nb;               // rows of B per expert (ROWGROUPED) or in total (KGROUPED)
    int64_t kc;               // ROWGROUPED: contraction length
    const int32_t* offs;
    int32_t G;
    int64_t M;                // tokens
    __nv_bfloat16* out;
    int64_t ldo;              // ROWGROUPED: output row pitch (elements)
    int mode;
    int need32;               // group sizes must be multiples of 32 (token-wise blocks or TMA coordinates)
    int32_t* dev_status;
    uint64_t timeout_ns;
    // SwiGLU gate/up variant only (CTA-pair kernel): the even CTA's B rows come from the gate weights
    // (sfb), the odd CTA's from the up weights (sfb2); out = h1, out2 = h3; h = silu(h1) * h3 quantized
    // along its row into hq/hs (blocked, row groups) and along the tokens into hTq/hTs (blocked, token
    // groups).
    const uint8_t* sfb2;      // also: second B operand's scales of the two-operand dgrad
    const uint8_t* sfa2;      // two-operand dgrad only: second A operand's scales
    __nv_bfloat16* out2;
    uint8_t* hq;
    uint8_t* hs;
    int64_t hs_ct;            // column tiles of the row-wise h scales (= ceil(H / 128))
    uint8_t* hTq;             // nullable (with hTs): no token-wise copy
    uint8_t* hTs;
};

struct TileInfo {
    int g;
    int64_t a_row, b_row;     // TMA row coordinates
    int64_t a_x0;             // TMA contraction coordinate of k-tile 0
    int k_tiles;
    int kb_last;              // 32-wide K blocks of the last k-tile that belong to the tile (KGROUPED: the
                              // group's own tokens; the rest of that TMA box is the next group's)
    int64_t sfa_base;         // byte offset of k-tile 0's A scale tile
    int64_t sfb_base[2];      // byte offsets of k-tile 0's B scale tiles
    int64_t sf_kstep;         // bytes between consecutive k-tiles' scale tiles (always 512)
    __nv_bfloat16* out;       // first element of the tile
    int64_t ldo;
    int valid_rows, valid_cols;
    int64_t prow0;            // ROWGROUPED: padded (per-group 128-aligned) row of the tile's first row
    int64_t col0;             // first output column
};

// Tile l of an mt x nt grid walked in bands of `bandw` m-tiles, each band n-tile by n-tile.
__device__ __forceinline__ int band_split(int64_t l, int64_t mt, int64_t nt, int64_t& m, int64_t& n,
                                          int64_t bandw = kBand) {
    const int64_t band = l / (bandw * nt);
    const int64_t bm = min64(bandw, mt - band * bandw);
    const int64_t idx = l - band * bandw * nt;
    n = idx / bm;
    m = band * bandw + (idx - n * bm);
    return 0;
}

// kDualK (ROWGROUPED): the contraction runs over two operand pairs one after the other, k-tiles
// 0 .. k/2-1 over (A, B) and k/2 .. k-1 over (A2, B2), into one accumulator.
template <int BN, bool kDualK = false>
__device__ __forceinline__ TileInfo tile_info(const GemmParams& p, int64_t t, const int32_t* ends_s,
                                              const int32_t* pstart_s, int64_t ptotal) {
    constexpr int TN = BN;  // output columns per tile
    TileInfo ti;
    const int64_t ntb = (p.nb + TN - 1) / TN;  // tiles along B rows
    if (p.mode == ROWGROUPED) {
        // group of tile t: last g whose tile range starts at or before t
        int lo = 0, hi = p.G;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)(pstart_s[mid] / BM) * ntb <= t) lo = mid + 1;
            else hi = mid;
        }
        const int g = lo - 1;
        const int64_t start = g ? ends_s[g - 1] : 0, size = ends_s[g] - start;
        const int64_t mt = (size + BM - 1) / BM;
        int64_t m, n;
        band_split(t - (int64_t)(pstart_s[g] / BM) * ntb, mt, ntb, m, n);
        ti.g = g;
        ti.a_row = start + m * BM;
        ti.b_row = (int64_t)g * p.nb + n * TN;
        ti.a_x0 = 0;
        ti.k_tiles = (int)((p.kc + BK - 1) / BK) * (kDualK ? 2 : 1);
        ti.kb_last = BK / 32;  // a K tail past the contraction reads TMA's zero fill
        ti.sfa_base = ((int64_t)(pstart_s[g] / BM + m) * p.sfa_ct) * 512;
        const int64_t last_chunk = (p.nb + 127) / 128 - 1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t ch = min64(n * (BN / 128) + j, last_chunk);
            ti.sfb_base[j] = (int64_t)g * p.sfb_estride + ch * p.sfb_ct * 512;
        }
        ti.out = p.out + ti.a_row * p.ldo + n * TN;
        ti.ldo = p.ldo;
        ti.valid_rows = (int)min64(BM, size - m * BM);
        ti.valid_cols = (int)min64(TN, p.nb - n * TN);
        ti.prow0 = (int64_t)pstart_s[g] + m * BM;
        ti.col0 = n * TN;
    } else {
        const int64_t nta = (p.na + BM - 1) / BM;
        const int64_t per_g = nta * ntb;
        const int g = (int)(t / per_g);
        int64_t m, n;
        band_split(t - g * per_g, nta, ntb, m, n);
        const int64_t start = g ? ends_s[g - 1] : 0, size = ends_s[g] - start;
        const int64_t ct = ptotal / 128;           // column tiles of the token-grouped scale layout
        const int64_t kt0 = pstart_s[g] / 128;     // this group's first column tile
        ti.g = g;
        ti.a_row = m * BM;
        ti.b_row = n * BN;
        ti.a_x0 = start;
        ti.k_tiles = (int)((size + BK - 1) / BK);
        ti.kb_last = (int)(((size - 1) & (BK - 1)) / 32) + 1;  // size % 32 == 0 (checked)
        ti.sfa_base = (m * ct + kt0) * 512;
        const int64_t last_chunk = (p.nb + 127) / 128 - 1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t ch = min64(n * (BN / 128) + j, last_chunk);
            ti.sfb_base[j] = (ch * ct + kt0) * 512;
        }
        ti.out = p.out + ((int64_t)g * p.na + m * BM) * p.nb + n * BN;
        ti.ldo = p.nb;
        ti.valid_rows = (int)min64(BM, p.na - m * BM);
        ti.valid_cols = (int)min64(BN, p.nb - n * BN);
        ti.prow0 = 0;
        ti.col0 = n * BN;
    }
    ti.sf_kstep = 512;
    return ti;
}

__device__ __forceinline__ void st_shared_u8(void* p, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Codes of a non-finite block (scale 0xFF): 0x7F with each element's sign, for a bf16 pair.
__device__ __forceinline__ uint32_t nonfinite_codes2(uint32_t v) {
    return 0x7F7Fu | ((v >> 8) & 0x80u) | ((v >> 16) & 0x8000u);
}

// One bf16 pair times f (a power of two, exact) -> two E4M3 codes (RNE, satfinite).
__device__ __forceinline__ uint32_t quant_pair(uint32_t v, float f) { return cvt_e4m3x2(bf16lo(v) * f, bf16hi(v) * f); }

// One tile of the SwiGLU epilogue, for one warp: TMEM lane quarter `quarter` (32 rows of the tile,
// one per lane) and 32-column block jb of the tile's 128 h columns.  acc: tensor-memory address of the
// warp's gate columns (the up columns sit 128 further).  h1 (gate) and h3 (up) are rounded to bf16 and
// stored; h = bf16(bf16(silu(h1)) * h3) with silu(x) = x / (1 + e^-x) in fp32 (the bf16 rounding points
// of an elementwise bf16 SwiGLU); h is quantized to MXFP8 along its row and, if p.hTq, along the tokens.
// release() hands the accumulator back once it is in registers.  a_row: the tile's first token row;
// valid_rows / valid_cols: rows inside the group and columns inside H; prow0: the padded (128-aligned per
// group) row of the tile's first row; col0: its first column; ct_T: column tiles of the h^T scales.
__device__ __forceinline__ void st_shared_u32(void* p, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Largest magnitude of each half of two bf16 pairs, NaN winning (the sign bits left are not used).
__device__ __forceinline__ uint32_t amax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 32 bf16 values (16 pairs) -> their MXFP8 block: the E8M0 scale byte s from the amax's exponent field
// and, in c[8], the 32 E4M3 codes (RNE, satfinite) of x * 2^(127 - s).  The products come from one
// mixed-precision fma per element with the scale as a bf16 (exact, and zero keeps its sign); a block
// whose amax is Inf or NaN gets scale 0xFF and the codes 0x7F with each element's sign.
__device__ __forceinline__ uint32_t mx_block32(const uint32_t (&w)[16], uint32_t (&c)[8]) {
    uint32_t m = w[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) m = amax_bf16x2(m, w[i]);
    const uint32_t sc = e8m0_from_absbits(max(m & 0x7FFFu, (m >> 16) & 0x7FFFu));
    const uint32_t f2 = (254u - sc) << 7;  // 2^(127 - sc) as a bf16 (sc <= 246 for a finite amax)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t pr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float lo, hi;
            asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
                "fma.rn.f32.bf16 %0, a0, b0, 0f80000000;\n\tfma.rn.f32.bf16 %1, a1, b0, 0f80000000;\n\t}"
                : "=f"(lo), "=f"(hi)
                : "r"(w[2 * i + h]), "r"(f2));
            pr[h] = cvt_e4m3x2(lo, hi);
        }
        c[i] = pr[0] | (pr[1] << 16);
    }
    if (sc == 0xFFu) {  // a non-finite block (rare): the codes are 0x7F with each element's sign
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = nonfinite_codes2(w[2 * i]) | (nonfinite_codes2(w[2 * i + 1]) << 16);
    }
    return sc;
}

// Row-wise and (if qT) token-wise MXFP8 quantization of one 32 x 32 bf16 block held by a warp: lane l owns
// row 32 * quarter + l of a 128-row tile, w[i] its columns c0 + 2i, c0 + 2i + 1.  Row-wise: codes into
// q [rows, H], scale bytes into the blocked row-group layout s (s_ct column tiles of 128); token-wise: the
// block's 32 tokens of each column are one block, codes into qT [H, M], scale bytes into the blocked
// token-group layout sT (ct_T column tiles).  stg: the warp's 2 KB of shared memory, through which the
// block is transposed (word (pair p, row r) at p * 32 + (r ^ p): conflict-free both ways).  a_row: the
// tile's first token row; valid_rows: its rows inside the group (group sizes are multiples of 32 where
// qT is given); prow0: the padded (128-aligned per group) row of its first row.  Blocks past H write
// padding (0) up to the layouts' 128-column round-up and nothing beyond it.
__device__ __forceinline__ void quant_block_rowcol(const uint32_t (&w)[16], uint8_t* q, uint8_t* s, int64_t s_ct,
                                                   uint8_t* qT, uint8_t* sT, int64_t H, int64_t M, int64_t ct_T,
                                                   int quarter, int lane, uint8_t* stg, int64_t a_row, int valid_rows,
                                                   int64_t prow0, int64_t c0) {
    if ((c0 >> 7) >= s_ct) return;
    const int r = quarter * 32 + lane;
    const bool bvalid = c0 < H;          // this column block lies inside H
    const bool rvalid = r < valid_rows;  // this row lies inside the group
    // row-wise: this thread's 32 elements are one block -> 32 codes and one scale byte
    {
        uint32_t codes[8];
        const uint32_t sc = mx_block32(w, codes);
        if (bvalid && rvalid) {
            uint4* gq = reinterpret_cast<uint4*>(q + (a_row + r) * H + c0);
            gq[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            gq[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        }
        // the tile's row scales are one 512-byte blocked tile: row r -> (r%32)*16 + (r/32)*4,
        // block (c0 / 32) % 4 -> that byte; rows past the group and blocks past H are padding (0)
        s[((prow0 >> 7) * s_ct + (c0 >> 7)) * 512 + lane * 16 + quarter * 4 + ((c0 >> 5) & 3)] =
            (uint8_t)((bvalid && rvalid) ? sc : 0u);
    }
    if (qT != nullptr) {
        // token-wise: lane t takes column c0 + t, whose 32 tokens (the warp's rows) are one block.
        // Group sizes are multiples of 32 here (device-checked), so the warp's rows are all inside the
        // group or all padding.
        const bool cvalid = c0 + lane < H && valid_rows > quarter * 32;
        uint32_t sc = 0;
        if (bvalid && valid_rows > quarter * 32) {
#pragma unroll
            for (int p2 = 0; p2 < 16; ++p2) st_shared_u32(stg + 4 * (p2 * 32 + (lane ^ p2)), w[p2]);
            __syncwarp();
            const int pc = lane >> 1;  // the pair that holds column c0 + lane
            uint32_t tw[16];           // its tokens 2i, 2i + 1 as bf16 pairs
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t x0 = ld_shared_u32(stg + 4 * (pc * 32 + ((2 * i) ^ pc)));
                const uint32_t x1 = ld_shared_u32(stg + 4 * (pc * 32 + ((2 * i + 1) ^ pc)));
                tw[i] = __byte_perm(x0, x1, (lane & 1) ? 0x7632u : 0x5410u);
            }
            __syncwarp();
            uint32_t codes[8];
            sc = mx_block32(tw, codes);
            if (cvalid) {
                uint4* gq = reinterpret_cast<uint4*>(qT + (c0 + lane) * M + a_row + quarter * 32);
                gq[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
                gq[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
            } else {
                sc = 0;
            }
        }
        const int64_t cq = prow0 / 32 + quarter;  // scale column of this 32-token block
        const int64_t cH = c0 + lane;             // row of h^T (columns past H: padding 0)
        sT[((cH >> 7) * ct_T + (cq >> 2)) * 512 + (cH & 31) * 16 + ((cH >> 5) & 3) * 4 + (cq & 3)] = (uint8_t)sc;
    }
}

template <class Release>
__device__ __forceinline__ void swiglu_tile_epilogue(const GemmParams& p, uint32_t acc, int quarter, int jb, int lane,
                                                     uint8_t* stg, int64_t a_row, int valid_rows, int valid_cols,
                                                     int64_t prow0, int64_t col0, int64_t ct_T, Release release) {
    const int64_t H = p.nb;
    uint32_t hg[16], hu[16];  // bf16 pairs (columns 2i, 2i+1 of the block) of h1 and h3
    {
        uint32_t v[32];
        tmem_ld_32x32b_x32(acc, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) hg[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        tmem_ld_32x32b_x32(acc + 128, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) hu[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    }
    tc_fence_before();
    __syncwarp();
    release();

    const bool bvalid = 32 * jb < valid_cols;  // this column block lies inside H
    const int64_t c0 = col0 + 32 * jb;         // first column of the block
    // h1 and h3 through the warp's 1 KB staging buffer, 16 columns (32 bytes) of each of the
    // 32 rows per pass, so every store instruction writes 16 whole 32-byte row segments
    // instead of 32 scattered 16-byte pieces.  Chunk c of row l sits at l * 32 + 16 (c ^ s),
    // s = (l >> 2) & 1, which spreads a pass's writes over all banks.
    auto stage_store = [&](const uint32_t* w, __nv_bfloat16* dst_base, int h) {
        const int sw = (lane >> 2) & 1;
        st_shared_v4(stg + lane * 32 + 16 * (0 ^ sw), make_uint4(w[0], w[1], w[2], w[3]));
        st_shared_v4(stg + lane * 32 + 16 * (1 ^ sw), make_uint4(w[4], w[5], w[6], w[7]));
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int rl = (lane >> 1) + 16 * k, ch = lane & 1;
            const uint4 v = ld_shared_v4(stg + rl * 32 + 16 * (ch ^ ((rl >> 2) & 1)));
            if (bvalid && quarter * 32 + rl < valid_rows)
                *reinterpret_cast<uint4*>(dst_base + (a_row + quarter * 32 + rl) * H + c0 + 16 * h + 8 * ch) = v;
        }
        __syncwarp();
    };
    stage_store(hg, p.out, 0);
    stage_store(hg + 8, p.out, 1);
    stage_store(hu, p.out2, 0);
    stage_store(hu + 8, p.out2, 1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = bf16lo(hg[i]), b = bf16hi(hg[i]);
        const uint32_t sl = pack_bf16x2(a / (1.0f + expf(-a)), b / (1.0f + expf(-b)));
        hg[i] = pack_bf16x2(bf16lo(sl) * bf16lo(hu[i]), bf16hi(sl) * bf16hi(hu[i]));
    }
    quant_block_rowcol(hg, p.hq, p.hs, p.hs_ct, p.hTq, p.hTs, H, p.M, ct_T, quarter, lane, stg, a_row, valid_rows,
                       prow0, c0);
}

template <int BN, bool kDualK = false>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_mm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_b2, const __grid_constant__ CUtensorMap tmap_a2,
                      const GemmParams p) {
    using C = Cfg<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int32_t ends_s[kMaxGroups];
    __shared__ int32_t pstart_s[kMaxGroups];
    __shared__ int32_t ptotal_s;
    __shared__ int32_t bad_s;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + C::kAcc;
    uint64_t* drain = tempty + C::kAcc;
    uint64_t* sfull = drain + 1;             // a stage's scale tiles are in tensor memory
    uint64_t* sfdrain = sfull + C::kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- group table (warp 0), barriers (warp 1 lane 0), tensor memory (warp 1)
    if (warp == 0) {
        // clamped monotone ends and padded starts (multiples of 128 rows / tokens)
        const int G = p.G;
        const int per = (G + 31) / 32;
        const int g0 = lane * per, g1 = min(G, g0 + per);
        const int32_t Mc = (int32_t)p.M;
        int32_t mx = 0;
        for (int g = g0; g < g1; ++g) mx = max(mx, min(max(p.offs[g], 0), Mc));
        int32_t incl = mx;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl = max(incl, o);
        }
        int32_t run = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) run = 0;
        int32_t prev = run, psum = 0, bad = 0;
        for (int g = g0; g < g1; ++g) {
            const int32_t e = max(prev, min(max(p.offs[g], 0), Mc));
            ends_s[g] = e;
            if (p.need32 && (e - prev) % 32 != 0) bad = 1;  // token blocks / 16-byte TMA token coordinates
            psum += ((e - prev + 127) / 128) * 128;
            prev = e;
        }
        int32_t sincl = psum;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, sincl, d);
            if (lane >= d) sincl += o;
        }
        int32_t sexcl = sincl - psum;
        prev = run;
        for (int g = g0; g < g1; ++g) {
            pstart_s[g] = sexcl;
            const int32_t e = ends_s[g];
            sexcl += ((e - prev + 127) / 128) * 128;
            prev = e;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 31) ptotal_s = sincl;
        if (lane == 0) {
            bad_s = bad;
            abort_s = 0;
            prefetch_tmap(&tmap_a);
            prefetch_tmap(&tmap_b);
            if (kDualK) prefetch_tmap(&tmap_b2);
            if (kDualK) prefetch_tmap(&tmap_a2);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int s = 0; s < C::kStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            for (int a = 0; a < C::kAcc; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], 4);
            }
            mbar_init(drain, 1);
            for (int s = 0; s < C::kStages; ++s) mbar_init(&sfull[s], 1);
            mbar_init(sfdrain, 1);
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc(&tmem_base_s, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = tmem_base_s;
    volatile int* abort_flag = &abort_s;
    const int64_t ptotal = ptotal_s;
    if (bad_s) {
        if (threadIdx.x == 0) report(p.dev_status, MXFP8_ERR_OFFSETS);
    } else {
        const int64_t ntb = (p.nb + BN - 1) / BN;  // tiles along B rows (as in tile_info)
        const int64_t ntiles = p.mode == ROWGROUPED ? (ptotal / BM) * ntb
                                                    : (int64_t)p.G * ((p.na + BM - 1) / BM) * ntb;

        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, last_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info<BN, kDualK>(p, t, ends_s, pstart_s, ptotal);
                const int kt_half = kDualK ? ti.k_tiles / 2 : ti.k_tiles;
                for (int kt = 0; kt < ti.k_tiles; ++kt) {
                    if (!mbar_wait_bounded<true>(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * C::kABytes;
                    uint8_t* sb = smem + C::kOffB + stage * C::kBBytes;
                    uint8_t* ssa = smem + C::kOffSfa + stage * C::kSfaBytes;
                    uint8_t* ssb = smem + C::kOffSfb + stage * C::kSfbBytes;
                    mbar_arrive_expect_tx(&full[stage], C::kTx);
                    const bool second = kDualK && kt >= kt_half;  // second operand pair of a two-operand dgrad
                    const int kk = second ? kt - kt_half : kt;
                    const int32_t kx = (int32_t)(ti.a_x0 + (int64_t)kk * BK);
                    tma_load_2d(sa, second ? &tmap_a2 : &tmap_a, kx, (int32_t)ti.a_row, &full[stage]);
                    bulk_load(ssa, (second ? p.sfa2 : p.sfa) + ti.sfa_base + kk * ti.sf_kstep, 512, &full[stage]);
                    tma_load_2d(sb, second ? &tmap_b2 : &tmap_b, kx, (int32_t)ti.b_row, &full[stage]);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        bulk_load(ssb + j * 512, (second ? p.sfb2 : p.sfb) + ti.sfb_base[j] + kk * ti.sf_kstep, 512,
                                  &full[stage]);
                    issued_mask |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let copies already in flight land before the CTA exits
                for (int s = 0; s < C::kStages; ++s)
                    if (issued_mask & (1u << s)) {
                        volatile int no_abort = 0;
                        mbar_wait_bounded<true>(&full[s], (last_phase >> s) & 1u, p.timeout_ns, &no_abort, nullptr);
                    }
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info<BN, kDualK>(p, t, ends_s, pstart_s, ptotal);
                if (ti.k_tiles == 0) continue;
                if (!mbar_wait_bounded<true>(&tempty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * BN;
                for (int kt = 0; kt < ti.k_tiles; ++kt) {
                    const int cur = stage;
                    if (!mbar_wait_bounded<true>(&full[cur], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded<true>(&sfull[cur], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    const uint32_t sfa_t = tmem + C::kSfCol0 + cur * C::kSfCols;
                    const uint32_t sfb_t = sfa_t + 4;
                    const uint32_t a_s = smem_u32(smem + cur * C::kABytes);
                    const uint32_t b_s = smem_u32(smem + C::kOffB + cur * C::kBBytes);
                    if (kt + 1 < ti.k_tiles || ti.kb_last == BK / 32) {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint64_t ad = smem_desc(a_s + 32 * k, 16, 1024, 2);
                            const uint64_t bd = smem_desc(b_s + 32 * k, 16, 1024, 2);
                            tc_mma_mxf8(d_tmem, ad, bd, idesc_mxf8(BM, BN, k, k), sfa_t, sfb_t, (kt | k) != 0);
                        }
                    } else {
                        // K-grouped last k-tile: only the group's own 32-token blocks (the box's other
                        // columns hold the next group's tokens, whose codes may be NaN)
#pragma unroll 1
                        for (int k = 0; k < ti.kb_last; ++k) {
                            const uint64_t ad = smem_desc(a_s + 32 * k, 16, 1024, 2);
                            const uint64_t bd = smem_desc(b_s + 32 * k, 16, 1024, 2);
                            tc_mma_mxf8(d_tmem, ad, bd, idesc_mxf8(BM, BN, k, k), sfa_t, sfb_t, (kt | k) != 0);
                        }
                    }
                    tc_commit(&empty[cur]);
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
                if (++acc == C::kAcc) { acc = 0; acc_phase ^= 1u; }
            }
            // all tensor-core work of this CTA must be done before the columns are freed
            tc_commit(drain);
            volatile int no_abort = 0;
            mbar_wait_bounded<true>(drain, 0, p.timeout_ns, &no_abort, p.dev_status);
        } else if (warp == kSfWarp) {
            // ------------------------------------------------ scale copies
            // As soon as a stage lands, its scale tiles go to that stage's tensor-memory columns
            // (tcgen05.cp, SMEM -> TMEM) and the copy's completion is signalled on sfull; the MMA
            // thread waits for it before the stage's MMAs.  A stage's columns are rewritten only
            // after the stage was refilled, i.e. after the MMAs that read them completed.
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                    const TileInfo ti = tile_info<BN, kDualK>(p, t, ends_s, pstart_s, ptotal);
                    for (int kt = 0; kt < ti.k_tiles; ++kt) {
                        if (!mbar_wait_bounded<true>(&full[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sfa_t = tmem + C::kSfCol0 + stage * C::kSfCols;
                        const uint32_t sfa_s = smem_u32(smem + C::kOffSfa + stage * C::kSfaBytes);
                        const uint32_t sfb_s = smem_u32(smem + C::kOffSfb + stage * C::kSfbBytes);
                        tc_cp_32x128b_warpx4(sfa_t, smem_desc(sfa_s, 0, 128, 0));
#pragma unroll
                        for (int j = 0; j < BN / 128; ++j)
                            tc_cp_32x128b_warpx4(sfa_t + 4 + 4 * j, smem_desc(sfb_s + 512 * j, 0, 128, 0));
                        tc_commit(&sfull[stage]);
                        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    }
                }
                // this thread's copies complete before the columns are freed
                tc_commit(sfdrain);
                volatile int no_abort = 0;
                mbar_wait_bounded<true>(sfdrain, 0, p.timeout_ns, &no_abort, p.dev_status);
            }
        } else if (warp >= 2) {
          {
            // ------------------------------------------------ epilogue
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;  // accumulator row (= tensor-memory lane) of this thread
            uint8_t* stg = smem + C::kOffStage + (warp - 2) * (32 * 128);
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
                const TileInfo ti = tile_info<BN, kDualK>(p, t, ends_s, pstart_s, ptotal);
                const bool row_ok = r < ti.valid_rows;
                __nv_bfloat16* orow = ti.out + (int64_t)r * ti.ldo;
                __nv_bfloat16* wout = ti.out + (int64_t)(quarter * 32) * ti.ldo;  // first row of this warp
                if (ti.k_tiles == 0) {
                    if (row_ok)
                        for (int c = 0; c < ti.valid_cols; c += 8)
                            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
                    continue;
                }
                if (!mbar_wait_bounded<true>(&tfull[acc], acc_phase, p.timeout_ns, abort_flag, p.dev_status)) break;
                tc_fence_after();
                // Drain the whole accumulator row into registers as bf16 pairs, then hand the
                // columns back to the MMA warp before any global store is issued.
                uint32_t packed[BN / 2];
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * BN;
#pragma unroll
                for (int c = 0; c < BN; c += 64) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(taddr + c, v0);
                    tmem_ld_32x32b_x32(taddr + c + 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        packed[c / 2 + i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
                        packed[c / 2 + 16 + i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(&tempty[acc]);
                // Coalesced stores: per 64-column chunk, each lane parks its row's eight 16-byte pieces in
                // the warp's 32 x 128 B staging buffer (piece j of row r at slot j ^ (r & 7): no bank
                // conflicts), then every store instruction writes 4 full 128-byte row segments.
                const int vrows = ti.valid_rows - quarter * 32;  // rows of this warp inside the group
#pragma unroll
                for (int ch = 0; ch < BN / 64; ++ch) {
                    if (ch * 64 >= ti.valid_cols) break;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) * 16),
                                     make_uint4(packed[ch * 32 + 4 * j], packed[ch * 32 + 4 * j + 1],
                                                packed[ch * 32 + 4 * j + 2], packed[ch * 32 + 4 * j + 3]));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rl = (lane >> 3) + 4 * i, piece = lane & 7;
                        const uint4 val = ld_shared_v4(stg + rl * 128 + ((piece ^ (rl & 7)) * 16));
                        if (rl < vrows && ch * 64 + piece * 8 < ti.valid_cols)
                            *reinterpret_cast<uint4*>(wout + (int64_t)rl * ti.ldo + ch * 64 + piece * 8) = val;
                    }
                    __syncwarp();
                }
                if (++acc == C::kAcc) { acc = 0; acc_phase ^= 1u; }
            }
          }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}


// ============================================================================================
// CTA-pair variant (cluster of 2, tcgen05 cta_group::2): a 256 x 256 output tile per pair.
// Each CTA stages its own 128 rows of A and its own 128 rows of B (half of N) per k-tile, so a
// stage is 33.5 KB instead of 49.5 KB and the ring holds 5 stages; the even CTA issues one
// M=256 x N=256 x K=32 MMA per 32-wide K block that reads A and B from both CTAs' shared
// memory and writes rows 0-127 to its own tensor memory, rows 128-255 to the odd CTA's.
// Every copy of the pair completes on the even CTA's stage barrier (TMA cta_group::2 form),
// so the scale tiles are moved by TMA as well (tensor maps over the scale buffers, 512-byte
// boxes); the even CTA's scale-copy warp moves them into both CTAs' tensor memory.  Stage and
// accumulator release are multicast commits to both CTAs; the odd CTA's epilogue reports a
// drained accumulator to the even CTA with a remote mbarrier arrive.
// Variants: two-operand (a second (A2, B2) contraction into the same accumulator) and SwiGLU
// gate/up (a 128-column tile of h; the even CTA stages gate rows, the odd CTA the same up rows,
// and each CTA's 16 epilogue warps turn its own 128 token rows into h1, h3 and quantized h).
// ============================================================================================
constexpr int kSortGroups = 128;  // K-grouped schedules rank at most this many groups (O(G^2) per CTA)
// Epilogue warps of the pair kernel: two per tensor-memory lane quarter, each draining one 128-column
// half of the accumulator, so the single accumulator is handed back to the MMA warp in half the time
// (a K-grouped tile of a small group contracts over few k-tiles, and the drain is per tile).
constexpr int kPairEpiWarps = 8;
// The SwiGLU variant's epilogue (silu, two quantizations per element) runs 16 warps per CTA, four per
// lane quarter, one 32-column block of h each (swiglu_tile_epilogue).
constexpr int kPairSwiEpiWarps = 16;
template <bool kSwi>
constexpr int kPairEpiOf = kSwi ? kPairSwiEpiWarps : kPairEpiWarps;
template <bool kSwi>
constexpr int kPairSfWarpOf = 2 + kPairEpiOf<kSwi>;  // the scale-copy warp, after the epilogue warps
template <bool kSwi>
constexpr int kThreadsPairOf = 96 + 32 * kPairEpiOf<kSwi>;
// K-grouped pair tiles run in bands of 8 row-tiles: the 76 tiles of a wave then share about
// 8 A and 10 B operand slabs instead of 16 and 5 (a long group's slabs do not fit in L2 together).
constexpr int kBandPairK = 8;

// Operand stages: the plain and two-operand kernels stage their epilogue through 1 KB a warp, which
// leaves room in shared memory for six; the SwiGLU kernel's 16 epilogue warps stage 2 KB each and it
// keeps five.
template <bool kSwi>
struct CfgPair {
    static constexpr int BN = 256;
    static constexpr int kStages = kSwi ? 5 : 6;
    static constexpr int kABytes = BM * BK;          // this CTA's 128 rows of A
    static constexpr int kBBytes = 128 * BK;         // this CTA's 128 rows of B
    static constexpr int kSfaBytes = 512;
    static constexpr int kSfbBytes = 2 * 512;        // both 128-row scale tiles of the 256 B rows
    static constexpr int kTx = 2 * (kABytes + kBBytes + kSfaBytes + kSfbBytes);  // both CTAs' bytes
    static constexpr int kSfCols = 4 + BN / 32;
    static constexpr int kSfCol0 = BN;
    static constexpr int kTmemCols = 512;
    static_assert(kSfCol0 + kStages * kSfCols <= kTmemCols, "tensor memory overflow");
    static constexpr int kOffB = kStages * kABytes;
    static constexpr int kOffSfa = kOffB + kStages * kBBytes;
    static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
    static constexpr int kOffStage = kOffSfb + kStages * kSfbBytes;
    static constexpr int kStageBytes = kSwi ? kPairSwiEpiWarps * 2048 : kPairEpiWarps * 1024;
    static constexpr int kOffBar = kOffStage + kStageBytes;
    static constexpr int kBarBytes = (3 * kStages + 2 + 2) * 8 + 16;
    static constexpr int kSmem = kOffBar + kBarBytes + 1024;
};
static_assert(CfgPair<false>::kSmem + 3 * MXFP8_MAX_GROUPS * 4 + kSortGroups * 4 + 16 <= 227 * 1024,
              "pair kernel shared memory");
static_assert(CfgPair<true>::kSmem + 3 * MXFP8_MAX_GROUPS * 4 + kSortGroups * 4 + 16 <= 227 * 1024,
              "pair kernel shared memory");

struct PairTile {
    int g;
    int64_t a_row, b_row, a_x0;
    int k_tiles;
    int kb_last;                      // 32-wide K blocks of the last k-tile inside the tile's contraction
    int64_t sfa_chunk, sfb_chunk[2];  // 512-byte scale tiles of k-tile 0 (index = byte offset / 512)
    __nv_bfloat16* out;               // first element of this CTA's 128 rows
    int64_t prow0, col0;              // ROWGROUPED: padded (128-aligned per group) first row; first column
    int64_t ldo;
    int valid_rows, valid_cols;
};

// Tile t of the pair schedule, seen from CTA `half` (0: rows 0-127 of the pair tile, 1: 128-255).
// K-grouped: tile t belongs to the group at position t / per_g of gorder_s (or of the natural order).
// kSwi (ROWGROUPED): a pair tile is 128 output columns of h; the even CTA stages those 128 rows of the
// gate weights, the odd CTA the same rows of the up weights, so accumulator columns 0-127 of either
// CTA hold h1 for its own 128 token rows and columns 128-255 hold h3.
template <bool kDualK = false, bool kSwi = false>
__device__ __forceinline__ PairTile pair_tile(const GemmParams& p, int64_t t, int half, const int32_t* ends_s,
                                              const int32_t* pstart_s, const int32_t* tstart_s, int64_t ptotal,
                                              const int32_t* gorder_s, bool sorted) {
    constexpr int BN = 256;
    constexpr int TN = kSwi ? 128 : BN;  // output columns per tile
    PairTile ti;
    const int64_t ntb = (p.nb + TN - 1) / TN;
    const int64_t last_chunk = (p.nb + 127) / 128 - 1;
    if (p.mode == ROWGROUPED) {
        int lo = 0, hi = p.G;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)tstart_s[mid] * ntb <= t) lo = mid + 1;
            else hi = mid;
        }
        const int g = lo - 1;
        const int64_t start = g ? ends_s[g - 1] : 0, size = ends_s[g] - start;
        int64_t m2, n;
        band_split(t - (int64_t)tstart_s[g] * ntb, (size + 255) / 256, ntb, m2, n);
        const int64_t rows0 = m2 * 256 + half * 128;
        ti.g = g;
        ti.a_row = start + rows0;
        ti.b_row = (int64_t)g * p.nb + n * TN + (kSwi ? 0 : half * 128);
        ti.a_x0 = 0;
        ti.k_tiles = (int)((p.kc + BK - 1) / BK) * (kDualK ? 2 : 1);
        ti.kb_last = BK / 32;
        const int64_t cA = min64(2 * m2 + half, (size + 127) / 128 - 1);  // clamp: rows past the group are masked
        ti.sfa_chunk = (pstart_s[g] / 128 + cA) * p.sfa_ct;
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // kSwi: chunk n of the gate scales (j = 0) and of the up scales (j = 1)
            const int64_t ch = kSwi ? n : min64(n * 2 + j, last_chunk);
            ti.sfb_chunk[j] = (int64_t)g * (p.sfb_estride / 512) + ch * p.sfb_ct;
        }
        ti.out = p.out + ti.a_row * p.ldo + n * TN;
        ti.ldo = p.ldo;
        ti.valid_rows = (int)max64(-1, min64(128, size - rows0));  // <= 0: past the group's padded rows
        ti.valid_cols = (int)min64(TN, p.nb - n * TN);
        ti.prow0 = (int64_t)pstart_s[g] + rows0;
        ti.col0 = n * TN;
    } else {
        const int64_t nta2 = (p.na + 255) / 256;
        const int64_t per_g = nta2 * ntb;
        const int gp = (int)(t / per_g);
        const int g = sorted ? gorder_s[gp] : gp;
        int64_t m2, n;
        band_split(t - gp * per_g, nta2, ntb, m2, n, kBandPairK);
        const int64_t start = g ? ends_s[g - 1] : 0, size = ends_s[g] - start;
        const int64_t ct = ptotal / 128, kt0 = pstart_s[g] / 128;
        const int64_t rows0 = m2 * 256 + half * 128;
        ti.g = g;
        ti.a_row = rows0;
        ti.b_row = n * BN + half * 128;
        ti.a_x0 = start;
        ti.k_tiles = (int)((size + BK - 1) / BK);
        ti.kb_last = (int)(((size - 1) & (BK - 1)) / 32) + 1;  // size % 32 == 0 (checked)
        const int64_t cA = min64(2 * m2 + half, (p.na + 127) / 128 - 1);
        ti.sfa_chunk = cA * ct + kt0;
#pragma unroll
        for (int j = 0; j < 2; ++j) ti.sfb_chunk[j] = min64(n * 2 + j, last_chunk) * ct + kt0;
        ti.out = p.out + ((int64_t)g * p.na + rows0) * p.nb + n * BN;
        ti.ldo = p.nb;
        ti.valid_rows = (int)max64(-1, min64(128, p.na - rows0));
        ti.valid_cols = (int)min64(BN, p.nb - n * BN);
    }
    return ti;
}

// kDualK (row-grouped only): the contraction runs over two operand sets one after the other, k-tiles
// 0 .. k/2-1 over (A, B) and k/2 .. k-1 over (A2, B2), into one accumulator.
// kSwi: the SwiGLU gate/up variant (pair_tile, swiglu_tile_epilogue); tmap_b2 / tmap_sfb2 are the up
// weights and their scales.
template <bool kDualK, bool kSwi = false>
__global__ void __launch_bounds__(kThreadsPairOf<kSwi>, 1)
    grouped_mm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                           const __grid_constant__ CUtensorMap tmap_a2, const __grid_constant__ CUtensorMap tmap_b2,
                           const __grid_constant__ CUtensorMap tmap_sfa2, const __grid_constant__ CUtensorMap tmap_sfb2,
                           const GemmParams p) {
    using C = CfgPair<kSwi>;
    constexpr int BN = 256;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ int32_t ends_s[kMaxGroups];
    __shared__ int32_t pstart_s[kMaxGroups];
    __shared__ int32_t tstart_s[kMaxGroups];  // ROWGROUPED: first pair tile (256 rows) of each group
    __shared__ int32_t gorder_s[kSortGroups];  // K-grouped, G <= kSortGroups: groups by size, largest first
    __shared__ int32_t ptotal_s;
    __shared__ int32_t bad_s;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + C::kStages;
    uint64_t* tfull = empty + C::kStages;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;
    uint64_t* sfull = drain + 1;             // a stage's scale tiles are in tensor memory (even CTA)
    uint64_t* sfdrain = sfull + C::kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
    const int half = (int)(rank & 1u);
    const bool leader = half == 0;

    if (warp == 0) {
        const int G = p.G;
        const int per = (G + 31) / 32;
        const int g0 = lane * per, g1 = min(G, g0 + per);
        const int32_t Mc = (int32_t)p.M;
        int32_t mx = 0;
        for (int g = g0; g < g1; ++g) mx = max(mx, min(max(p.offs[g], 0), Mc));
        int32_t incl = mx;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl = max(incl, o);
        }
        int32_t run = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) run = 0;
        int32_t prev = run, psum = 0, tsum = 0, bad = 0;
        for (int g = g0; g < g1; ++g) {
            const int32_t e = max(prev, min(max(p.offs[g], 0), Mc));
            ends_s[g] = e;
            if ((p.mode == KGROUPED || p.need32) && (e - prev) % 32 != 0) bad = 1;  // token blocks of 32
            psum += ((e - prev + 127) / 128) * 128;
            tsum += (e - prev + 255) / 256;
            prev = e;
        }
        int32_t sincl = psum, tincl = tsum;
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, sincl, d);
            const int32_t q = __shfl_up_sync(0xffffffffu, tincl, d);
            if (lane >= d) {
                sincl += o;
                tincl += q;
            }
        }
        int32_t sexcl = sincl - psum, texcl = tincl - tsum;
        prev = run;
        for (int g = g0; g < g1; ++g) {
            pstart_s[g] = sexcl;
            tstart_s[g] = texcl;
            const int32_t e = ends_s[g];
            sexcl += ((e - prev + 127) / 128) * 128;
            texcl += (e - prev + 255) / 256;
            prev = e;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 31) ptotal_s = sincl;
        if (lane == 0) {
            bad_s = bad;
            abort_s = 0;
            prefetch_tmap(&tmap_a);
            prefetch_tmap(&tmap_b);
            prefetch_tmap(&tmap_sfa);
            prefetch_tmap(&tmap_sfb);
            if (kDualK) {
                prefetch_tmap(&tmap_a2);
                prefetch_tmap(&tmap_b2);
                prefetch_tmap(&tmap_sfa2);
                prefetch_tmap(&tmap_sfb2);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int s = 0; s < C::kStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            mbar_init(tfull, 1);
            mbar_init(tempty, 2 * kPairEpiOf<kSwi>);  // every epilogue warp of both CTAs of the pair
            mbar_init(drain, 1);
            for (int s = 0; s < C::kStages; ++s) mbar_init(&sfull[s], 1);
            mbar_init(sfdrain, 1);
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc_pair(&tmem_base_s, C::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer may signal this CTA's barriers from here on
    tc_fence_after();

    const uint32_t tmem = tmem_base_s;
    volatile int* abort_flag = &abort_s;
    const int64_t ptotal = ptotal_s;
    if (bad_s) {
        if (threadIdx.x == 0 && leader) report(p.dev_status, MXFP8_ERR_OFFSETS);
    } else {
        const int64_t ntb = (p.nb + (kSwi ? 128 : BN) - 1) / (kSwi ? 128 : BN);
        int64_t ntiles;
        if (p.mode == ROWGROUPED) {
            ntiles = (int64_t)tstart_s[p.G - 1] + (ends_s[p.G - 1] - (p.G > 1 ? ends_s[p.G - 2] : 0) + 255) / 256;
            ntiles *= ntb;
        } else {
            ntiles = (int64_t)p.G * ((p.na + 255) / 256) * ntb;
        }
        const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
        // K-grouped (wgrad) tiles cost their group's k-tiles (tokens / 128), so plain round robin leaves
        // the clusters' totals several percent apart.  With few groups the schedule takes the groups
        // largest first and deals each round of ncl tiles out in alternating cluster order (snake):
        // on the 8-expert Scout-like token split, busiest cluster 1.01x the mean instead of 1.04x.
        // Both CTAs of a pair derive the same order; every role walks the same sequence.
        const bool sorted = p.mode == KGROUPED && p.G <= kSortGroups;
        if (sorted) {
            for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
                const int32_t sg = ends_s[g] - (g ? ends_s[g - 1] : 0);
                int r = 0;
                for (int h = 0; h < p.G; ++h) {
                    const int32_t sh = ends_s[h] - (h ? ends_s[h - 1] : 0);
                    r += (sh > sg) || (sh == sg && h < g);
                }
                gorder_s[r] = g;
            }
        }
        __syncthreads();
        auto tile_at = [&](int64_t j) -> int64_t { return j * ncl + ((sorted && (j & 1)) ? ncl - 1 - cid : cid); };

        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t j = 0; j * ncl < ntiles; ++j) {
                const int64_t t = tile_at(j);
                if (t >= ntiles) continue;
                const PairTile ti = pair_tile<kDualK, kSwi>(p, t, half, ends_s, pstart_s, tstart_s, ptotal, gorder_s, sorted);
                bool ok = true;
                for (int kt = 0; kt < ti.k_tiles; ++kt) {
                    if (!mbar_wait_bounded<true>(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = cluster_addr(&full[stage], 0);  // the even CTA's stage barrier
                    if (leader) mbar_arrive_expect_tx(&full[stage], C::kTx);
                    // second operand set of a two-operand tile: the same coordinates in the second maps
                    const bool second = kDualK && kt >= ti.k_tiles / 2;
                    const int kk = second ? kt - ti.k_tiles / 2 : kt;
                    const int32_t kx = (int32_t)(ti.a_x0 + (int64_t)kk * BK);
                    tma_load_2d_pair(smem + stage * C::kABytes, second ? &tmap_a2 : &tmap_a, kx, (int32_t)ti.a_row, fb);
                    // kSwi: the even CTA's B rows are the gate weights', the odd CTA's the up weights'
                    tma_load_2d_pair(smem + C::kOffB + stage * C::kBBytes,
                                     (second || (kSwi && half)) ? &tmap_b2 : &tmap_b, kx, (int32_t)ti.b_row, fb);
                    tma_load_2d_pair(smem + C::kOffSfa + stage * C::kSfaBytes, second ? &tmap_sfa2 : &tmap_sfa, 0,
                                     (int32_t)(2 * (ti.sfa_chunk + kk)), fb);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        tma_load_2d_pair(smem + C::kOffSfb + stage * C::kSfbBytes + 512 * j,
                                         (second || (kSwi && j == 1)) ? &tmap_sfb2 : &tmap_sfb, 0,
                                         (int32_t)(2 * (ti.sfb_chunk[j] + kk)), fb);
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
        } else if (warp == 1 && lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (even CTA only)
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            constexpr uint32_t idesc0 = idesc_mxf8(256, BN, 0, 0);
            for (int64_t j = 0; j * ncl < ntiles && ok; ++j) {
                const int64_t t = tile_at(j);
                if (t >= ntiles) continue;
                const PairTile ti = pair_tile<kDualK, kSwi>(p, t, half, ends_s, pstart_s, tstart_s, ptotal, gorder_s, sorted);
                if (ti.k_tiles == 0) continue;
                if (!mbar_wait_bounded<true>(tempty, acc_phase ^ 1u, p.timeout_ns, abort_flag, p.dev_status)) break;
                tc_fence_after();
                for (int kt = 0; kt < ti.k_tiles; ++kt) {
                    const int cur = stage;
                    if (!mbar_wait_bounded<true>(&full[cur], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded<true>(&sfull[cur], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    const uint32_t sfa_t = tmem + C::kSfCol0 + cur * C::kSfCols;
                    const uint32_t sfb_t = sfa_t + 4;
                    const uint32_t a_s = smem_u32(smem + cur * C::kABytes);
                    const uint32_t b_s = smem_u32(smem + C::kOffB + cur * C::kBBytes);
                    if (kt + 1 < ti.k_tiles || ti.kb_last == BK / 32) {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint64_t ad = smem_desc(a_s + 32 * k, 16, 1024, 2);
                            const uint64_t bd = smem_desc(b_s + 32 * k, 16, 1024, 2);
                            tc_mma_pair_mxf8(tmem, ad, bd, idesc0 | ((uint32_t)k << 4) | ((uint32_t)k << 29), sfa_t,
                                             sfb_t, (kt | k) != 0);
                        }
                    } else {
                        // K-grouped last k-tile: only the group's own 32-token blocks (the box's other
                        // columns hold the next group's tokens, whose codes may be NaN)
#pragma unroll 1
                        for (int k = 0; k < ti.kb_last; ++k) {
                            const uint64_t ad = smem_desc(a_s + 32 * k, 16, 1024, 2);
                            const uint64_t bd = smem_desc(b_s + 32 * k, 16, 1024, 2);
                            tc_mma_pair_mxf8(tmem, ad, bd, idesc0 | ((uint32_t)k << 4) | ((uint32_t)k << 29), sfa_t,
                                             sfb_t, (kt | k) != 0);
                        }
                    }
                    tc_commit_pair(&empty[cur], 0x3);
                }
                if (!ok) break;
                tc_commit_pair(tfull, 0x3);
                acc_phase ^= 1u;
            }
            tc_commit_pair(drain, 0x1);
            volatile int no_abort = 0;
            mbar_wait_bounded<true>(drain, 0, p.timeout_ns, &no_abort, p.dev_status);
        } else if (warp == kPairSfWarpOf<kSwi>) {
            // ------------------------------------------------ scale copies (even CTA only)
            // Each landed stage's scale tiles go to its tensor-memory columns in both CTAs (the
            // cta_group::2 copy), signalled on the even CTA's sfull; the MMA thread waits for it.
            if (lane == 0 && leader) {
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                for (int64_t j = 0; j * ncl < ntiles && ok; ++j) {
                    const int64_t t = tile_at(j);
                    if (t >= ntiles) continue;
                    const PairTile ti = pair_tile<kDualK, kSwi>(p, t, half, ends_s, pstart_s, tstart_s, ptotal, gorder_s, sorted);
                    for (int kt = 0; kt < ti.k_tiles; ++kt) {
                        if (!mbar_wait_bounded<true>(&full[stage], phase, p.timeout_ns, abort_flag, p.dev_status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sfa_t = tmem + C::kSfCol0 + stage * C::kSfCols;
                        tc_cp_pair_32x128b_warpx4(sfa_t, smem_desc(smem_u32(smem + C::kOffSfa + stage * C::kSfaBytes), 0, 128, 0));
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
                            tc_cp_pair_32x128b_warpx4(
                                sfa_t + 4 + 4 * jj,
                                smem_desc(smem_u32(smem + C::kOffSfb + stage * C::kSfbBytes + 512 * jj), 0, 128, 0));
                        tc_commit_pair(&sfull[stage], 0x1);
                        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                    }
                }
                tc_commit_pair(sfdrain, 0x1);
                volatile int no_abort = 0;
                mbar_wait_bounded<true>(sfdrain, 0, p.timeout_ns, &no_abort, p.dev_status);
            }
        } else if (warp >= 2 && kSwi) {
            // ------------------------------------------------ SwiGLU epilogue (both CTAs: own 128 rows)
            const int quarter = warp & 3;
            const int jb = (warp - 2) >> 2;  // 32-column block of h of this warp
            uint8_t* stg = smem + C::kOffStage + (warp - 2) * 2048;  // 2 KB a warp (16 warps: 32 KB)
            const int64_t ct_T = ptotal / 128;
            const uint32_t tempty_leader = cluster_addr(tempty, 0);
            uint32_t acc_phase = 0;
            for (int64_t j = 0; j * ncl < ntiles; ++j) {
                const int64_t t = tile_at(j);
                if (t >= ntiles) continue;
                const PairTile ti = pair_tile<kDualK, kSwi>(p, t, half, ends_s, pstart_s, tstart_s, ptotal, gorder_s, sorted);
                if (!mbar_wait_bounded<true>(tfull, acc_phase, p.timeout_ns, abort_flag, p.dev_status)) break;
                acc_phase ^= 1u;
                tc_fence_after();
                auto release = [&] { if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader); };
                if (ti.valid_rows > 0) {
                    swiglu_tile_epilogue(p, tmem + ((uint32_t)(quarter * 32) << 16) + 32 * jb, quarter, jb, lane, stg,
                                         ti.a_row, ti.valid_rows, ti.valid_cols, ti.prow0, ti.col0, ct_T, release);
                } else {
                    // this CTA's half lies past the group's padded rows: it owns no output, not even padding
                    tc_fence_before();
                    __syncwarp();
                    release();
                }
            }
        } else if (warp >= 2) {
            // ------------------------------------------------ epilogue (both CTAs: own 128 rows)
            // Warp w drains lane quarter w % 4 (the quarter its tensor-memory access is bound to) and
            // column half (w - 2) / 4 of the accumulator.
            constexpr int kHalfCols = BN / 2;
            const int quarter = warp & 3;
            const int c_base = ((warp - 2) >> 2) * kHalfCols;
            uint8_t* stg = smem + C::kOffStage + (warp - 2) * 1024;  // 32 rows x 32 bytes
            const uint32_t tempty_leader = cluster_addr(tempty, 0);
            uint32_t acc_phase = 0;
            for (int64_t j = 0; j * ncl < ntiles; ++j) {
                const int64_t t = tile_at(j);
                if (t >= ntiles) continue;
                const PairTile ti = pair_tile<kDualK, kSwi>(p, t, half, ends_s, pstart_s, tstart_s, ptotal, gorder_s, sorted);
                __nv_bfloat16* wout = ti.out + (int64_t)(quarter * 32) * ti.ldo + c_base;
                const int vrows = ti.valid_rows - quarter * 32;
                const int vcols = ti.valid_cols - c_base;  // columns of this warp's half inside the output
                if (ti.k_tiles == 0) {
                    for (int rl = 0; rl < 32; ++rl)
                        if (rl < vrows)
                            for (int c = lane * 8; c < kHalfCols && c < vcols; c += 256)
                                *reinterpret_cast<uint4*>(wout + (int64_t)rl * ti.ldo + c) = make_uint4(0, 0, 0, 0);
                    continue;
                }
                if (!mbar_wait_bounded<true>(tfull, acc_phase, p.timeout_ns, abort_flag, p.dev_status)) break;
                acc_phase ^= 1u;
                tc_fence_after();
                uint32_t packed[kHalfCols / 2];
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + c_base;
#pragma unroll
                for (int c = 0; c < kHalfCols; c += 64) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(taddr + c, v0);
                    tmem_ld_32x32b_x32(taddr + c + 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        packed[c / 2 + i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
                        packed[c / 2 + 16 + i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
                // 16 columns a pass: lane = row writes its two 16-byte pieces (the piece order flips every
                // 4 rows, so each 8-lane phase covers all 32 banks), then two lanes a row store whole
                // 32-byte sectors of 16 rows per instruction.
#pragma unroll
                for (int ch = 0; ch < kHalfCols / 16; ++ch) {
                    if (ch * 16 >= vcols) break;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        st_shared_v4(stg + lane * 32 + ((j ^ ((lane >> 2) & 1)) * 16),
                                     make_uint4(packed[ch * 8 + 4 * j], packed[ch * 8 + 4 * j + 1],
                                                packed[ch * 8 + 4 * j + 2], packed[ch * 8 + 4 * j + 3]));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int rl = (lane >> 1) + 16 * i, piece = lane & 1;
                        const uint4 val = ld_shared_v4(stg + rl * 32 + ((piece ^ ((rl >> 2) & 1)) * 16));
                        if (rl < vrows && ch * 16 + piece * 8 < vcols)
                            *reinterpret_cast<uint4*>(wout + (int64_t)rl * ti.ldo + ch * 16 + piece * 8) = val;
                    }
                    __syncwarp();
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA frees tensor memory or exits while the pair still works
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
// 2D uint8 tensor [rows][cols] (row pitch = cols bytes), box = box_rows x 128 bytes, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    host::EncodeTiledFn fn = host::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// b2: SwiGLU variant: the up weights, same shape as b (each B map then has 128-row boxes); two-operand
// dgrad (kDualK): the second B operand.  a2: two-operand dgrad only, the second A operand.
template <int BN, bool kDualK = false>
static mxfp8_status_t launch_gemm(const void* a, int64_t a_rows, int64_t a_cols, const void* b, int64_t b_rows,
                                  int64_t b_cols, GemmParams& p, int64_t tiles_bound, cudaStream_t st,
                                  const void* b2 = nullptr, const void* a2 = nullptr) {
    using C = Cfg<BN>;
    CUtensorMap ma, mb, mb2, ma2;
    if (!make_map(&ma, a, a_rows, a_cols, BM) || !make_map(&mb, b, b_rows, b_cols, BN)) return MXFP8_ERR_DRIVER;
    if (kDualK ? !make_map(&mb2, b2, b_rows, b_cols, BN) : false) return MXFP8_ERR_DRIVER;
    if (kDualK ? !make_map(&ma2, a2, a_rows, a_cols, BM) : false) return MXFP8_ERR_DRIVER;
    if (!kDualK) {
        mb2 = mb;
        ma2 = ma;
    }
    static std::atomic<int> attr_set[host::kMaxDevices];
    if (!host::ensure_smem(reinterpret_cast<const void*>(grouped_mm_kernel<BN, kDualK>), C::kSmem, attr_set))
        return MXFP8_ERR_LAUNCH;
    const int grid = (int)max64(1, min64(tiles_bound, host::num_sms()));
    grouped_mm_kernel<BN, kDualK><<<grid, kThreads, C::kSmem, st>>>(ma, mb, mb2, ma2, p);
    return host::last_launch_status();
}

static uint64_t default_timeout_ns() { return 2000000000ull; }

// Kernel choice: the CTA-pair kernel wherever the output is at least 256 wide (fwd, dgrad and
// wgrad alike); the single-CTA kernel for narrower outputs and for the SwiGLU and two-operand
// variants.  Measured with the scale copies on their own warp (TFLOP/s, single-CTA with 256-wide
// tiles / pair): forward of the 8-expert Scout-like workload 2533 / 2782, of the 2-expert SwiGLU
// shapes 2694 / 3070 (N=16384, K=5120) and 2725 / 3057 (N=5120, K=8192).  Padding ragged token
// groups to 256 rows instead of 128 costs less than the pair's halved B traffic per CTA saves.

// A scale buffer as [bytes/256][256] uint8, 2 x 256 B boxes (= one 512-byte scale tile).
static bool make_scale_map(CUtensorMap* m, const void* base, int64_t bytes) {
    host::EncodeTiledFn fn = host::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {256, (cuuint64_t)(bytes / 256)};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, 2};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kDualK, bool kSwi>
static int max_pair_clusters(const cudaLaunchConfig_t& cfg) {
    static std::atomic<int> cache[host::kMaxDevices];
    const int d = host::current_device();
    if (d < 0 || d >= host::kMaxDevices) return 1;
    int v = cache[d].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveClusters(&v, grouped_mm_pair_kernel<kDualK, kSwi>, &cfg) != cudaSuccess || v <= 0)
            v = host::num_sms() / 2;
        cudaGetLastError();
        cache[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

// sfa_bytes / sfb_bytes: extents of the scale buffers the maps may address (the ABI's sizing bounds).
// kDualK: a2 / b2 (same shapes as a / b) with scales p.sfa2 / p.sfb2 are the second operand set.
// kSwi: b2 with scales p.sfb2 are the up weights (b the gate weights).
template <bool kDualK = false, bool kSwi = false>
static mxfp8_status_t launch_pair(const void* a, int64_t a_rows, int64_t a_cols, const void* b, int64_t b_rows,
                                  int64_t b_cols, int64_t sfa_bytes, int64_t sfb_bytes, GemmParams& p,
                                  int64_t pair_tiles_bound, cudaStream_t st, const void* a2 = nullptr,
                                  const void* b2 = nullptr) {
    using C = CfgPair<kSwi>;
    CUtensorMap ma, mb, msa, msb, ma2, mb2, msa2, msb2;
    if (!make_map(&ma, a, a_rows, a_cols, BM) || !make_map(&mb, b, b_rows, b_cols, 128) ||
        !make_scale_map(&msa, p.sfa, sfa_bytes) || !make_scale_map(&msb, p.sfb, sfb_bytes))
        return MXFP8_ERR_DRIVER;
    if (kDualK) {
        if (!make_map(&ma2, a2, a_rows, a_cols, BM) || !make_map(&mb2, b2, b_rows, b_cols, 128) ||
            !make_scale_map(&msa2, p.sfa2, sfa_bytes) || !make_scale_map(&msb2, p.sfb2, sfb_bytes))
            return MXFP8_ERR_DRIVER;
    } else if (kSwi) {
        if (!make_map(&mb2, b2, b_rows, b_cols, 128) || !make_scale_map(&msb2, p.sfb2, sfb_bytes))
            return MXFP8_ERR_DRIVER;
        ma2 = ma;
        msa2 = msa;
    } else {
        ma2 = ma;
        mb2 = mb;
        msa2 = msa;
        msb2 = msb;
    }
    static std::atomic<int> attr_set[host::kMaxDevices];
    if (!host::ensure_smem(reinterpret_cast<const void*>(grouped_mm_pair_kernel<kDualK, kSwi>), C::kSmem, attr_set))
        return MXFP8_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreadsPairOf<kSwi>);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * host::num_sms() / 2);
    const int clusters = (int)max64(1, min64(pair_tiles_bound, max_pair_clusters<kDualK, kSwi>(cfg)));
    cfg.gridDim = dim3(2 * clusters);
    if (cudaLaunchKernelEx(&cfg, grouped_mm_pair_kernel<kDualK, kSwi>, ma, mb, msa, msb, ma2, mb2, msa2, msb2, p) !=
        cudaSuccess)
        return MXFP8_ERR_LAUNCH;
    return host::last_launch_status();
}

// fwd and dgrad: token operand tok_q [M, Kc], expert operand ex_q [G, Nb, Kc].  With tok2_q (two-operand
// dgrad) a second pair tok2 / ex2 of the same shapes is contracted into the same output.
static mxfp8_status_t rowgrouped(const void* tok_q, const void* tok_s, const void* ex_q, const void* ex_s,
                                 const int32_t* offs, int32_t G, int64_t M, int64_t Nb, int64_t Kc, void* out,
                                 int32_t* dev_status, cudaStream_t st, const void* tok2_q = nullptr,
                                 const void* tok2_s = nullptr, const void* ex2_q = nullptr, const void* ex2_s = nullptr) {
    if (!tok_q || !tok_s || !ex_q || !ex_s || !offs || !out) return MXFP8_ERR_NULL;
    const bool dual = tok2_q != nullptr;
    if (dual && (!tok2_s || !ex2_q || !ex2_s)) return MXFP8_ERR_NULL;
    if (dual && (!host::aligned16(tok2_q) || !host::aligned16(tok2_s) || !host::aligned16(ex2_q) ||
                 !host::aligned16(ex2_s)))
        return MXFP8_ERR_ALIGN;
    if (G < 1 || G > MXFP8_MAX_GROUPS || M < 0 || Nb <= 0 || Kc <= 0 || M > INT32_MAX || (int64_t)G * Nb > INT32_MAX)
        return MXFP8_ERR_SHAPE;
    if (Kc % 32 || Nb % 32) return MXFP8_ERR_ALIGN;
    if (!host::aligned16(tok_q) || !host::aligned16(tok_s) || !host::aligned16(ex_q) || !host::aligned16(ex_s) ||
        !host::aligned16(out))
        return MXFP8_ERR_ALIGN;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    if (M == 0) return MXFP8_OK;
    GemmParams p{};
    p.sfa = static_cast<const uint8_t*>(tok_s);
    p.sfb = static_cast<const uint8_t*>(ex_s);
    p.sfa_ct = (Kc + 127) / 128;
    p.sfb_ct = (Kc + 127) / 128;
    p.sfb_estride = ((Nb + 127) / 128) * 128 * p.sfb_ct * 4;
    p.nb = Nb;
    p.kc = Kc;
    p.offs = offs;
    p.G = G;
    p.M = M;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.ldo = Nb;
    p.mode = ROWGROUPED;
    p.dev_status = dev_status;
    p.timeout_ns = default_timeout_ns();
    if (dual) {
        p.sfa2 = static_cast<const uint8_t*>(tok2_s);
        p.sfb2 = static_cast<const uint8_t*>(ex2_s);
        if (Nb >= 256) {
            const int64_t bound = ((M + 255) / 256 + G) * ((Nb + 255) / 256);
            const int64_t sfa_bytes = ((M + 127) / 128 + G) * 128 * p.sfa_ct * 4;
            return launch_pair<true>(tok_q, M, Kc, ex_q, (int64_t)G * Nb, Kc, sfa_bytes, (int64_t)G * p.sfb_estride, p,
                                     bound, st, tok2_q, ex2_q);
        }
        const int64_t bound = ((M + BM - 1) / BM + G) * ((Nb + 127) / 128);
        return launch_gemm<128, true>(tok_q, M, Kc, ex_q, (int64_t)G * Nb, Kc, p, bound, st, ex2_q, tok2_q);
    }
    if (Nb >= 256) {
        const int64_t bound = ((M + 255) / 256 + G) * ((Nb + 255) / 256);
        const int64_t sfa_bytes = ((M + 127) / 128 + G) * 128 * p.sfa_ct * 4;
        return launch_pair(tok_q, M, Kc, ex_q, (int64_t)G * Nb, Kc, sfa_bytes, (int64_t)G * p.sfb_estride, p, bound,
                           st);
    }
    const int64_t bound = ((M + BM - 1) / BM + G) * ((Nb + 127) / 128);
    return launch_gemm<128>(tok_q, M, Kc, ex_q, (int64_t)G * Nb, Kc, p, bound, st);
}

}  // namespace mx

using namespace mx;

extern "C" mxfp8_status_t mxfp8_grouped_mm_fwd(const void* a_q, const void* a_s, const void* w_q, const void* w_s,
                                               const int32_t* offs, int32_t G, int64_t M, int64_t N, int64_t K,
                                               void* out_bf16, int32_t* dev_status, mxfp8_stream_t stream) {
    return rowgrouped(a_q, a_s, w_q, w_s, offs, G, M, N, K, out_bf16, dev_status,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" mxfp8_status_t mxfp8_grouped_mm_dgrad(const void* dout_q, const void* dout_s, const void* wt_q,
                                                 const void* wt_s, const int32_t* offs, int32_t G, int64_t M,
                                                 int64_t N, int64_t K, void* da_bf16, int32_t* dev_status,
                                                 mxfp8_stream_t stream) {
    return rowgrouped(dout_q, dout_s, wt_q, wt_s, offs, G, M, K, N, da_bf16, dev_status,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" mxfp8_status_t mxfp8_grouped_mm_wgrad(const void* doutT_q, const void* doutT_s, const void* aT_q,
                                                 const void* aT_s, const int32_t* offs, int32_t G, int64_t M,
                                                 int64_t N, int64_t K, void* dw_bf16, int32_t* dev_status,
                                                 mxfp8_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!doutT_q || !doutT_s || !aT_q || !aT_s || !offs || !dw_bf16) return MXFP8_ERR_NULL;
    if (G < 1 || G > MXFP8_MAX_GROUPS || M < 0 || N <= 0 || K <= 0 || M > INT32_MAX || N > INT32_MAX ||
        K > INT32_MAX)
        return MXFP8_ERR_SHAPE;
    if (N % 32 || K % 32 || M % 32) return MXFP8_ERR_ALIGN;
    if (!host::aligned16(doutT_q) || !host::aligned16(doutT_s) || !host::aligned16(aT_q) || !host::aligned16(aT_s) ||
        !host::aligned16(dw_bf16))
        return MXFP8_ERR_ALIGN;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    if (M == 0) {
        return cudaMemsetAsync(dw_bf16, 0, (size_t)G * N * K * 2, st) == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
    }
    GemmParams p{};
    p.sfa = static_cast<const uint8_t*>(doutT_s);
    p.sfb = static_cast<const uint8_t*>(aT_s);
    p.na = N;
    p.nb = K;
    p.offs = offs;
    p.G = G;
    p.M = M;
    p.out = static_cast<__nv_bfloat16*>(dw_bf16);
    p.mode = KGROUPED;
    p.need32 = 1;
    p.dev_status = dev_status;
    p.timeout_ns = default_timeout_ns();
    if (K >= 256) {
        const int64_t bound = (int64_t)G * ((N + 255) / 256) * ((K + 255) / 256);
        const int64_t tiles_m = (M + 127) / 128 + G;
        return launch_pair(doutT_q, N, M, aT_q, K, M, ((N + 127) / 128) * 128 * tiles_m * 4,
                           ((K + 127) / 128) * 128 * tiles_m * 4, p, bound, st);
    }
    const int64_t bound = (int64_t)G * ((N + BM - 1) / BM) * ((K + 127) / 128);
    return launch_gemm<128>(doutT_q, N, M, aT_q, K, M, p, bound, st);
}

extern "C" mxfp8_status_t mxfp8_grouped_mm_swiglu_fwd(const void* x_q, const void* x_s, const void* wg_q,
                                                      const void* wg_s, const void* wu_q, const void* wu_s,
                                                      const int32_t* offs, int32_t G, int64_t M, int64_t H, int64_t D,
                                                      void* h1_bf16, void* h3_bf16, void* h_q, void* h_s, void* hT_q,
                                                      void* hT_s, int32_t* dev_status, mxfp8_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!x_q || !x_s || !wg_q || !wg_s || !wu_q || !wu_s || !offs || !h1_bf16 || !h3_bf16 || !h_q || !h_s)
        return MXFP8_ERR_NULL;
    if ((hT_q == nullptr) != (hT_s == nullptr)) return MXFP8_ERR_NULL;
    if (G < 1 || G > MXFP8_MAX_GROUPS || M < 0 || H <= 0 || D <= 0 || M > INT32_MAX || (int64_t)G * H > INT32_MAX ||
        D > INT32_MAX)
        return MXFP8_ERR_SHAPE;
    if (H % 32 || D % 32 || (hT_q && M % 32)) return MXFP8_ERR_ALIGN;
    const void* ptrs[] = {x_q, x_s, wg_q, wg_s, wu_q, wu_s, h1_bf16, h3_bf16, h_q, h_s};
    for (const void* q : ptrs)
        if (!host::aligned16(q)) return MXFP8_ERR_ALIGN;
    if (hT_q && (!host::aligned16(hT_q) || !host::aligned16(hT_s))) return MXFP8_ERR_ALIGN;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    if (M == 0) return MXFP8_OK;
    GemmParams p{};
    p.sfa = static_cast<const uint8_t*>(x_s);
    p.sfb = static_cast<const uint8_t*>(wg_s);
    p.sfb2 = static_cast<const uint8_t*>(wu_s);
    p.sfa_ct = (D + 127) / 128;
    p.sfb_ct = (D + 127) / 128;
    p.sfb_estride = ((H + 127) / 128) * 128 * p.sfb_ct * 4;
    p.nb = H;
    p.kc = D;
    p.offs = offs;
    p.G = G;
    p.M = M;
    p.out = static_cast<__nv_bfloat16*>(h1_bf16);
    p.out2 = static_cast<__nv_bfloat16*>(h3_bf16);
    p.ldo = H;
    p.hq = static_cast<uint8_t*>(h_q);
    p.hs = static_cast<uint8_t*>(h_s);
    p.hs_ct = (H + 127) / 128;
    p.hTq = static_cast<uint8_t*>(hT_q);
    p.hTs = static_cast<uint8_t*>(hT_s);
    p.mode = ROWGROUPED;
    p.need32 = hT_q != nullptr;
    p.dev_status = dev_status;
    p.timeout_ns = default_timeout_ns();
    const int64_t bound = ((M + 255) / 256 + G) * ((H + 127) / 128);
    const int64_t sfa_bytes = ((M + 127) / 128 + G) * 128 * p.sfa_ct * 4;
    return launch_pair<false, true>(x_q, M, D, wg_q, (int64_t)G * H, D, sfa_bytes, (int64_t)G * p.sfb_estride, p, bound,
                                    st, nullptr, wu_q);
}

extern "C" mxfp8_status_t mxfp8_grouped_mm_dgrad2(const void* dout1_q, const void* dout1_s, const void* wt1_q,
                                                  const void* wt1_s, const void* dout2_q, const void* dout2_s,
                                                  const void* wt2_q, const void* wt2_s, const int32_t* offs, int32_t G,
                                                  int64_t M, int64_t N, int64_t K, void* da_bf16, int32_t* dev_status,
                                                  mxfp8_stream_t stream) {
    if (!dout2_q) return MXFP8_ERR_NULL;
    return rowgrouped(dout1_q, dout1_s, wt1_q, wt1_s, offs, G, M, K, N, da_bf16, dev_status,
                      reinterpret_cast<cudaStream_t>(stream), dout2_q, dout2_s, wt2_q, wt2_s);
}
