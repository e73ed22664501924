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
// (2 shuffles); amax is an integer max over bf16 magnitude bits (two per
// max.u16x2), the scale byte comes from the exponent field, the elements are
// multiplied by 2^(127-s) exactly in fp32 and converted with
// cvt.rn.satfinite.e4m3x2.  Stores are 8-byte vectors.  The grid is persistent
// (a multiple of the SM count), striding over tiles.

#include "common.cuh"
#include "host_common.h"

namespace mx {

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
};

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

__device__ __forceinline__ uint32_t shfl_xor_max16x2(uint32_t v, int m) {
    return vmax_u16x2(v, __shfl_xor_sync(0xffffffffu, v, m));
}

// Eight bf16 (4 packed words) times f -> eight E4M3 codes (little-endian in a u64).
__device__ __forceinline__ uint2 quant8(const uint32_t (&w)[4], float f) {
    uint2 r;
    r.x = cvt_e4m3x2(bf16lo(w[0]) * f, bf16hi(w[0]) * f) | (cvt_e4m3x2(bf16lo(w[1]) * f, bf16hi(w[1]) * f) << 16);
    r.y = cvt_e4m3x2(bf16lo(w[2]) * f, bf16hi(w[2]) * f) | (cvt_e4m3x2(bf16lo(w[3]) * f, bf16hi(w[3]) * f) << 16);
    return r;
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

template <unsigned DIRS>
__global__ void __launch_bounds__(256) quant_tile_kernel(QParams p) {
    constexpr bool kRow = (DIRS & MXFP8_ROW) != 0;
    constexpr bool kCol = (DIRS & MXFP8_COL) != 0;
    constexpr bool kB32 = (DIRS & MXFP8_BLOCK32X32) != 0;
    __shared__ int32_t ends_s[kMaxGroups];
    __shared__ int32_t pstart_s[kMaxGroups];
    __shared__ int32_t ptotal_s;

    const bool grouped = p.offs != nullptr && p.G > 1;
    if (grouped && p.blocked) {
        if (threadIdx.x < 32) build_group_table(p.offs, p.G, p.R, ends_s, pstart_s, &ptotal_s);
        __syncthreads();
    }
    const int64_t R = p.R, C = p.C;
    const int64_t Cb = C / kBlk;
    const int64_t ct_row = (C + 127) / 128;                                  // row-scale column tiles
    const int64_t ct_col = grouped ? (int64_t)ptotal_s / 128 : (R + 127) / 128;  // col-scale column tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wi = warp >> 1, wj = warp & 1;
    const int li = lane >> 3, lj = lane & 7;

    for (int64_t t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const int64_t per_b = p.tiles_r * p.tiles_c;
        const int64_t b = t / per_b;
        const int64_t rem = t - b * per_b;
        const int64_t tr = rem / p.tiles_c, tc = rem - tr * p.tiles_c;
        const int64_t row0 = tr * 128 + wi * 32, col0 = tc * 128 + wj * 64;
        if (row0 >= R || col0 >= C) continue;  // warp-uniform

        const uint16_t* xb = p.x + b * R * C;
        const int64_t c8 = col0 + 8 * lj;  // first column of this lane
        const bool cval = c8 < C;          // C % 32 == 0: 8-column chunks are all-in or all-out
        uint32_t v[8][4];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
            const int64_t row = row0 + 8 * li + rr;
            uint4 u = make_uint4(0, 0, 0, 0);
            if (cval && row < R) u = __ldg(reinterpret_cast<const uint4*>(xb + row * C + c8));
            v[rr][0] = u.x; v[rr][1] = u.y; v[rr][2] = u.z; v[rr][3] = u.w;
        }

        if constexpr (kRow || kB32) {
            uint32_t rmax[8];  // per-row amax over this lane's 8 columns (16-bit)
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                uint32_t m = vmax_u16x2(vmax_u16x2(v[rr][0] & 0x7FFF7FFFu, v[rr][1] & 0x7FFF7FFFu),
                                        vmax_u16x2(v[rr][2] & 0x7FFF7FFFu, v[rr][3] & 0x7FFF7FFFu));
                rmax[rr] = max(m & 0xFFFFu, m >> 16);
            }
            uint32_t s8[8];
            if constexpr (kB32) {
                // one amax over the 32x32 block: 8 rows here, 4 lanes across (lj bits 0-1)
                // and 4 lanes down (li, lane bits 3-4)
                uint32_t m = 0;
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) m = max(m, rmax[rr]);
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
                const uint32_t s = e8m0_from_absbits(m);
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) s8[rr] = s;
            } else {
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    uint32_t m = rmax[rr];
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    s8[rr] = e8m0_from_absbits(m);
                }
            }
            uint8_t* qb = p.q_row + b * R * C;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int64_t row = row0 + 8 * li + rr;
                uint2 q = quant8(v[rr], inv_scale_from_e8m0(s8[rr]));
                if (s8[rr] == 0xFFu) { uint2 sg = signs8(v[rr]); q.x = 0x7F7F7F7Fu | sg.x; q.y = 0x7F7F7F7Fu | sg.y; }
                if (cval && row < R) *reinterpret_cast<uint2*>(qb + row * C + c8) = q;
            }
            // scales: one lane per 32-column block writes
            if (cval && (lj & 3) == 0) {
                uint8_t* sb = p.s_row + b * p.s_row_bstride;
                const int64_t cb = c8 / kBlk;
                if constexpr (kB32) {
                    if (li == 0) sb[(row0 / kBlk) * Cb + cb] = (uint8_t)s8[0];
                } else {
                    int g = 0;
                    if (grouped && p.blocked) g = find_group(ends_s, p.G, row0 + 8 * li);
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int64_t row = row0 + 8 * li + rr;
                        if (row >= R) break;
                        if (!p.blocked) {
                            sb[row * Cb + cb] = (uint8_t)s8[rr];
                        } else if (!grouped) {
                            sb[blocked_off(row, cb, ct_row)] = (uint8_t)s8[rr];
                        } else {
                            while (g < p.G && row >= ends_s[g]) ++g;
                            if (g < p.G) {
                                const int64_t start = g ? ends_s[g - 1] : 0;
                                sb[blocked_off(pstart_s[g] + (row - start), cb, ct_row)] = (uint8_t)s8[rr];
                            }
                        }
                    }
                }
            }
        }

        if constexpr (kCol) {
            // column amax over 32 rows: 8 here (packed pairs of columns), then lanes li = 0..3
            uint32_t cm[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t m = v[0][k] & 0x7FFF7FFFu;
#pragma unroll
                for (int rr = 1; rr < 8; ++rr) m = vmax_u16x2(m, v[rr][k] & 0x7FFF7FFFu);
                m = shfl_xor_max16x2(m, 8);
                m = shfl_xor_max16x2(m, 16);
                cm[k] = m;
            }
            uint8_t* qb = p.q_col + b * R * C;
            uint32_t sc[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sc[2 * k] = e8m0_from_absbits(cm[k] & 0xFFFFu);
                sc[2 * k + 1] = e8m0_from_absbits(cm[k] >> 16);
            }
            if (cval) {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const float f = inv_scale_from_e8m0(sc[cc]);
                    const int k = cc >> 1;
                    uint32_t w[4];
#pragma unroll
                    for (int rr = 0; rr < 8; rr += 2) {
                        const float a = (cc & 1) ? bf16hi(v[rr][k]) : bf16lo(v[rr][k]);
                        const float c = (cc & 1) ? bf16hi(v[rr + 1][k]) : bf16lo(v[rr + 1][k]);
                        w[rr >> 1] = cvt_e4m3x2(a * f, c * f);
                    }
                    uint2 q;
                    q.x = w[0] | (w[1] << 16);
                    q.y = w[2] | (w[3] << 16);
                    if (sc[cc] == 0xFFu) {
                        uint32_t sg[4];
#pragma unroll
                        for (int rr = 0; rr < 8; rr += 2) {
                            const uint32_t a = (cc & 1) ? (v[rr][k] >> 31) : ((v[rr][k] >> 15) & 1u);
                            const uint32_t c = (cc & 1) ? (v[rr + 1][k] >> 31) : ((v[rr + 1][k] >> 15) & 1u);
                            sg[rr >> 1] = (a << 7) | (c << 15);
                        }
                        q.x = 0x7F7F7F7Fu | sg[0] | (sg[1] << 16);
                        q.y = 0x7F7F7F7Fu | sg[2] | (sg[3] << 16);
                    }
                    *reinterpret_cast<uint2*>(qb + (c8 + cc) * R + row0 + 8 * li) = q;
                }
                if (li == 0) {
                    uint8_t* sb = p.s_col + b * p.s_col_bstride;
                    const int64_t rb = row0 / kBlk;
                    int64_t pc = rb;
                    bool ok = true;
                    if (p.blocked && grouped) {
                        const int g = find_group(ends_s, p.G, row0);
                        ok = g < p.G;
                        if (ok) pc = pstart_s[g] / kBlk + (row0 - (g ? ends_s[g - 1] : 0)) / kBlk;
                    }
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int64_t c = c8 + cc;
                        if (!p.blocked) sb[c * (R / kBlk) + rb] = (uint8_t)sc[cc];
                        else if (ok) sb[blocked_off(c, pc, ct_col)] = (uint8_t)sc[cc];
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------- padding of blocked layouts
// Row-grouped blocked scales of a [R x Cb] scale matrix: zero every byte that
// is not a scale -- the padding rows of each group (up to its next multiple of
// 128) and the block-columns Cb..4*ct-1.  One thread per padded row.
__global__ void __launch_bounds__(256) pad_rowgroups_kernel(uint8_t* s, int64_t bstride, const int32_t* offs,
                                                            int32_t G, int64_t R, int64_t Cb, int64_t rows_bound) {
    __shared__ int32_t ends_s[kMaxGroups];
    __shared__ int32_t pstart_s[kMaxGroups];
    __shared__ int32_t ptotal_s;
    const bool grouped = offs != nullptr && G > 1;
    if (grouped) {
        if (threadIdx.x < 32) build_group_table(offs, G, R, ends_s, pstart_s, &ptotal_s);
        __syncthreads();
    }
    const int64_t ct = (Cb + 3) / 4;
    const int64_t ptotal = grouped ? ptotal_s : ((R + 127) / 128) * 128;
    uint8_t* sb = s + blockIdx.y * bstride;
    for (int64_t pr = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; pr < min(ptotal, rows_bound);
         pr += (int64_t)gridDim.x * blockDim.x) {
        int64_t local = pr, size = R;
        if (grouped) {
            // group whose padded range holds pr: last g with pstart_s[g] <= pr and a non-empty range
            int lo = 0, hi = G;
            while (lo < hi) {
                int mid = (lo + hi) >> 1;
                if (pstart_s[mid] <= pr) lo = mid + 1;
                else hi = mid;
            }
            int g = lo - 1;
            local = pr - pstart_s[g];
            size = ends_s[g] - (g ? ends_s[g - 1] : 0);
        }
        const int64_t base = (pr >> 7) * ct * 512 + (pr & 31) * 16 + ((pr >> 5) & 3) * 4;
        if (local >= size) {
            for (int64_t t = 0; t < ct; ++t) *reinterpret_cast<uint32_t*>(sb + base + t * 512) = 0u;
        } else if (Cb & 3) {
            for (int64_t c = Cb; c < ct * 4; ++c) sb[base + (ct - 1) * 512 + (c & 3)] = 0;
        }
    }
}

// Column-grouped blocked scales of a [Rs x (tokens/32)] scale matrix (Rs = the
// rows of the transposed operand): zero the padding block-columns of each group
// and the padding rows Rs..ceil(Rs/128)*128.  One thread per (row, column tile).
__global__ void __launch_bounds__(256) pad_colgroups_kernel(uint8_t* s, int64_t bstride, const int32_t* offs,
                                                            int32_t G, int64_t M, int64_t Rs, int64_t tiles_bound) {
    __shared__ int32_t ends_s[kMaxGroups];
    __shared__ int32_t pstart_s[kMaxGroups];
    __shared__ int32_t ptotal_s;
    const bool grouped = offs != nullptr && G > 1;
    if (grouped) {
        if (threadIdx.x < 32) build_group_table(offs, G, M, ends_s, pstart_s, &ptotal_s);
        __syncthreads();
    }
    const int64_t ct = grouped ? ptotal_s / 128 : (M + 127) / 128;
    const int64_t rows_p = ((Rs + 127) / 128) * 128;
    uint8_t* sb = s + blockIdx.y * bstride;
    const int64_t n = rows_p * min(ct, tiles_bound);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / ct, t = idx - r * ct;
        const int64_t base = (r >> 7) * ct * 512 + t * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        if (r >= Rs) {
            *reinterpret_cast<uint32_t*>(sb + base) = 0u;
            continue;
        }
        // the group owning column tile t, and how many of its 4 block-columns hold scales
        int64_t valid;
        if (grouped) {
            int lo = 0, hi = G;
            while (lo < hi) {
                int mid = (lo + hi) >> 1;
                if (pstart_s[mid] <= t * 128) lo = mid + 1;
                else hi = mid;
            }
            const int g = lo - 1;
            const int64_t size = ends_s[g] - (g ? ends_s[g - 1] : 0);
            valid = size / kBlk - (t * 128 - pstart_s[g]) / kBlk;
        } else {
            valid = M / kBlk - t * 4;
        }
        for (int64_t c = valid > 0 ? valid : 0; c < 4; ++c) sb[base + c] = 0;
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
static mxfp8_status_t launch_tiles(unsigned dirs, const QParams& p, cudaStream_t st) {
    if (p.ntiles == 0) return MXFP8_OK;
    const int sms = host::num_sms();
    const int64_t grid = std::min<int64_t>(p.ntiles, (int64_t)sms * 8);
    switch (dirs) {
        case MXFP8_ROW: quant_tile_kernel<MXFP8_ROW><<<grid, 256, 0, st>>>(p); break;
        case MXFP8_COL: quant_tile_kernel<MXFP8_COL><<<grid, 256, 0, st>>>(p); break;
        case MXFP8_ROW | MXFP8_COL: quant_tile_kernel<MXFP8_ROW | MXFP8_COL><<<grid, 256, 0, st>>>(p); break;
        case MXFP8_BLOCK32X32: quant_tile_kernel<MXFP8_BLOCK32X32><<<grid, 256, 0, st>>>(p); break;
        default: return MXFP8_ERR_LAYOUT;
    }
    return host::last_launch_status();
}

static mxfp8_status_t pad_rows(uint8_t* s, int64_t bstride, int32_t batch, const int32_t* offs, int32_t G, int64_t R,
                               int64_t Cb, cudaStream_t st) {
    const int64_t bound = ((R + 127) / 128 + (offs && G > 1 ? G : 1)) * 128;
    const int64_t blocks = std::min<int64_t>((bound + 255) / 256, (int64_t)host::num_sms() * 4);
    pad_rowgroups_kernel<<<dim3((unsigned)blocks, (unsigned)batch), 256, 0, st>>>(s, bstride, offs, G, R, Cb, bound);
    return host::last_launch_status();
}

static mxfp8_status_t pad_cols(uint8_t* s, int64_t bstride, int32_t batch, const int32_t* offs, int32_t G, int64_t M,
                               int64_t Rs, cudaStream_t st) {
    const int64_t tb = (M + 127) / 128 + (offs && G > 1 ? G : 1);
    const int64_t n = ((Rs + 127) / 128) * 128 * tb;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)host::num_sms() * 4);
    pad_colgroups_kernel<<<dim3((unsigned)blocks, (unsigned)batch), 256, 0, st>>>(s, bstride, offs, G, M, Rs, tb);
    return host::last_launch_status();
}

}  // namespace mx

using namespace mx;

extern "C" mxfp8_status_t mxfp8_quantize_2d(const void* x_bf16, int64_t M, int64_t K, unsigned dirs,
                                            int scale_layout, const int32_t* offs, int32_t G, void* q_row,
                                            void* s_row, void* q_col, void* s_col, int32_t* dev_status,
                                            mxfp8_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (M < 0 || K <= 0 || G < 0 || G > MXFP8_MAX_GROUPS || M > INT32_MAX) return MXFP8_ERR_SHAPE;
    if (K % 32) return MXFP8_ERR_ALIGN;
    if (scale_layout != MXFP8_SCALES_COMPACT && scale_layout != MXFP8_SCALES_BLOCKED) return MXFP8_ERR_LAYOUT;
    const bool row = dirs & MXFP8_ROW, col = dirs & MXFP8_COL, b32 = dirs & MXFP8_BLOCK32X32;
    if (dirs == 0 || (dirs & ~7u) || (b32 && (row || col))) return MXFP8_ERR_LAYOUT;
    if (b32 && scale_layout != MXFP8_SCALES_COMPACT) return MXFP8_ERR_LAYOUT;
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
    if (mxfp8_status_t s = launch_tiles(dirs, p, st); s != MXFP8_OK) return s;
    if (blocked && row) {
        if (mxfp8_status_t s = pad_rows(p.s_row, 0, 1, p.offs, p.G, M, K / 32, st); s != MXFP8_OK) return s;
    }
    if (blocked && col) {
        if (mxfp8_status_t s = pad_cols(p.s_col, 0, 1, p.offs, p.G, M, K, st); s != MXFP8_OK) return s;
    }
    return MXFP8_OK;
}

extern "C" mxfp8_status_t mxfp8_quantize_3d_experts(const void* w_bf16, int32_t G, int64_t N, int64_t K, unsigned dirs,
                                                    int scale_layout, void* q, void* s, void* qT, void* sT,
                                                    int32_t* dev_status, mxfp8_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (G < 1 || G > MXFP8_MAX_GROUPS || N <= 0 || K <= 0) return MXFP8_ERR_SHAPE;
    if (N % 32 || K % 32) return MXFP8_ERR_ALIGN;
    if (scale_layout != MXFP8_SCALES_COMPACT && scale_layout != MXFP8_SCALES_BLOCKED) return MXFP8_ERR_LAYOUT;
    const bool row = dirs & MXFP8_ROW, col = dirs & MXFP8_COL;
    if (dirs == 0 || (dirs & ~3u)) return MXFP8_ERR_LAYOUT;
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
    if (mxfp8_status_t r = launch_tiles(dirs, p, st); r != MXFP8_OK) return r;
    if (blocked && row) {
        if (mxfp8_status_t r = pad_rows(p.s_row, p.s_row_bstride, G, nullptr, 0, N, K / 32, st); r != MXFP8_OK) return r;
    }
    if (blocked && col) {
        if (mxfp8_status_t r = pad_cols(p.s_col, p.s_col_bstride, G, nullptr, 0, N, K, st); r != MXFP8_OK) return r;
    }
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
