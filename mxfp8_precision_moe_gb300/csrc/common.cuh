// common.cuh -- device helpers shared by the sm_103a kernels: status reporting,
// bounded mbarrier waits, TMA / bulk copies, tcgen05 (tensor memory + MMA)
// wrappers, and the E4M3 / E8M0 element rules.  Inline PTX only; no library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mxfp8moe.h"

#ifndef __CUDACC_RTC__
#include <stdio.h>
#endif

namespace mx {

constexpr int kBlk = 32;          // elements per MX block
constexpr int kMaxGroups = MXFP8_MAX_GROUPS;

// ---------------------------------------------------------------- status
__device__ __forceinline__ void report(int32_t* dev_status, int32_t code) {
    if (dev_status != nullptr) atomicCAS(dev_status, 0, code);
}

// ---------------------------------------------------------------- element rules
// Shared scale byte from the largest |x| of a block given as bf16 magnitude bits
// (x & 0x7FFF, compared as integers: NaN > Inf > any finite, and finite values
// order like their magnitudes).  With E the 8-bit exponent field of that bf16
// amax, floor(log2(amax)) = E - 127 for normal values, so the OCP rule
// e = floor(log2 amax) - 8 clamped at -127 becomes s = max(E - 8, 0); bf16
// subnormals and zero (E = 0) land on the clamp.  E = 255 (Inf/NaN) -> 0xFF.
__device__ __forceinline__ uint32_t e8m0_from_absbits(uint32_t amax_bits16) {
    uint32_t E = amax_bits16 >> 7;
    if (E == 0xFFu) return 0xFFu;
    return E > 8u ? E - 8u : 0u;
}

// 2^(127 - s) as an fp32 (s <= 246 keeps the exponent field 254 - s normal).
// For s == 0xFF returns a quiet NaN so every element of the block becomes NaN.
__device__ __forceinline__ float inv_scale_from_e8m0(uint32_t s) {
    return s == 0xFFu ? __int_as_float(0x7fc00000) : __int_as_float((int)((254u - s) << 23));
}

// Two fp32 -> two E4M3 codes, round-to-nearest-even, satfinite.  lo goes to
// byte 0, hi to byte 1.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// Two fp32 -> a bf16 pair (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// bf16 pair packed in a u32 -> the two fp32 values (exact).
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// SwiGLU backward of one bf16 pair, elementwise at the rounding points of the bf16 autograd ops, fp32
// inside: g = dh, x = h1, u = h3 of h = silu(h1) * h3 with sig = 1 / (1 + e^-h1):
//   dh3 = bf16(dh * bf16(silu(h1))),  dh1 = bf16(bf16(dh * h3) * sig * (1 + h1 * (1 - sig))).
__device__ __forceinline__ void swiglu_bwd_pair(uint32_t g, uint32_t x, uint32_t u, uint32_t& dh1, uint32_t& dh3) {
    const float g0 = bf16lo(g), g1 = bf16hi(g);
    const float x0 = bf16lo(x), x1 = bf16hi(x);
    const float sg0 = 1.0f / (1.0f + expf(-x0)), sg1 = 1.0f / (1.0f + expf(-x1));
    const uint32_t sl = pack_bf16x2(x0 * sg0, x1 * sg1);              // bf16(silu(h1))
    const uint32_t ds = pack_bf16x2(g0 * bf16lo(u), g1 * bf16hi(u));  // bf16(dh * h3)
    dh3 = pack_bf16x2(g0 * bf16lo(sl), g1 * bf16hi(sl));
    dh1 = pack_bf16x2(bf16lo(ds) * sg0 * (1.0f + x0 * (1.0f - sg0)), bf16hi(ds) * sg1 * (1.0f + x1 * (1.0f - sg1)));
}

// max over the two 16-bit halves (unsigned), one instruction on sm_90+.
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// ---------------------------------------------------------------- blocked scale layout
// Byte offset of scale (row r, block-column c) in the 128x4-tile layout with
// `ct` column tiles per 128-row band.
__device__ __forceinline__ int64_t blocked_off(int64_t r, int64_t c, int64_t ct) {
    return ((r >> 7) * ct + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// ---------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same with a suspend-time hint: a thread whose phase has not completed sleeps until it completes
// or kSuspendNs pass, instead of re-polling.  In the GEMM kernels the waiting epilogue warps then leave
// the issue slots to the producer, MMA and scale-copy threads (3-6% faster GEMMs, identical outputs).
// The quantize kernels keep the default wait: their stages turn over every few microseconds, and the
// folded-producer stability kernels ran up to 28% slower with the hint.
constexpr uint32_t kSuspendNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase.  Returns false (after recording
// MXFP8_ERR_TIMEOUT) once `limit_ns` of wall time has passed, or at once when
// another role of the CTA has already given up (*abort != 0).  Never traps.
// kSleep: wait with the suspend-time hint (mbar_try_wait_sleep).
template <bool kSleep = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile int* abort, int32_t* dev_status) {
    auto try_wait = [&] { return kSleep ? mbar_try_wait_sleep(bar, parity) : mbar_try_wait(bar, parity); };
    if (try_wait()) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (true) {
        if (try_wait()) return true;
        // a failed sleeping wait has already slept up to kSuspendNs: check on every one of those
        if (kSleep || ((++spins) & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1;
                report(dev_status, MXFP8_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void st_shared_v4(void* p, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p))
                 : "memory");
    return v;
}

// ---------------------------------------------------------------- TMA / bulk copies
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Copy 32 rows x 16 bytes of shared memory (one 128x4 scale tile) into tensor
// memory at column `taddr`, replicated to all four 32-lane sub-partitions.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D(tmem) (+)= A(smem) x B(smem)^T with per-32-K block scales from tensor memory.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- CTA pairs (clusters of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Relaxed arrives, for handing a tensor-memory accumulator back to the MMA warp.  The epilogue's
// reads of it are complete (tcgen05.wait::ld blocks until they are) and tcgen05.fence::before_thread_sync
// orders them before the arrive; nothing in generic memory is handed over.  A release arrive would
// also wait until every earlier global store of the thread is performed -- the previous tile's
// output, tens of KB in flight -- and so hold the tensor pipe idle for thousands of cycles per tile.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// 2D TMA load into this CTA's shared memory, completing on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t cluster_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive on the mbarrier at this shared offset in every CTA of `cta_mask` once all tcgen05
// operations issued so far by this thread are done.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Scale tile copy for a CTA pair: each CTA's shared memory -> its own tensor memory, same addresses.
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 256-row pair MMA (rows 0-127 in the even CTA's tensor memory, 128-255 in the odd CTA's).
__device__ __forceinline__ void tc_mma_pair_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in bits
// [0,14), leading-dimension byte offset >> 4 in [16,30), stride-dimension byte
// offset >> 4 in [32,46), descriptor version 1 in [46,48), swizzle mode in
// [61,64) (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(swizzle & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::mxf8f6f4 with E4M3 x E4M3, both operands
// K-major, E8M0 scales, dense, M x N tile; a_sf / b_sf select which byte of
// the 32-bit scale column word (i.e. which 32-wide K block) the MMA uses.
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t M, uint32_t N, uint32_t a_sf, uint32_t b_sf) {
    return ((b_sf & 3u) << 4)        // B scale-factor id
           | (0u << 7)               // A format: E4M3
           | (0u << 10)              // B format: E4M3
           | (0u << 15)              // A K-major
           | (0u << 16)              // B K-major
           | ((N >> 3) << 17)        // N / 8
           | (1u << 23)              // scale type: UE8M0
           | ((M >> 4) << 24)        // M / 16
           | ((a_sf & 3u) << 29);    // A scale-factor id
}

}  // namespace mx
