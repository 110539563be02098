// moe_internal.cuh -- shared device/host definitions of the sm_103a MoE path.
//
// Inline-PTX wrappers for mbarriers, TMA (cp.async.bulk[.tensor]) and the 5th-generation
// tensor cores (tcgen05: TMEM allocation, MMA, commit, TMEM loads), the packed 4-bit weight
// layout, the workspace layout and the bounded-wait machinery.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------------------------
// Packed 4-bit weight layout (written by moe_pack_weights, read by the FFN kernels).
//
// A weight stack [E][N][K] is cut into chunks of 128 rows x 64 input columns (one quant
// group wide).  Chunk (e, m, kb) holds, contiguously:
//   codes   4096 B = [2 halves][128 rows][16 B]; half h covers columns 32h..32h+31 of the
//           K block; 16 B = 4 words, word w covers columns 32h+8w .. +7 with nibble p of the
//           word (bits 4p..4p+3) holding column offset {0,2,4,6,1,3,5,7}[p], so that
//           ((word >> 4s) & 0x000F000F) is the consecutive pair (2s, 2s+1) for s = 0..3, each
//           code sitting in the low mantissa bits of one bf16 half;
//   scales  256 B = bf16 [128 rows];   biases 256 B = bf16 [128 rows].
// Chunks come in pairs: gate/up stacks interleave the gate chunk and the up chunk of the same
// (e, m, kb): [E][I/128][d/64][2][4608 B]; down stacks pair the two 128-row halves of a
// 256-row tile: [E][d/256][I/64][2][4608 B].  One pair (9216 B) is one 256-row MMA operand.
// ------------------------------------------------------------------------------------
// A packed buffer starts with a 256-byte header; int32 header[0] is the scale encoding of the
// whole buffer:
//   kScaleDenorm (0): every scale satisfies |s| < 2^-5 and is stored as S = s * 2^133 (exact).
//     A code q placed in the low mantissa bits of a zero-exponent bf16 is the subnormal
//     q * 2^-133, so fma.rn.bf16x2(code, S, bias) = bf16(s*q + bias) with one rounding.
//   kScaleMagic (1): scales stored as is; codes go through the bf16 128 + q form and one
//     exact subtraction of 128 first.
constexpr int kPackHeader = 256;
constexpr int kScaleDenorm = 0;
constexpr int kScaleMagic = 1;
constexpr int kTileRows = 128;          // rows of a packed chunk = MMA M
constexpr int kBK = 64;                 // columns of a packed chunk = one quant group
constexpr int kChunkCodes = 4096;
constexpr int kChunkBytes = 4608;       // codes + 128 scales + 128 biases
constexpr int kChunkPairBytes = 2 * kChunkBytes;

// ------------------------------------------------------------------------------------
// Workspace layout (byte offsets from the caller's workspace pointer, 256-aligned).
// ------------------------------------------------------------------------------------
struct WsLayout {
    size_t status;      // int32[64]: [0] status bits, [1] decode done-counter, [2..] per-tile counters
    size_t rpart;       // fp32 [KS][T][E] tensor-core partial router logits
    size_t wnorm;       // fp32 [E] router weight row norms
    size_t blk;         // int32 [nblk][E] per-block counts, then per-block bases
    size_t gu_tiles;    // int4 [max_gu]: (expert, first row, rows, weight tile)
    size_t gu_num;      // int32
    size_t dn_tiles;    // int4 [max_dn]
    size_t dn_num;      // int32
    size_t xs;          // bf16 [k*T][d] rows in expert-group order
    size_t H;           // bf16 [(k+1)*T][2*I] (hi | lo)
    size_t acc;         // fp32 [T][d] token-order sum (decode kernels)
    size_t Y;           // fp32 [(k+1)T][d] weighted down-projection rows (prefill), row order of H
    size_t dec;         // decode scratch: logits fp32 [8][E], g/u fp32 [8][k+1][2][I]
    size_t fzlog;       // u64 [8][E]: tagged logits of the one-launch decode kernel (eight copies)
    size_t trace;       // tuning builds (MOE_TRACE): 64 KB of phase timestamps
    size_t total;       // bytes of the workspace
    size_t wbf;         // bf16-weight ablation only (beyond total): every chunk pair of the routed
                        // then the shared packed buffer, dequantised, 32 KB each
    size_t total_unfused;
    int nblk, max_gu, max_dn;
};

constexpr int kRouteBlockTokens = 32;   // tokens per routing block (one warp, one bitmask)
constexpr int kMaxN = 128;              // max token rows of a GEMM tile (MMA M)
constexpr int kDecodeMaxT = 8;          // largest T the decode (GEMV) kernels take
// Token rows of a GEMM block (moe_options.gemm_rows; one value for gate/up and down): an expert's
// rows are cut into near-equal blocks of at most this many rows.  128 by default: smaller blocks
// were measured slower at 4096 tokens (per-token dequant and MMA issue outweigh the overlap they
// allow, and every block re-reads its expert's weights).  The workspace's tile lists are sized
// for the smallest block.
constexpr int kGemmRowsDefault = 128;
// The down projection caps its blocks at 96 rows: four 96-column accumulator slots then hold two
// tiles (two matrices each), so a tile's MMAs never wait for the previous tile's epilogue.
constexpr int kDnMaxRows = 96;
constexpr int kGemmRowsMin = 16;
inline bool gemm_rows_valid(int r) { return r == 16 || r == 32 || r == 64 || r == 128; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Prefill output path of the down projection.  By default the weighted rows are added into
// the fp32 token-order sum (T x d, L2-resident) with bulk reduce-adds issued by the epilogue
// (addition order not fixed).  Deterministic mode stores every weighted row ((k+1) T x d fp32)
// and combine_rows sums each token's rows in a fixed order.  The reduce-adds were faster at
// every measured size, from 128 to 4096 tokens (the rows make a round trip through L2 or HBM).
inline bool ffn_rows_output(int /*T*/, int /*d*/, int /*k*/, bool deterministic) { return deterministic; }

// K slices of the tensor-core router GEMM (partial sums, combined when picking candidates):
// enough that (token blocks of 128) x slices reaches ~128 CTAs, at most 16 and at most one
// slice per 64-column K block
#ifndef MOE_ROUTER_KS_MAX
#define MOE_ROUTER_KS_MAX 16
#endif
inline int router_kslices(int T, int d) {
    const int blocks = (T + 127) / 128, kb = d / 64;
    int ks = 1;
    while (ks < MOE_ROUTER_KS_MAX && ks < kb && blocks * ks < 128) ks *= 2;
    return ks;
}

// Decode scratch of the GEMV kernels: router logits fp32 [8][E], g/u sums fp32 [8][k+1][2][I].
inline size_t decode_scratch_bytes(int d, int E, int k, int I) {
    (void)d;
    return (size_t)kDecodeMaxT * E * 4 + (size_t)kDecodeMaxT * (k + 1) * 2 * I * 4;
}

inline WsLayout ws_layout(const moe_shape& s) {
    WsLayout L{};
    const int T = s.T, d = s.d, E = s.E, k = s.k, I = s.I;
    L.nblk = (T + kRouteBlockTokens - 1) / kRouteBlockTokens;
    // GEMM blocks of at most kGemmRowsMin rows (the smallest option): at most
    // rows / kGemmRowsMin + groups per expert set, times the weight tiles
    const int shared_nt = (T + kGemmRowsMin - 1) / kGemmRowsMin;
    const int routed_nt = k * T / kGemmRowsMin + E + 1;
    L.max_gu = (routed_nt + shared_nt) * (I / kTileRows);
    L.max_dn = (routed_nt + shared_nt) * (d / 256);
    size_t o = 0;
    L.status = o; o = align_up(o + 64 * 4, 256);
    L.rpart = o; o = align_up(o + (size_t)router_kslices(T, d) * T * E * 4, 256);
    L.wnorm = o; o = align_up(o + (size_t)E * 4, 256);
    L.blk = o; o = align_up(o + (size_t)2 * L.nblk * E * 4, 256);
    L.gu_tiles = o; o = align_up(o + (size_t)L.max_gu * 16, 256);
    L.gu_num = o; o = align_up(o + 16, 256);
    L.dn_tiles = o; o = align_up(o + (size_t)L.max_dn * 16, 256);
    L.dn_num = o; o = align_up(o + 16, 256);
    L.xs = o; o = align_up(o + (size_t)k * T * d * 2 + 256 * d * 2, 1024);
    L.H = o; o = align_up(o + (size_t)(k + 1) * T * 2 * I * 2 + 256 * 2 * I * 2, 1024);
    L.acc = o; o = align_up(o + (size_t)T * d * 4, 256);
    L.Y = o; o = align_up(o + (size_t)(k + 1) * T * d * 4, 256);
    L.dec = o; o = align_up(o + decode_scratch_bytes(d, E, k, I), 256);
    L.fzlog = o; o = align_up(o + (size_t)8 * E * 8, 256);
#ifdef MOE_TRACE
    L.trace = o; o += 65536;
#endif
    L.total = o;
    // pairs per expert: gate/up (I/128 row tiles x d/64 K blocks), down (d/256 x I/64)
    const size_t pairs = (size_t)(I / 128) * (d / 64) + (size_t)(d / 256) * (I / 64);
    L.wbf = align_up(o, 1024);
    L.total_unfused = L.wbf + (size_t)(E + 1) * pairs * (2 * 128 * 64 * 2);
    return L;
}

// ------------------------------------------------------------------------------------
// Device helpers
// ------------------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A wait gives up after this many SM cycles (about 2 s at 2 GHz); the kernel then records
// MOE_STATUS_TIMEOUT and unwinds.  clock64 is cheap to read, unlike %globaltimer.  (The
// timeout test builds a separate copy of the library with a shorter limit.)
#ifndef MOE_WAIT_LIMIT_CYCLES
#define MOE_WAIT_LIMIT_CYCLES 4000000000ll
#endif
constexpr long long kWaitLimitCycles = MOE_WAIT_LIMIT_CYCLES;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
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

// Expect `bytes` more transaction bytes in the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes (or the hint
// runs out) instead of spinning, so waiting warps leave the issue slots to working warps.
constexpr uint32_t kSuspendHintNs = 1000000;   // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded spin (non-suspending test_wait) for single-thread roles, whose wake-up latency is
// on the critical path.  Same contract as mbar_wait.
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t n = 0;
    while (true) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((++n & 255u) == 0) {
            if (*abort) return false;
            if (clock64() - t0 > kWaitLimitCycles) return false;
        }
    }
}

// Bounded wait for the phase with the given parity to complete.  Returns false when the
// wait ran out or another role of the CTA already aborted (*abort != 0).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
}

// mbar_wait by every lane of a warp, with one answer for all (false if any lane gave up), so the
// warp's control flow stays uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// One lane of the (converged) warp: true in exactly one lane.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Bulk copy global -> shared (contiguous bytes; 16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled TMA load (coordinates: c0 innermost, in elements).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Warm L2 with a contiguous range (16-byte multiple); no shared memory, no completion.
__device__ __forceinline__ void prefetch_l2(const void* gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem), "r"(bytes) : "memory");
}

// Warm L2 with one tile of a 2-D tensor map.
__device__ __forceinline__ void prefetch_l2_tile(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Hardware named barrier (ids 1..15; 0 is __syncthreads): waiting warps use no issue slots.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a predicate over its threads: all of them get the same answer,
// so a decision taken right after it (such as unwinding) is the same in every warp that waits
// on the barrier.  (Reading a shared flag after a plain barrier is not: another role may set it
// between two warps' reads, and the warps that go on would then wait at the next barrier for
// the ones that left.)
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------- tcgen05 ------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
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

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B
// apart (SBO), rows of 128 B; start address advanced by 32 B per 16-element K step.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);          // start address  [0,14)
    d |= (uint64_t)(16u >> 4) << 16;                        // leading byte offset (unused)
    d |= (uint64_t)(1024u >> 4) << 32;                      // stride byte offset  [32,46)
    d |= (uint64_t)1 << 46;                                 // descriptor version  [46,48)
    d |= (uint64_t)2 << 61;                                 // layout: 128B swizzle [61,64)
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                       // D format f32
           | (1u << 7)                     // A format bf16
           | (1u << 10)                    // B format bf16
           | ((uint32_t)(N >> 3) << 17)    // N >> 3
           | ((uint32_t)(M >> 4) << 24);   // M >> 4
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA with A (M x K, K-major: row m in lane m, K pairs packed per 32-bit column) read
// from tensor memory at column a_tmem.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 bits x 16 columns (one column per register) from TMEM.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// The same wait with the loaded registers as operands: arithmetic on them cannot be scheduled
// before it (needed when other code sits between a tcgen05.ld and its wait).
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// 32 lanes x 32 bits x 32 columns (one column per register) into TMEM.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------- misc ---------------------------------------------------
__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// Eight weights of one packed 32-bit word (pairs (0,1) (2,3) (4,5) (6,7) as bf16x2) with the
// per-row scale and bias pairs s2 / b2 of the buffer's scale encoding.
// Scaled-code encoding: a bf16 bit pattern n < 256 has the value n * 2^-133 (a subnormal, or a
// number of the lowest normal binade), so the code at bits 0..3 of a half is read in place as
// q * 2^-133 and the code at bits 4..7 as 16 q * 2^-133, the latter against the stored scale
// divided by 16 (exact).  Both products are exactly q * scale, and the FMA rounds q * scale +
// bias once: the same bf16 as with each code shifted down first.  Codes at bits 8..15 take
// one shift of the word.
template <bool kDenorm>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t b2, uint32_t (&v)[4]) {
    if (kDenorm) {
        const uint32_t s16 = bf16x2_fma(s2, 0x3D803D80u, 0x80008000u);      // S * 2^-4 (+ -0)
        const uint32_t w8 = w >> 8;
        v[0] = bf16x2_fma(w & 0x000F000Fu, s2, b2);                         // q * 2^-133 * S + b
        v[1] = bf16x2_fma(w & 0x00F000F0u, s16, b2);                        // 16 q * 2^-133 * S / 16 + b
        v[2] = bf16x2_fma(w8 & 0x000F000Fu, s2, b2);
        v[3] = bf16x2_fma(w8 & 0x00F000F0u, s16, b2);
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t c = (u == 0 ? w : (w >> (4 * u))) & 0x000F000Fu;
            const uint32_t q = bf16x2_fma(c | 0x43004300u, 0x3F803F80u, 0xC300C300u);   // (128 + q) - 128
            v[u] = bf16x2_fma(q, s2, b2);
        }
    }
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_nc_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void set_status(int* status, int bits) { atomicOr(status, bits); }

// Programmatic dependent launch: wait for the previous grid's results / let the next grid start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization: the kernel may start (and run its prologue)
// while the previous kernel on the stream finishes; every such kernel calls pdl_wait() before
// its first global memory access and pdl_launch_dependents() only after that wait, so at most
// one launch waits ahead and every kernel still sees all earlier ones complete.
template <typename... KArgs, typename... Args>
cudaError_t launch_with_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// Order-preserving key: larger logit first, then lower expert index.  NaN counts as -inf
// and -0 as +0 (they compare equal to +0).
__device__ __forceinline__ unsigned long long topk_key(float v, int e) {
    if (v != v) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;
    uint32_t u = __float_as_uint(v);
    uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)o << 32) | (uint32_t)(0xFFFFu - (uint32_t)e);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        unsigned long long o = __shfl_xor_sync(0xffffffffu, v, m);
        v = o > v ? o : v;
    }
    return v;
}

// Top-k of the E=256 logits in lg (shared or global) with one warp; returns (in lane j < k)
// the expert and weight of slot j.  Weights: exp(l_j - l_0) / sum over the kept logits.
__device__ __forceinline__ void warp_topk256(const float* lg, int k, int lane, int& out_e, float& out_w) {
    unsigned long long key[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) key[s] = topk_key(lg[lane + 32 * s], lane + 32 * s);
    int my_e = -1;
    float my_l = 0.f, l0 = 0.f;
    for (int j = 0; j < k; ++j) {
        unsigned long long best = 0;
#pragma unroll
        for (int s = 0; s < 8; ++s) best = key[s] > best ? key[s] : best;
        best = warp_max_u64(best);
        const int e = 0xFFFF - (int)(best & 0xFFFFu);
        const float l = lg[e];
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if ((e & 31) == lane && (e >> 5) == s) key[s] = 0;   // remove the winner
        if (j == 0) l0 = (l != l) ? -INFINITY : l;
        if (lane == j) { my_e = e; my_l = (l != l) ? -INFINITY : l; }
    }
    float ex = (lane < k) ? expf(my_l - l0) : 0.f;
    float den = ex;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) den += __shfl_xor_sync(0xffffffffu, den, m);
    out_e = my_e;
    out_w = ex / den;
}

// Thread-block clusters: rank in the cluster, the split cluster barrier, and a 32-bit load
// from the same offset in another CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ float ld_dsmem_f32(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Hand-off into another CTA of the cluster: a 32-bit store to its shared memory and a release
// arrive on its mbarrier (same offsets as the local objects), and the matching acquire test.
__device__ __forceinline__ void st_dsmem_u32(void* local, uint32_t rank, uint32_t v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_release(uint64_t* local_bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
__device__ __forceinline__ bool mbar_test_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Fire-and-forget fp32 add into global memory.
__device__ __forceinline__ void red_add_f32_global(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// GPU-scope release add / acquire load on a global counter.
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Warp-level bf16 MMA m16n8k16 with fp32 accumulation (operands in registers).  Used by the
// one-token GEMV as a dot-product unit: every column of B holds the same activations, so
// every column of D holds the 16 row dots.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Warm L2 with [p, p + bytes) split over the threads of a grid (each thread up to 4 KB pieces).
__device__ __forceinline__ void prefetch_l2_range(const uint8_t* p, size_t bytes, size_t worker, size_t nworkers) {
    for (size_t o = worker * 4096; o < bytes; o += nworkers * 4096) {
        const uint32_t n = (uint32_t)(bytes - o < 4096 ? bytes - o : 4096) & ~15u;
        if (n) prefetch_l2(p + o, n);
    }
}

#endif  // __CUDACC__

// ------------------------------------------------------------------------------------
// Launch wrappers (host), one per translation unit
// ------------------------------------------------------------------------------------
struct RouteArgs {
    int T, d, E, k, tile_rows;
    int gu_rows, dn_rows;      // token rows of a gate/up and of a down GEMM block (at most)
    const uint16_t* x;
    const uint16_t* w_router;
    const float* bias;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* pos;
    int32_t* tiles;
    int32_t* num_tiles;
    int I;
    uint8_t* ws;
    WsLayout L;
    const uint8_t* pf_ptr;     // optional: weights to warm in L2 while routing (decode)
    size_t pf_bytes;
    int num_sms;               // grid of the persistent FFN kernels (tile j runs on CTA j % num_sms)
};

// Where the shared expert's tiles go in a GEMM tile list of `total` entries (`shared` of them):
// the persistent kernels give entry j to CTA j % grid, so the CTAs from total % grid on run
// one tile fewer; the shared expert's tiles (the chunk's full token blocks, the heaviest) are
// placed at entry total % grid when they fit before the end of that round and of the list,
// else first.  The experts' entries keep their order around them (a permutation of 0..total-1).
__host__ __device__ inline int shared_tiles_at(int total, int shared, int grid) {
    if (grid <= 0) return 0;
    const int p0 = total % grid;
    return p0 + shared <= grid && p0 + shared <= total ? p0 : 0;
}

struct FfnArgs {
    int T, d, E, k, I;
    const uint16_t* x;
    const int32_t* topk_idx;
    const float* topk_w;
    const int32_t* perm;
    const uint8_t* w_routed;   // packed buffer (header first)
    const uint8_t* w_shared;   // packed buffer (header first)
    uint8_t* ws;
    WsLayout L;
    int num_sms;
    bool rows_out;             // down projection: weighted rows (true) or reduce-adds into the sum
    bool unfused;              // ablation: dequantise every weight to bf16 in the workspace first
};

cudaError_t launch_route_prefill(const RouteArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_route_prefill_host(const RouteArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_router, const float* bias, float* out, int T,
                                 int d, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_route_decode(const RouteArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_combine(int T, int d, const float* acc, uint16_t* y, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_decode_gate_up(const FfnArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_decode_down(const FfnArgs& a, uint16_t* y, cudaStream_t st, unsigned long long* launches);
// One-token forward in one launch (route + gate/up + down + combine).  Returns
// cudaErrorNotSupported, with nothing launched, when the shape or the GPU does not fit it.
struct FusedDecodeArgs {
    int d, E, k, I;
    const uint16_t* x;
    const uint16_t* w_router;
    const float* bias;
    const uint8_t* w_routed;   // packed buffers (header first)
    const uint8_t* w_shared;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* pos;
    int32_t* tiles;
    int32_t* num_tiles;
    int* status;               // status word and counters (64 ints)
    unsigned long long* logit_words;   // [8][E]: (call tag << 32) | fp32 logit bits, one copy per cluster rank; no other kernel writes it
    float* acc;                // fp32 [d], zero between calls: the weighted sum
    uint16_t* y;
    unsigned long long* trace; // tuning builds (MOE_TRACE) only
};
cudaError_t launch_gate_up_tm(const FfnArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_combine_rows(int T, int d, int k, const float* Y, const int32_t* pos, uint16_t* y, cudaStream_t st,
                                unsigned long long* launches);
cudaError_t launch_down_tm(const FfnArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_decode_fused(const FusedDecodeArgs& a, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_pack(int E, int N, int K, const moe_q4& m, int pair_slot, int pair_count, uint8_t* dst,
                        const int* mode, cudaStream_t st, unsigned long long* launches);
cudaError_t launch_scale_check(size_t n, const uint16_t* scales, int* mode, cudaStream_t st,
                               unsigned long long* launches);

// Encodes 2-D bf16 tensor maps (host; driver entry point fetched through the runtime).
cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                              bool swizzle128 = true);

}  // namespace moe
