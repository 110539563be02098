// ffn.cu -- grouped SwiGLU FFN over packed 4-bit group-affine weights, sm_103a tcgen05 with
// the dequantised weights as the MMA's A operand in tensor memory.
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026), section "Dequantize
// weights during matrix multiplication": the grouped GEMM rebuilds one small bf16 weight tile
// at a time on chip, multiplies it with the routed activation rows, accumulates in fp32 and
// writes bf16; the expanded weight matrix never exists in memory.  Section "Match tile size to
// expert load": the token side of a tile follows the expert's row count (16 to 128 rows), so
// small expert groups cost little tensor work.  Section "Reduce intermediate and state
// traffic": gate/up fused with the gated activation; the output projection fused with the
// routing score and the shared-expert sum.
//
// A tile is (expert, block of token rows, weight tile): blocks of at most 128 rows (gate/up)
// or 96 rows (down).  Every MMA computes
//     D[m][n] (+)= sum_k W[m][k] X[n][k]     M = 128 weight rows, N = 16 ceil(rows / 16), K = 16
// with W, bf16, read from tensor memory (TMEM) and X, the block's token rows, read from shared
// memory (128-byte swizzled, K-major).  Writing the dequantised weights to TMEM keeps them off
// the shared-memory path entirely: shared memory carries only the packed codes, the token rows
// and the tensor core's reads of the token rows.
//   gate/up  two A matrices per K block: 128 gate rows and the same 128 up rows (i = 128 wt ..),
//            so g and u of one (i, token) sit in the same TMEM lane and column of D_0 / D_1;
//            h = silu(g) u is written as a bf16 hi/lo pair.
//   down     two A matrices: output rows 256 wt .. +127 and +128 .. +255; h enters as its hi
//            half and its lo half: for N <= 32 as one B operand of 2N rows (hi rows, then lo
//            rows; y = D[n] + D[N + n]), else as two MMAs per K step into the same D; weight * y
//            (fp32) of both matrices is staged per 32-token chunk and leaves in one of two ways:
//            added into the fp32 token-order sum with one 1 KB bulk reduce-add per token
//            (default), or, in deterministic mode, stored into Y [d/128][(k+1)T][128] at the
//            row index of h with bulk copies (plain stores, no atomics).
// combine_rows sums each token's k routed rows and its shared row of Y in a fixed order.
// Warp roles (28 warps):
//   0-15  dequant, two sets of 8 warps taking alternate K blocks: warp w owns row 32 (w & 3) +
//         lane of matrix (w >> 2) & 1; per K block a thread loads its 64 codes (two 16-byte
//         loads), dequantises them exactly (eight words, one bf16x2 FMA per two weights) and
//         writes the row with one tcgen05.st (32 columns)
//   16-23 epilogue, two warps per TMEM lane quadrant taking alternate 16-token column groups:
//         D -> registers (lane = weight row, column = token) -> token-major staging in shared
//         memory -> 16-byte stores of h, or bulk copies / reduce-adds of weight * y
//   24    codes producer: cp.async.bulk of the 9216-byte packed chunk pair of each K block
//   25    token-row producer: TMA loads of the block's token rows (64-row boxes, then 16-row
//         boxes for the rest)
//   26-27 MMA issuers: warp 26 + m issues every MMA into D_m (two issuers: the tensor core
//         finishes a 128 x N x 16 MMA with A in TMEM in about N / 2 cycles, so for small N the
//         issue rate matters); warp 26 owns the TMEM allocation
// Warps 24-27 walk their loops with all 32 lanes, so counters, descriptors and addresses stay
// warp-uniform, and one lane chosen by elect.sync issues the copies, TMA loads, MMAs and
// commits (a single lane in a divergent branch issued about one tcgen05.mma per 50 cycles).
// TMEM (512 columns): an A ring of slots of 64 columns from column 0 (slot s, matrix m, K step ks
// at 64 s + 32 m + 8 ks), then the accumulator slots.
//   gate/up  4 A slots, 2 D slots of 128 columns: a tile whose two accumulators fit in 128
//            columns (N <= 64) takes one slot, so the next tile's MMAs run while the epilogue
//            drains it; a larger tile takes both (D_m in its own slot).
//   down     2 A slots, 4 D slots of 96 columns, one matrix each: matrix m of the t-th tile is
//            use j = 2t + m of the slot ring (slot j % 4), so the next tile's two matrices use
//            the two slots the current tile does not.
// MMA issuers and epilogue walk the same slot sequence.
// Each MMA issuer commits once per K block to a ring of "K block done" barriers (two arrivals);
// the dequant sets (A slot reuse) and the token-row producer (token-row slot reuse) wait on it.
// One "ready" barrier per K block collects the dequant set's warps and the token-row bytes, so
// an MMA issuer waits once per K block.
// All waits are bounded (MOE_STATUS_TIMEOUT, then the CTA unwinds).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTmDeqSet = 8;                  // warps of one dequant set
constexpr int kTmDeqWarps = 2 * kTmDeqSet;
constexpr int kTmEpiWarp0 = kTmDeqWarps;      // 16
constexpr int kTmEpiWarps = 8;                   // two per TMEM lane quadrant
constexpr int kTmEpiThreads = kTmEpiWarps * 32;
constexpr int kTmCodeWarp = kTmEpiWarp0 + kTmEpiWarps;
constexpr int kTmXWarp = kTmCodeWarp + 1;
constexpr int kTmMmaWarp = kTmXWarp + 1;                 // two MMA warps
constexpr int kTmThreads = (kTmMmaWarp + 2) * 32;

constexpr int kTmBox = 16;                    // token rows per small TMA box
constexpr int kTmBoxL = 64;                   // token rows per large TMA box
constexpr int kTmKD = 8;                      // "K block done" barriers

// Ring chunk of the bf16-weight ablation (moe_options.unfused_dequant): the two 128-row
// matrices of a K block as dequantised bf16, [matrix][16-byte word w4][row][16 bytes], so the
// thread of row r reads its 64 weights conflict-free.
constexpr int kBf16PairBytes = 2 * kTileRows * kBK * 2;

template <bool kDown, bool kBf16 = false>
struct TmCfg {
    // TMEM: A ring of A slots x 64 columns from column 0, then NDS accumulator slots of DW
    // columns from column DCOL0.  Down: four slots of 96 columns, one matrix each, so the two
    // matrices of the next tile never wait for the epilogue of the current one (token blocks of
    // at most kDnMaxRows rows)
    static constexpr int A = kDown ? 2 : 4;
    static constexpr int NDS = kDown ? 4 : 2;
    static constexpr uint32_t DW = kDown ? 96u : 128u;
    static constexpr uint32_t DCOL0 = 64u * A;
    static_assert(DCOL0 + DW * NDS == 512u, "TMEM columns");
    static_assert(!kDown || kDnMaxRows <= (int)DW, "down token block wider than its accumulator slot");
    static constexpr int RX = kDown ? (kBf16 ? 2 : 4) : 8;   // token-row ring slots
    static constexpr int CH = kBf16 ? kBf16PairBytes : kChunkPairBytes;   // bytes of a weight chunk
    static constexpr int RC = kBf16 ? 2 : (kDown ? 6 : 8);  // weight-chunk ring slots
    // The two dequant sets take alternate K blocks.  With an even ring every slot belongs to
    // one set, whose parity waits on it are then never more than one phase ahead.  With an odd
    // ring consecutive uses of a slot alternate between the sets: a set reaching block it has
    // finished block it - 2, which waited for block it - 2 - A, so the slot's previous block
    // it - RC is certain to be done only when RC >= A + 2.  A smaller odd ring lets a parity wait
    // pass a phase early, and the ring's barriers fall out of step.
    static_assert(RC % 2 == 0 || RC >= A + 2, "weight-chunk ring: even, or at least A + 2 slots");
    static constexpr int PARTS = kDown ? 2 : 1;              // hi, lo halves of h
    static constexpr int XPART = (kDown ? kDnMaxRows : kMaxN) * 128;   // bytes of one part of a slot
    static constexpr int XS = PARTS * XPART;                 // bytes of a token-row slot
    // staging of 32 tokens: gate/up bf16 [32][hi 128 | lo 128]; down a ring of NSTG buffers of
    // fp32 [32][256] (both matrices of a tile)
    static constexpr int NSTG = kDown ? 2 : 1;
    static constexpr int STAGE = kDown ? NSTG * 32 * 1024 : 32 * 512;
    // bits of a lane's issue history that may still read a staging buffer: the last NSTG - 2 chunks
    static constexpr uint32_t HIST_MASK = NSTG >= 2 ? (1u << (NSTG >= 2 ? NSTG - 2 : 0)) - 1u : 0u;
    static constexpr int x_off = 0;
    static constexpr int c_off = x_off + RX * XS;
    static constexpr int stage_off = c_off + RC * CH;
    static constexpr int tab_off = stage_off + STAGE;        // down: float weight[2][128], int token[2][128]
    static constexpr int bar_off = tab_off + 2048;
};

struct TmBars {
    uint64_t c_full[8], c_empty[8], ready[kTmKD], kb_done[kTmKD];
    uint64_t d_full[4], d_empty[4], drain[2];
    uint32_t tmem_slot;
    int abort;
};

template <bool kDown, bool kBf16 = false>
constexpr int tm_smem_bytes() {
    return TmCfg<kDown, kBf16>::bar_off + (int)sizeof(TmBars) + 1024;   // + alignment slack
}
static_assert(tm_smem_bytes<false>() <= 232448, "gate/up smem");
static_assert(tm_smem_bytes<true>() <= 232448, "down smem");
static_assert(tm_smem_bytes<false, true>() <= 232448, "gate/up smem (bf16 weights)");
static_assert(tm_smem_bytes<true, true>() <= 232448, "down smem (bf16 weights)");

struct TmParams {
    const uint8_t* w_routed;   // packed stack: [E][tiles][K/64][2][4608]
    const uint8_t* w_shared;
    const int* mode_routed;    // scale encoding of each packed buffer (header word)
    const int* mode_shared;
    const int4* tiles;         // (expert, first row, rows, weight tile); expert == E: shared
    const int* num_tiles;
    uint16_t* H;               // [(k+1)T][2I] bf16, hi | lo
    float* Y;                  // [d/256][(k+1)T][256] fp32 weighted down-projection rows
    float* acc;                // [T][d] fp32 token-order sum
    int rows_out;              // down: 1 = store rows into Y, 0 = bulk reduce-add into acc
    const int32_t* perm;
    const float* topk_w;
    int* status;
    unsigned long long* trace;
    int T, d, I, E, k;
};

__device__ __forceinline__ int tile_n(int rows) { return (rows + 15) & ~15; }

// D placement of a tile, from the running slot counter sc: TMEM columns of D_0 / D_1 and the
// slot(s) they occupy.
struct DSlots {
    int s0, s1;
    bool two;
    uint32_t col0, col1;
};
// Down tiles of at most 32 token rows stack the hi and lo halves of h as one B operand of 2N
// rows (one MMA per K step and matrix, y = D[n] + D[N + n]); larger ones run both halves into the
// same accumulator (two MMAs).
__device__ __forceinline__ bool down_stacked(int N) { return N <= 32; }

__device__ __forceinline__ DSlots d_slots(uint32_t sc, int N, bool down) {
    DSlots r;
    const int w = down && down_stacked(N) ? 2 * N : N;   // columns of one accumulator
    r.s0 = (int)(sc & 1);
    r.two = 2 * w > 128;
    r.s1 = r.two ? r.s0 ^ 1 : r.s0;
    r.col0 = 256u + 128u * r.s0;
    r.col1 = r.two ? 256u + 128u * r.s1 : r.col0 + w;
    return r;
}

// Tuning builds (MOE_TRACE): clock64 stamps of CTA 0's first K blocks / tiles.
#ifdef MOE_TRACE
constexpr int kTmTraceK = 96;
#define TM_TRACE(ev, g)                                                                       \
    do {                                                                                      \
        if (blockIdx.x == 0 && (g) < kTmTraceK) p.trace[(ev) * kTmTraceK + (g)] = clock64(); \
    } while (0)
#else
#define TM_TRACE(ev, g) \
    do {                \
    } while (0)
#endif
enum { TT_PC = 0, TT_PX, TT_DW, TT_DD, TT_DS, TT_MW, TT_MD, TT_ET, TT_ED };

__device__ __forceinline__ void tm_abort(volatile int* abort, int* status) {
    *abort = 1;
    set_status(status, MOE_STATUS_TIMEOUT);
}

// Wait (bounded, not cut short by the abort flag) until the last `last` arms of a ring of
// `ring` full barriers have completed, so no copy is still writing shared memory at exit.
__device__ void tm_drain(uint64_t* full, int ring, int last, uint32_t issued) {
    int never = 0;
    const uint32_t first = issued > (uint32_t)last ? issued - last : 0;
    for (uint32_t i = first; i < issued; ++i) mbar_wait(&full[i % ring], (i / ring) & 1, &never);
}

// One row of 64 weights: 16 bytes of codes per half K block, per-row scale and bias pairs.
template <bool kDenorm>
__device__ __forceinline__ void dequant_row64(uint4 c0, uint4 c1, uint32_t s2, uint32_t b2, uint32_t (&v)[32]) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint32_t o[4];
        dequant_word<kDenorm>(w[q], s2, b2, o);
#pragma unroll
        for (int u = 0; u < 4; ++u) v[4 * q + u] = o[u];
    }
}


// Bulk copy of `bytes` from shared to global memory (16-byte aligned, bytes % 16 == 0);
// completion tracked per thread by bulk groups.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent bulk groups still read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <bool kDown, bool kBf16>
__global__ void __launch_bounds__(kTmThreads, 1)
    ffn_tm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_al,
                  const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_bl, TmParams p) {
    using C = TmCfg<kDown, kBf16>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t* xring = smem + C::x_off;
    uint8_t* cring = smem + C::c_off;
    TmBars* b = reinterpret_cast<TmBars*>(smem + C::bar_off);
    volatile int* abort = &b->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = (kDown ? p.I : p.d) / kBK;                 // weight K blocks
    const int WT = kDown ? p.d / 256 : p.I / kTileRows;      // weight tiles per expert

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::RC; ++i) { mbar_init(&b->c_full[i], 1); mbar_init(&b->c_empty[i], kTmDeqSet); }
        // ready: the 8 dequant warps of a K block's set + the token-row producer (with its bytes)
        for (int i = 0; i < kTmKD; ++i) { mbar_init(&b->ready[i], kTmDeqSet + 1); mbar_init(&b->kb_done[i], 2); }
        // gate/up: both MMA threads commit to a tile's slot(s); down: slot = one matrix's accumulator
        for (int i = 0; i < C::NDS; ++i) { mbar_init(&b->d_full[i], kDown ? 1 : 2); mbar_init(&b->d_empty[i], kTmEpiWarps); }
        mbar_init(&b->drain[0], 1);
        mbar_init(&b->drain[1], 1);
        b->abort = 0;
        fence_barrier_init();
    }
    if (warp == kTmXWarp && lane == 0) {
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_al);
        if (!kDown) { prefetch_tmap(&tm_b); prefetch_tmap(&tm_bl); }
    }
    if (warp == kTmMmaWarp) { tmem_alloc(&b->tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b->tmem_slot;
    // the prologue above may overlap the previous kernel; the tile list comes from it
    pdl_wait();
    pdl_launch_dependents();
    const int num = *p.num_tiles;
    if ((int)blockIdx.x >= num) {
        if (warp == kTmMmaWarp) tmem_dealloc(tmem, 512);
        return;
    }

    if (warp == kTmCodeWarp) {
        // packed codes of every (tile, K block), up to RC K blocks ahead of the dequant; the whole
        // warp walks the loop (warp-uniform counters and addresses), one elected lane issues
        const bool leader = elect_one();
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            const int4 t = p.tiles[tile];
            const uint8_t* w = t.x < p.E ? p.w_routed + (size_t)(t.x * WT + t.w) * KB * C::CH
                                         : p.w_shared + (size_t)t.w * KB * C::CH;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int cs = it % C::RC;
                if (!mbar_wait_warp(&b->c_empty[cs], ((it / C::RC) & 1) ^ 1, abort)) { ok = false; break; }
                if (leader) {
                    mbar_arrive_expect_tx(&b->c_full[cs], C::CH);
                    bulk_g2s(cring + cs * C::CH, w + (size_t)kb * C::CH, C::CH, &b->c_full[cs]);
                    TM_TRACE(TT_PC, it);
                }
                __syncwarp();
            }
        }
        if (leader) {
            if (!ok) tm_abort(abort, p.status);
            tm_drain(b->c_full, C::RC, C::RC, it);
        }
        __syncwarp();
    } else if (warp == kTmXWarp) {
        // token rows of every (tile, K block), up to RX K blocks ahead of the MMA; for the down
        // projection the lo half of h follows the hi rows directly when the tile stacks (N <= 32);
        // the whole warp walks the loop, one elected lane issues
        const bool leader = elect_one();
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            const int4 t = p.tiles[tile];
            const int e = t.x, row0 = t.y, N = tile_n(t.z);
            const int xrow0 = kDown ? (e < p.E ? row0 : p.k * p.T + row0) : row0;
            const CUtensorMap* tms = (kDown || e < p.E) ? &tm_a : &tm_b;
            const CUtensorMap* tml = (kDown || e < p.E) ? &tm_al : &tm_bl;
            const int lo_off = down_stacked(N) ? N * 128 : C::XPART;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int xs = it % C::RX;
                if (it >= (uint32_t)C::RX) {
                    const uint32_t g = it - C::RX;
                    if (!mbar_wait_warp(&b->kb_done[g % kTmKD], (g / kTmKD) & 1, abort)) { ok = false; break; }
                }
                // (the wait above also means that the ready barrier's phase for K block
                // it - 8 has completed: its MMAs were issued)
#ifdef MOE_TEST_DROP_TOKEN_BLOCK
                // timeout test build only: CTA 0 never arms this K block's ready barrier, so
                // the MMA threads' bounded wait on it runs out and the CTA unwinds
                if (blockIdx.x == 0 && it == (uint32_t)(MOE_TEST_DROP_TOKEN_BLOCK)) continue;
#endif
                if (leader) {
                    uint64_t* rdy = &b->ready[it % kTmKD];
                    mbar_arrive_expect_tx(rdy, C::PARTS * N * 128);
                    uint8_t* dst = xring + xs * C::XS;
                    for (int part = 0; part < C::PARTS; ++part) {
                        const int x = part * p.I + kb * kBK;
                        int r = 0;
                        for (; r + kTmBoxL <= N; r += kTmBoxL)
                            tma_load_2d(dst + part * lo_off + r * 128, tml, x, xrow0 + r, rdy);
                        for (; r < N; r += kTmBox)
                            tma_load_2d(dst + part * lo_off + r * 128, tms, x, xrow0 + r, rdy);
                    }
                    TM_TRACE(TT_PX, it);
                }
                __syncwarp();
            }
        }
        if (leader) {
            if (!ok) tm_abort(abort, p.status);
            tm_drain(b->ready, kTmKD, C::RX, it);   // the token rows of the last RX blocks have landed
        }
        __syncwarp();
    } else if (warp >= kTmMmaWarp) {
        // MMA issuer m: the whole warp walks the loop, so its counters and descriptors stay
        // warp-uniform; one elected lane issues every tcgen05.mma and commit
        const int m = warp - kTmMmaWarp;   // this warp's accumulator D_m and A matrix m
        const bool leader = elect_one();
        uint32_t it = 0, tcount = 0, sc = 0, use[3] = {0, 0, 0};
        bool ok = true;
        const uint64_t xdesc0 = sw128_desc(smem_u32(xring));   // start address advances 16 B per unit
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x, ++tcount) {
            const int N = tile_n(p.tiles[tile].z);
            const bool stacked = kDown && down_stacked(N);   // hi and lo rows as one B operand of 2N rows
            const uint32_t idesc = idesc_bf16_f32(128, stacked ? 2 * N : N);
            // gate/up: one or two slots per tile (d_slots); down: use j = 2 tcount + m of the
            // slot ring, slot j % 4, phase j / 4 (the next tile's two matrices take the two
            // slots the current tile does not use)
            const DSlots ds = d_slots(sc, N, kDown);
            const uint32_t dj = 2 * tcount + m;
            const int dsl = kDown ? (int)(dj % 4) : 0;
            if (kDown) {
                if (!mbar_wait_warp(&b->d_empty[dsl], ((dj / 4) & 1) ^ 1, abort)) { ok = false; break; }
            } else if (!mbar_wait_warp(&b->d_empty[ds.s0], (use[ds.s0] & 1) ^ 1, abort) ||
                       (ds.two && !mbar_wait_warp(&b->d_empty[ds.s1], (use[ds.s1] & 1) ^ 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dm = tmem + (kDown ? C::DCOL0 + C::DW * dsl : (m ? ds.col1 : ds.col0));
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int as = it % C::A, xs = it % C::RX;
                if (!mbar_wait_warp(&b->ready[it % kTmKD], (it / kTmKD) & 1, abort)) { ok = false; break; }
                tc_fence_after();
                if (m == 0 && leader) TM_TRACE(TT_MW, it);
                const uint64_t xd = xdesc0 + (uint64_t)((xs * C::XS) >> 4);
                const uint32_t a0 = tmem + 64u * as + 32u * m;
                // both loops fully unrolled: the issuing thread's instruction count sets its pace
                if (leader) {
                    if (C::PARTS == 1 || stacked) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc_mma_bf16_ts(dm, a0 + 8u * ks, xd + (uint64_t)(ks * 2), idesc, (kb | ks) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                            for (int part = 0; part < C::PARTS; ++part)
                                tc_mma_bf16_ts(dm, a0 + 8u * ks, xd + (uint64_t)((part * C::XPART + ks * 32) >> 4),
                                               idesc, (kb | ks | part) ? 1u : 0u);
                        }
                    }
                    tc_commit(&b->kb_done[it % kTmKD]);
                    if (m == 0) TM_TRACE(TT_MD, it);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (leader) {
                if (kDown) {
                    tc_commit(&b->d_full[dsl]);
                } else {
                    tc_commit(&b->d_full[ds.s0]);
                    if (ds.two) tc_commit(&b->d_full[ds.s1]);
                }
            }
            __syncwarp();
            if (!kDown) {
                use[ds.s0]++;
                if (ds.two) use[ds.s1]++;
                sc += ds.two ? 2 : 1;
            }
        }
        if (leader) {
            if (!ok) tm_abort(abort, p.status);
            tc_commit(&b->drain[m]);
        }
        __syncwarp();
        int never = 0;
        mbar_wait(&b->drain[m], 0, &never);
    } else if (warp < kTmDeqWarps) {
        // dequant: set (warp >> 3) takes the K blocks of its parity; thread -> row r of matrix m
        const int set = warp >> 3, m = (warp >> 2) & 1, q = warp & 3, r = 32 * q + lane;
        const uint32_t code_off = m * kChunkBytes + r * 16;
        const uint32_t sb_off = m * kChunkBytes + kChunkCodes + 2 * r;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + 32u * m;
        const int mode_r = *p.mode_routed, mode_s = *p.mode_shared;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            const bool denorm = __all_sync(0xffffffffu, (p.tiles[tile].x < p.E ? mode_r : mode_s) == kScaleDenorm);
            for (int kb = 0; kb < KB; ++kb, ++it) {
                if ((int)(it & 1) != set) continue;
                const int cs = it % C::RC, as = it % C::A;
                const uint32_t g = it - C::A;   // the K block that last used this A slot
                const bool got = mbar_wait(&b->c_full[cs], (it / C::RC) & 1, abort) &&
                                 (it < (uint32_t)C::A || mbar_wait(&b->kb_done[g % kTmKD], (g / kTmKD) & 1, abort));
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (threadIdx.x == 0) TM_TRACE(TT_DW, it);
                const uint8_t* ch = cring + cs * C::CH;
                uint32_t v[32];
                if constexpr (kBf16) {   // already dequantised: this row's 64 bf16 weights
                    const uint4* src = reinterpret_cast<const uint4*>(ch + m * (kBf16PairBytes / 2)) + r;
#pragma unroll
                    for (int w4 = 0; w4 < 8; ++w4) {
                        const uint4 q4 = src[w4 * kTileRows];
                        v[4 * w4] = q4.x; v[4 * w4 + 1] = q4.y; v[4 * w4 + 2] = q4.z; v[4 * w4 + 3] = q4.w;
                    }
                } else {
                    const uint4 c0 = *reinterpret_cast<const uint4*>(ch + code_off);
                    const uint4 c1 = *reinterpret_cast<const uint4*>(ch + code_off + 2048);
                    const uint32_t s2 = *reinterpret_cast<const uint16_t*>(ch + sb_off) * 0x10001u;
                    const uint32_t b2 = *reinterpret_cast<const uint16_t*>(ch + sb_off + 256) * 0x10001u;
                    if (denorm) dequant_row64<true>(c0, c1, s2, b2, v);
                    else dequant_row64<false>(c0, c1, s2, b2, v);
                }
                __syncwarp();
                if (threadIdx.x == 0) TM_TRACE(TT_DD, it);
                // the dequantisation above consumed the words read from the slot; the bf16 path
                // only moves them, so it frees the slot once the store has read the registers
                if (!kBf16 && lane == 0) mbar_arrive(&b->c_empty[cs]);
                tc_fence_after();   // the MMAs that read this A slot before have completed
                tmem_st32(trow + 64u * as, v);
                tmem_st_wait();
                if constexpr (kBf16) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&b->c_empty[cs]);
                }
                if (threadIdx.x == 0) TM_TRACE(TT_DS, it);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&b->ready[it % kTmKD]);
            }
        }
        if (!ok && lane == 0) tm_abort(abort, p.status);
    } else if (warp < kTmCodeWarp) {
        // epilogue: thread -> weight row r of D_0 and D_1 (TMEM lane quadrant warp & 3); warp
        // group `half` takes the 16-token column groups of its parity.  32 tokens at a time are
        // staged token-major in shared memory, then written out: h with 16-byte stores by all
        // epilogue threads; weight * y as one bulk copy (the chunk's 32 rows of one 256-column
        // tile of Y are one contiguous block).
        const int q = warp & 3, half = (warp - kTmEpiWarp0) >> 2, r = 32 * q + lane, et = threadIdx.x - kTmEpiWarp0 * 32;
        uint8_t* stage = smem + C::stage_off;
        float* s_w = reinterpret_cast<float*>(smem + C::tab_off);          // [2][128]
        int* s_tok = reinterpret_cast<int*>(smem + C::tab_off + 1024);     // [2][128]
        const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16);
        const size_t yrows = (size_t)(p.k + 1) * p.T;
        uint32_t tcount = 0, chunk = 0, sc = 0, use[3] = {0, 0, 0};
        uint32_t hist = 0;   // down: bit i = this lane committed a bulk operation i + 1 chunks ago
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x, ++tcount) {
            const int4 t = p.tiles[tile];
            const int e = t.x, row0 = t.y, rows = t.z, wt = t.w, N = tile_n(rows);
            const size_t orow0 = e < p.E ? (size_t)row0 : (size_t)p.k * p.T + row0;   // row of H / Y
            if (kDown && et < rows) {
                // tables of this tile, double-buffered by tile parity: the previous tile's last
                // bulk issues (after its last barrier) may still read the other half
                const int asg = e < p.E ? p.perm[row0 + et] : 0;
                s_w[128 * (tcount & 1) + et] = e < p.E ? p.topk_w[asg] : 1.0f;
                s_tok[128 * (tcount & 1) + et] = e < p.E ? asg / p.k : row0 + et;
            }
            if (!kDown) {
                const DSlots ds = d_slots(sc, N, false);
                bool failed = false;
                if (et == 0 && (!mbar_wait(&b->d_full[ds.s0], use[ds.s0] & 1, abort) ||
                                (ds.two && !mbar_wait(&b->d_full[ds.s1], use[ds.s1] & 1, abort)))) {
                    tm_abort(abort, p.status);
                    failed = true;
                }
                // one decision for all epilogue warps (see named_bar_or)
                if (named_bar_or(2, kTmEpiThreads, failed || *abort != 0)) { ok = false; break; }
                tc_fence_after();
                const uint32_t td0 = tlane + ds.col0, td1 = tlane + ds.col1;   // this lane quadrant's D_0, D_1
                if (et == 0) TM_TRACE(TT_ET, tcount);
                for (int c0 = 0; c0 < N; c0 += 32) {
                    const int c = c0 + 16 * half;          // this warp's 16 tokens: c .. c+15
                    const bool last = c0 + 32 >= N;
                    uint16_t* st = reinterpret_cast<uint16_t*>(stage);   // [32][hi 128 | lo 128]
                    uint32_t G[16], U[16];
                    if (c < N) {
                        tmem_ld16(td0 + c, G);
                        tmem_ld16(td1 + c, U);
                        tmem_ld_wait();
                    }
                    if (last) {   // D is no longer read: the next tile's MMAs may start
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&b->d_empty[ds.s0]);
                            if (ds.two) mbar_arrive(&b->d_empty[ds.s1]);
                        }
                    }
                    if (c < N) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float gv = __uint_as_float(G[u]), uv = __uint_as_float(U[u]);
                            const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            const uint16_t hi = f32_to_bf16_rn(h);
                            const int n = 16 * half + u;
                            st[n * 256 + r] = hi;
                            st[n * 256 + 128 + r] = f32_to_bf16_rn(h - __uint_as_float((uint32_t)hi << 16));
                        }
                    }
                    named_bar_sync(2, kTmEpiThreads);
                    // tokens c0 .. c0+31: 32 pieces of 16 bytes each (16 hi, 16 lo)
                    for (int pi = et; pi < 32 * 32; pi += kTmEpiThreads) {
                        const int n = pi >> 5, pc = pi & 31, tok = c0 + n;
                        if (tok < rows) {
                            const int col = (pc < 16 ? 0 : p.I - 128) + wt * 128 + 8 * pc;
                            *reinterpret_cast<uint4*>(p.H + (orow0 + tok) * 2 * p.I + col) =
                                *reinterpret_cast<const uint4*>(st + n * 256 + 8 * pc);
                        }
                    }
                    named_bar_sync(2, kTmEpiThreads);
                }
                use[ds.s0]++;
                if (ds.two) use[ds.s1]++;
                sc += ds.two ? 2 : 1;
            } else {
                // down: wait for both accumulators of the tile (matrices m = 0, 1: output rows
                // 256 wt + 128 m ..), then per chunk of 32 tokens: weight * y of both matrices from
                // TMEM into a staging buffer [32][256] (a token's 256 outputs contiguous), one
                // barrier, and one 1 KB bulk reduce-add per token (or one row copy per chunk).  The
                // two slots are released once their last chunk has been read; the next chunk's TMEM
                // loads are issued before the barrier, so their latency overlaps the barrier and the
                // bulk issues.  A staging buffer is written again NSTG chunks later: before each
                // barrier the issuing lanes wait until their operations of NSTG - 1 chunks back have
                // read it.
                if (et == 0) TM_TRACE(TT_ET, tcount);
                const bool stacked = down_stacked(N);   // the lo half's products sit N columns further
                const float* tw = s_w + 128 * (tcount & 1);
                const int* ttok = s_tok + 128 * (tcount & 1);
                const int n_me = (warp - kTmEpiWarp0) + 8 * lane;   // reduce-adds: this lane's token
                const uint32_t j0 = 2 * tcount;   // uses j0, j0 + 1 of the slot ring: slot j % 4, phase j / 4
                const int sl0 = (int)(j0 % 4), sl1 = (int)((j0 + 1) % 4);
                bool failed = false;
                if (et == 0 && (!mbar_wait(&b->d_full[sl0], (j0 / 4) & 1, abort) ||
                                !mbar_wait(&b->d_full[sl1], ((j0 + 1) / 4) & 1, abort))) {
                    tm_abort(abort, p.status);
                    failed = true;
                }
                // (also: the weight / token tables are written); one decision for all warps
                if (named_bar_or(2, kTmEpiThreads, failed || *abort != 0)) { ok = false; break; }
                tc_fence_after();
                const uint32_t td0 = tlane + C::DCOL0 + C::DW * sl0, td1 = tlane + C::DCOL0 + C::DW * sl1;
                uint32_t R0[16], R1[16];
                if (16 * half < N) {
                    tmem_ld16(td0 + 16 * half, R0);
                    tmem_ld16(td1 + 16 * half, R1);
                    if (stacked) {   // one chunk: y = hi products + lo products, summed right away
                        uint32_t L[16];
                        tmem_ld16(td0 + N + 16 * half, L);
                        tmem_ld_wait_regs(R0);
                        tmem_ld_wait_regs(L);
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            R0[u] = __float_as_uint(__uint_as_float(R0[u]) + __uint_as_float(L[u]));
                        tmem_ld16(td1 + N + 16 * half, L);
                        tmem_ld_wait_regs(R1);
                        tmem_ld_wait_regs(L);
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            R1[u] = __float_as_uint(__uint_as_float(R1[u]) + __uint_as_float(L[u]));
                    }
                }
                for (int c0 = 0; c0 < N; c0 += 32, ++chunk) {
                    const int c = c0 + 16 * half;          // this warp's 16 tokens: c .. c+15
                    const bool last = c0 + 32 >= N;
                    float* st = reinterpret_cast<float*>(stage) + (chunk % C::NSTG) * (32 * 256);   // [32][256]
                    if (c < N && !stacked) {
                        tmem_ld_wait_regs(R0);
                        tmem_ld_wait_regs(R1);
                    }
                    if (last) {   // both accumulators are no longer read: their slots are free
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&b->d_empty[sl0]);
                            mbar_arrive(&b->d_empty[sl1]);
                        }
                    }
                    if (c < N) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float w = c + u < rows ? tw[c + u] : 0.0f;
                            st[(16 * half + u) * 256 + r] = w * __uint_as_float(R0[u]);
                            st[(16 * half + u) * 256 + 128 + r] = w * __uint_as_float(R1[u]);
                        }
                    }
                    if (c + 32 < N) {   // the next chunk (never stacked)
                        tmem_ld16(td0 + c + 32, R0);
                        tmem_ld16(td1 + c + 32, R1);
                    }
                    fence_proxy_async_smem();
                    const int nv = rows - c0 < 32 ? rows - c0 : 32;   // rows of this chunk
                    if (p.rows_out ? et < 2 : lane < 4) {   // issuing lanes: chunk - (NSTG - 1) has been read
                        const int pend = __popc(hist & C::HIST_MASK);
                        if (pend >= 2) bulk_wait_read<2>();
                        else if (pend == 1) bulk_wait_read<1>();
                        else bulk_wait_read<0>();
                    }
                    named_bar_sync(2, kTmEpiThreads);
                    uint32_t issued = 0;
                    if (p.rows_out) {
                        // rows of Y [d/128][(k+1)T][128]: the chunk's rows of one 128-column tile are
                        // one contiguous block (thread et = matrix m copies its half of the staging);
                        // the staging rows hold 256 floats, so the copy runs row by row
                        if (et < 2) {
                            float* ydst = p.Y + ((size_t)(2 * wt + et) * yrows + orow0 + c0) * 128;
                            for (int n = 0; n < nv; ++n) bulk_s2g(ydst + (size_t)n * 128, st + n * 256 + 128 * et, 512);
                            bulk_commit();
                            issued = 1;
                        }
                    } else if (lane < 4 && n_me < nv) {
                        // token n = (epilogue warp) + 8 lane: its 1 KB row piece added into acc; the
                        // issues are spread over the eight warps
                        bulk_reduce_add_f32(p.acc + (size_t)ttok[c0 + n_me] * p.d + (size_t)wt * 256, st + n_me * 256, 1024);
                        bulk_commit();
                        issued = 1;
                    }
                    hist = (hist << 1) | issued;
                }
            }
            if (et == 0) TM_TRACE(TT_ED, tcount);
        }
        if (!ok && lane == 0) tm_abort(abort, p.status);
        if (kDown && (et == 0 || lane < 4)) bulk_wait0();   // every bulk copy / reduce-add has completed
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTmMmaWarp) tmem_dealloc(tmem, 512);
}

// y[t] = bf16( sum_j Y[pos[t k + j]] + Y[k T + t] ), j = 0..k-1 in order, then the shared row;
// Y is [d/128][(k+1)T][128]; one thread per 4 columns of a token (16-byte loads, 8-byte store).
__global__ void combine_rows_kernel(const float4* __restrict__ Y, const int32_t* __restrict__ pos,
                                    uint2* __restrict__ y, int T, int d4, int k) {
    const size_t n = (size_t)T * d4, tile4 = (size_t)(k + 1) * T * 32;   // float4s of a 128-column tile
    pdl_wait();
    pdl_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / d4), c = (int)(i % d4);
        const float4* Yc = Y + (size_t)(c >> 5) * tile4 + (c & 31);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float4 v = __ldcs(Yc + (size_t)pos[(size_t)t * k + j] * 32);
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        const float4 v = __ldcs(Yc + ((size_t)k * T + t) * 32);
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        y[i] = make_uint2((uint32_t)f32_to_bf16_rn(s.x) | ((uint32_t)f32_to_bf16_rn(s.y) << 16),
                          (uint32_t)f32_to_bf16_rn(s.z) | ((uint32_t)f32_to_bf16_rn(s.w) << 16));
    }
}

TmParams make_tm_params(const FfnArgs& a, bool gate_up) {
    TmParams p{};
    // packed buffer: header, gate/up pairs, down pairs
    const size_t gu_bytes = (size_t)(a.I / kTileRows) * (a.d / kBK) * kChunkPairBytes;
    p.w_routed = a.w_routed + kPackHeader + (gate_up ? 0 : (size_t)a.E * gu_bytes);
    p.w_shared = a.w_shared + kPackHeader + (gate_up ? 0 : gu_bytes);
    p.mode_routed = reinterpret_cast<const int*>(a.w_routed);
    p.mode_shared = reinterpret_cast<const int*>(a.w_shared);
    p.tiles = reinterpret_cast<const int4*>(a.ws + (gate_up ? a.L.gu_tiles : a.L.dn_tiles));
    p.num_tiles = reinterpret_cast<const int*>(a.ws + (gate_up ? a.L.gu_num : a.L.dn_num));
    p.H = reinterpret_cast<uint16_t*>(a.ws + a.L.H);
    p.Y = reinterpret_cast<float*>(a.ws + a.L.Y);
    p.acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    p.rows_out = a.rows_out ? 1 : 0;
    p.perm = a.perm;
    p.topk_w = a.topk_w;
    p.status = reinterpret_cast<int*>(a.ws + a.L.status);
#ifdef MOE_TRACE
    p.trace = reinterpret_cast<unsigned long long*>(a.ws + a.L.trace);
#endif
    p.T = a.T; p.d = a.d; p.I = a.I; p.E = a.E; p.k = a.k;
    return p;
}

template <bool kDown, bool kBf16>
cudaError_t set_tm_smem_attr() {
    static bool done = false;
    if (done) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(ffn_tm_kernel<kDown, kBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           tm_smem_bytes<kDown, kBf16>());
    if (err == cudaSuccess) done = true;
    return err;
}

// bf16-weight ablation ("dequantise, then multiply" as separate passes): every chunk pair of
// a packed section dequantised to bf16 in the ring-chunk layout of the bf16 kernels, with the
// fused kernels' exact dequantisation (so the same bf16 weights); one thread per (pair,
// matrix, row), 16-byte stores that are contiguous across rows.
__global__ void __launch_bounds__(256) dequant_pairs_kernel(const uint8_t* __restrict__ src, size_t npairs,
                                                            const int* __restrict__ mode, uint8_t* __restrict__ dst) {
    pdl_wait();
    pdl_launch_dependents();
    const bool denorm = *mode == kScaleDenorm;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < npairs * 256; i += (size_t)gridDim.x * blockDim.x) {
        const size_t pair = i >> 8;
        const int m = (int)(i >> 7) & 1, r = (int)i & 127;
        const uint8_t* ch = src + pair * kChunkPairBytes + m * kChunkBytes;
        const uint4 c0 = *reinterpret_cast<const uint4*>(ch + r * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(ch + r * 16 + 2048);
        const uint32_t s2 = *reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 2 * r) * 0x10001u;
        const uint32_t b2 = *reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 256 + 2 * r) * 0x10001u;
        uint32_t v[32];
        if (denorm) dequant_row64<true>(c0, c1, s2, b2, v);
        else dequant_row64<false>(c0, c1, s2, b2, v);
        uint4* o = reinterpret_cast<uint4*>(dst + pair * kBf16PairBytes + m * (kBf16PairBytes / 2)) + r;
#pragma unroll
        for (int w4 = 0; w4 < 8; ++w4) o[w4 * kTileRows] = make_uint4(v[4 * w4], v[4 * w4 + 1], v[4 * w4 + 2], v[4 * w4 + 3]);
    }
}

cudaError_t launch_dequant_pairs(const uint8_t* packed, size_t first_pair, size_t npairs, uint8_t* dst,
                                 cudaStream_t st, unsigned long long* launches) {
    const size_t threads = npairs * 256;
    const int blocks = (int)((threads + 255) / 256 < 8192 ? (threads + 255) / 256 : 8192);
    *launches += 1;
    return launch_with_pdl(dequant_pairs_kernel, dim3(blocks), dim3(256), 0, st,
                           packed + kPackHeader + first_pair * kChunkPairBytes, npairs,
                           reinterpret_cast<const int*>(packed), dst);
}

// chunk pairs per expert of a packed buffer: gate/up section, then down section
size_t gu_pairs(const FfnArgs& a) { return (size_t)(a.I / kTileRows) * (a.d / kBK); }
size_t dn_pairs(const FfnArgs& a) { return (size_t)(a.d / 256) * (a.I / kBK); }

// bf16-weight ablation: dequantise one section (gate/up or down) of the routed and the shared
// buffer into the workspace, then point the kernel's weight bases there
cudaError_t unfused_prepare(const FfnArgs& a, bool gate_up, TmParams& p, cudaStream_t st,
                            unsigned long long* launches) {
    const size_t gu = gu_pairs(a), dn = dn_pairs(a), all = gu + dn;
    uint8_t* wbf = a.ws + a.L.wbf;
    uint8_t* routed = wbf + (gate_up ? 0 : (size_t)a.E * gu * kBf16PairBytes);
    uint8_t* shared = wbf + ((size_t)a.E * all + (gate_up ? 0 : gu)) * kBf16PairBytes;
    cudaError_t err = launch_dequant_pairs(a.w_routed, gate_up ? 0 : (size_t)a.E * gu, (size_t)a.E * (gate_up ? gu : dn),
                                           routed, st, launches);
    if (err == cudaSuccess)
        err = launch_dequant_pairs(a.w_shared, gate_up ? 0 : gu, gate_up ? gu : dn, shared, st, launches);
    p.w_routed = routed;
    p.w_shared = shared;
    return err;
}

}  // namespace

cudaError_t launch_gate_up_tm(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaError_t err = a.unfused ? set_tm_smem_attr<false, true>() : set_tm_smem_attr<false, false>();
    if (err != cudaSuccess) return err;
    CUtensorMap tm_xs, tm_xsl, tm_x, tm_xl;
    err = make_tmap_bf16_2d(&tm_xs, a.ws + a.L.xs, (uint64_t)a.k * a.T, a.d, (uint64_t)a.d * 2, kBK, kTmBox);
    if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&tm_xsl, a.ws + a.L.xs, (uint64_t)a.k * a.T, a.d, (uint64_t)a.d * 2, kBK, kTmBoxL);
    if (err == cudaSuccess) err = make_tmap_bf16_2d(&tm_x, a.x, a.T, a.d, (uint64_t)a.d * 2, kBK, kTmBox);
    if (err == cudaSuccess) err = make_tmap_bf16_2d(&tm_xl, a.x, a.T, a.d, (uint64_t)a.d * 2, kBK, kTmBoxL);
    if (err != cudaSuccess) return err;
    TmParams p = make_tm_params(a, true);
    if (a.unfused) {
        if ((err = unfused_prepare(a, true, p, st, launches)) != cudaSuccess) return err;
        *launches += 1;
        return launch_with_pdl(ffn_tm_kernel<false, true>, dim3(a.num_sms), dim3(kTmThreads),
                               tm_smem_bytes<false, true>(), st, tm_xs, tm_xsl, tm_x, tm_xl, p);
    }
    *launches += 1;
    return launch_with_pdl(ffn_tm_kernel<false, false>, dim3(a.num_sms), dim3(kTmThreads), tm_smem_bytes<false>(), st,
                           tm_xs, tm_xsl, tm_x, tm_xl, p);
}

cudaError_t launch_down_tm(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaError_t err = a.unfused ? set_tm_smem_attr<true, true>() : set_tm_smem_attr<true, false>();
    if (err != cudaSuccess) return err;
    CUtensorMap tm_h, tm_hl;
    err = make_tmap_bf16_2d(&tm_h, a.ws + a.L.H, (uint64_t)(a.k + 1) * a.T, 2 * (uint64_t)a.I, (uint64_t)a.I * 4,
                            kBK, kTmBox);
    if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&tm_hl, a.ws + a.L.H, (uint64_t)(a.k + 1) * a.T, 2 * (uint64_t)a.I,
                                (uint64_t)a.I * 4, kBK, kTmBoxL);
    if (err != cudaSuccess) return err;
    TmParams p = make_tm_params(a, false);
    if (a.unfused) {
        if ((err = unfused_prepare(a, false, p, st, launches)) != cudaSuccess) return err;
        *launches += 1;
        return launch_with_pdl(ffn_tm_kernel<true, true>, dim3(a.num_sms), dim3(kTmThreads), tm_smem_bytes<true, true>(),
                               st, tm_h, tm_hl, tm_h, tm_hl, p);
    }
    *launches += 1;
    return launch_with_pdl(ffn_tm_kernel<true, false>, dim3(a.num_sms), dim3(kTmThreads), tm_smem_bytes<true>(), st,
                           tm_h, tm_hl, tm_h, tm_hl, p);
}

}  // namespace moe

namespace moe {
cudaError_t launch_combine_rows(int T, int d, int k, const float* Y, const int32_t* pos, uint16_t* y, cudaStream_t st,
                                unsigned long long* launches) {
    const size_t n = (size_t)T * (d / 4);
    const int blocks = (int)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
    *launches += 1;
    return launch_with_pdl(combine_rows_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const float4*>(Y), pos,
                           reinterpret_cast<uint2*>(y), T, d / 4, k);
}
}  // namespace moe

// ======================================================================================
// combine of the decode kernels' fp32 token-order sum (and of large prefill chunks):
// y = bf16(sum), and the sum is left at zero (the one-launch decode kernel relies on that)
// ======================================================================================
namespace moe {
namespace {
__global__ void combine_kernel(float4* __restrict__ acc, uint2* __restrict__ y, size_t n4) {
    pdl_wait();
    pdl_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[i];
        y[i] = make_uint2((uint32_t)f32_to_bf16_rn(v.x) | ((uint32_t)f32_to_bf16_rn(v.y) << 16),
                          (uint32_t)f32_to_bf16_rn(v.z) | ((uint32_t)f32_to_bf16_rn(v.w) << 16));
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
}  // namespace

cudaError_t launch_combine(int T, int d, const float* acc, uint16_t* y, cudaStream_t st, unsigned long long* launches) {
    const size_t n4 = (size_t)T * d / 4;
    const int blocks = (int)((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
    *launches += 1;
    return launch_with_pdl(combine_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<float4*>(const_cast<float*>(acc)),
                           reinterpret_cast<uint2*>(y), n4);
}
}  // namespace moe
