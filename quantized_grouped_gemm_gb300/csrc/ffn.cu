// ffn.cu -- grouped SwiGLU FFN over packed 4-bit group-affine weights, sm_103a tcgen05.
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026), section "Dequantize
// weights during matrix multiplication": the grouped GEMM rebuilds one small bf16 weight tile
// at a time in on-chip memory, multiplies it with the routed activation rows, accumulates in
// fp32 and writes bf16; the expanded weight matrix never exists in memory.  Section "Reduce
// intermediate and state traffic": gate/up projections fused with the gated activation; the
// output projection fused with the routing score and the shared-expert result.
//
// GB300 design: one persistent CTA per SM; a tile is (expert, block of <= 128 token rows,
// 256-row weight tile).  Each tcgen05.mma is M = 128 token rows x N = 256 weight rows x K = 16:
//   gate/up  N = 128 gate rows + the same 128 up rows, so one accumulator row holds g and u of
//            the token for 128 values of i;
//   down     N = 256 rows of d; K runs over the hi half of h, then its lo half (h is carried to
//            16 bits as a bf16 pair).
// Warp roles (22 warps):
//   warps 0-15  dequant: packed chunk pair (smem) -> bf16 B tile (256 rows x 64) in the 128-byte
//               swizzled K-major layout the tensor core reads; w = fma.rn.bf16x2(q, scale, bias)
//   warps 16-19 epilogue: TMEM -> registers; one token row per thread
//   warp 20     producer: cp.async.bulk of 9216-byte weight pairs, TMA tiles of activations
//   warp 21     MMA issuer (one thread) and TMEM owner (2 accumulators of 256 columns)
// All waits are bounded (MOE_STATUS_TIMEOUT, then the CTA unwinds).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kDeqWarps = 16;
constexpr int kEpiWarps = 4;
constexpr int kProdWarp = kDeqWarps + kEpiWarps;   // 20
constexpr int kMmaWarp = kProdWarp + 1;            // 21
constexpr int kThreads = (kMmaWarp + 1) * 32;      // 704

constexpr int kTokRows = 128;                      // MMA M: token rows of a tile
constexpr int kWRows = 256;                        // MMA N: weight rows of a tile
constexpr int kActBytes = kTokRows * 128;          // 128 rows x 64 bf16 (one K block)
constexpr int kWdqBytes = kWRows * 128;            // 256 rows x 64 bf16
constexpr int kRawBytes = kChunkPairBytes;         // 9216
constexpr int kEpiRows = kEpiWarps * 32;           // token rows of the epilogue (one per thread)
constexpr int kStageStride = 64 * 4 + 16;          // 64 fp32 + 16 bytes of padding (bank spread)

#ifndef MOE_GU_RAW
#define MOE_GU_RAW 4
#endif
#ifndef MOE_GU_WDQ
#define MOE_GU_WDQ 4
#endif
#ifndef MOE_GU_ACT
#define MOE_GU_ACT 3
#endif
#ifndef MOE_DN_RAW
#define MOE_DN_RAW 3
#endif
#ifndef MOE_DN_WDQ
#define MOE_DN_WDQ 3
#endif
#ifndef MOE_DN_ACT
#define MOE_DN_ACT 4
#endif
template <bool kDown>
struct Cfg {
    static constexpr int RAW = kDown ? MOE_DN_RAW : MOE_GU_RAW;   // weight-pair ring (HBM -> smem)
    static constexpr int WDQ = kDown ? MOE_DN_WDQ : MOE_GU_WDQ;   // dequantised weight ring
    static constexpr int ACT = kDown ? MOE_DN_ACT : MOE_GU_ACT;   // activation ring (TMA)
    static constexpr int PARTS = kDown ? 2 : 1;    // activation K steps per weight K block
    static constexpr int act_off = 0;
    static constexpr int wdq_off = act_off + ACT * kActBytes;
    static constexpr int raw_off = wdq_off + WDQ * kWdqBytes;
    // down: epilogue staging of 64 output columns per token row (row stride 272 bytes)
    static constexpr int stage_off = raw_off + RAW * kRawBytes;
    static constexpr int stage_bytes = kDown ? kEpiRows * kStageStride : 0;
    static constexpr int bar_off = stage_off + stage_bytes;
};

struct Bars {
    uint64_t raw_full[8], raw_empty[8], act_full[8], act_empty[8], wdq_full[6], wdq_empty[6];
    uint64_t tm_full[2], tm_empty[2], drain;
    uint32_t tmem_slot;
    int abort;
};

template <bool kDown>
constexpr int smem_bytes() {
    return Cfg<kDown>::bar_off + (int)sizeof(Bars) + 1024;   // + alignment slack
}
static_assert(smem_bytes<false>() <= 232448, "gate/up smem");
static_assert(smem_bytes<true>() <= 232448, "down smem");

// Weight chunks come from HBM and run up to RAW K blocks ahead of the activation tiles.
// No deadlock: a wait on raw_empty for K block g needs the MMA of K block g - RAW - WDQ,
// whose activation tiles were issued earlier.

#ifdef MOE_TRACE
constexpr int kTraceK = 96;
#define TRACE(ev, g)                                                                     \
    do {                                                                                 \
        if (blockIdx.x == 0 && (g) < kTraceK) p.trace[(ev) * kTraceK + (g)] = clock64(); \
    } while (0)
#else
#define TRACE(ev, g) \
    do {             \
    } while (0)
#endif
enum { TR_PRAW = 0, TR_PACT, TR_DWAIT, TR_DDONE, TR_MWAIT, TR_MDONE, TR_ETILE, TR_EDONE, TR_N };

struct FfnParams {
    const uint8_t* w_routed;   // packed stack: [E][tiles][K/64][2][4608]
    const uint8_t* w_shared;
    const int* mode_routed;    // scale encoding of each packed buffer (header word)
    const int* mode_shared;
    const int4* tiles;         // (expert, first row, rows, weight tile); expert == E: shared
    const int* num_tiles;
    uint16_t* H;               // [(k+1)T][2I] bf16, hi | lo
    float* acc;                // [T][d] fp32 token-order sum
    const int32_t* perm;
    const float* topk_w;
    int* status;
    unsigned long long* trace;
    int T, d, I, E, k;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}

__device__ __forceinline__ void raise_abort(volatile int* abort, int* status) {
    *abort = 1;
    set_status(status, MOE_STATUS_TIMEOUT);
}

// Wait (bounded, not cut short by the abort flag) until the last `depth` arms of a ring's
// full barriers have landed, so no bulk copy is still writing shared memory at exit.
__device__ void drain_ring(uint64_t* full, int depth, uint32_t issued) {
    int never = 0;
    const uint32_t first = issued > (uint32_t)depth ? issued - depth : 0;
    for (uint32_t i = first; i < issued; ++i) mbar_wait(&full[i % depth], (i / depth) & 1, &never);
}

// Walks this CTA's (tile, K block, part) sequence.
struct Cursor {
    int tile, kb, part, num, KB, parts;
    int4 t;
    const int4* tiles;
    __device__ __forceinline__ void init(const int4* tl, int n, int kbs, int nparts) {
        tiles = tl; num = n; KB = kbs; parts = nparts;
        tile = blockIdx.x; kb = 0; part = 0;
        if (tile < num) t = tiles[tile];
    }
    __device__ __forceinline__ bool done() const { return tile >= num; }
    __device__ __forceinline__ void next() {
        if (++part < parts) return;
        part = 0;
        if (++kb < KB) return;
        kb = 0;
        tile += gridDim.x;
        if (tile < num) t = tiles[tile];
    }
};

// -------- dequant of 32 weights (one half row of a packed chunk) into the swizzled layout ----
template <bool kDenorm>
__device__ __forceinline__ void dequant_store4(uint4 codes, uint32_t s2, uint32_t b2, uint8_t* row_dst, int r,
                                               int c0) {
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t v[4];
        dequant_word<kDenorm>(words[q], s2, b2, v);
        const int c = c0 + q;
        const uint32_t addr = smem_u32(row_dst + ((c ^ (r & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                     "r"(v[3])
                     : "memory");
    }
}

// Bulk add of `bytes` fp32 from shared memory into global memory (TMA reduction; 16-byte
// aligned addresses, bytes % 16 == 0); completion tracked per thread by bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    return (uint32_t)f32_to_bf16_rn(a) | ((uint32_t)f32_to_bf16_rn(b) << 16);
}

// ======================================================================================
// The kernel: kDown == false -> gate/up + SwiGLU into h; true -> down + weighted fp32 sums.
// tm_a: activations of routed rows (xs for gate/up, h for down); tm_b: the shared expert's
// activation rows (x for gate/up; unused for down, whose shared rows follow in h).
// ======================================================================================
template <bool kDown>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, FfnParams p) {
    using C = Cfg<kDown>;
    extern __shared__ uint8_t smem_dyn[];
    const int num = *p.num_tiles;
    if ((int)blockIdx.x >= num) return;
    uint8_t* smem = align1024(smem_dyn);
    uint8_t* act = smem + C::act_off;
    uint8_t* wdq = smem + C::wdq_off;
    uint8_t* raw = smem + C::raw_off;
    Bars* bars = reinterpret_cast<Bars*>(smem + C::bar_off);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = (kDown ? p.I : p.d) / kBK;                  // weight K blocks
    const int WT = (kDown ? p.d : p.I * 2) / kWRows;          // weight tiles per expert

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::RAW; ++i) { mbar_init(&bars->raw_full[i], 1); mbar_init(&bars->raw_empty[i], kDeqWarps); }
        for (int i = 0; i < C::ACT; ++i) { mbar_init(&bars->act_full[i], 1); mbar_init(&bars->act_empty[i], 1); }
        for (int i = 0; i < C::WDQ; ++i) { mbar_init(&bars->wdq_full[i], kDeqWarps); mbar_init(&bars->wdq_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bars->tm_full[i], 1); mbar_init(&bars->tm_empty[i], kEpiWarps); }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kProdWarp && lane == 0) { prefetch_tmap(&tm_a); if (!kDown) prefetch_tmap(&tm_b); }
    if (warp == kMmaWarp) { tmem_alloc(&bars->tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    if (warp == kProdWarp) {
        if (lane == 0) {
            uint32_t rit = 0, ait = 0;
            bool ok = true;
            Cursor cr, ca;
            cr.init(p.tiles, num, KB, 1);
            ca.init(p.tiles, num, KB, C::PARTS);
            while (ok && !ca.done()) {
                while (ok && !cr.done() && rit < ait / C::PARTS + C::RAW) {
                    const int e = cr.t.x, wt = cr.t.w;
                    const uint8_t* w = (e < p.E ? p.w_routed + (size_t)(e * WT + wt) * KB * kRawBytes
                                                : p.w_shared + (size_t)wt * KB * kRawBytes) +
                                       (size_t)cr.kb * kRawBytes;
                    const int rs = rit % C::RAW;
                    if (!mbar_wait(&bars->raw_empty[rs], ((rit / C::RAW) & 1) ^ 1, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars->raw_full[rs], kRawBytes);
                    bulk_g2s(raw + rs * kRawBytes, w, kRawBytes, &bars->raw_full[rs]);
                    TRACE(TR_PRAW, rit);
                    ++rit;
                    cr.next();
                }
                if (!ok) break;
                const int e = ca.t.x, row0 = ca.t.y;
                const int as = ait % C::ACT;
                if (!mbar_wait(&bars->act_empty[as], ((ait / C::ACT) & 1) ^ 1, abort)) { ok = false; break; }
                mbar_arrive_expect_tx(&bars->act_full[as], kActBytes);
                if (kDown) {
                    const int hrow0 = e < p.E ? row0 : p.k * p.T + row0;
                    tma_load_2d(act + as * kActBytes, &tm_a, ca.part * p.I + ca.kb * kBK, hrow0, &bars->act_full[as]);
                } else {
                    tma_load_2d(act + as * kActBytes, e < p.E ? &tm_a : &tm_b, ca.kb * kBK, row0, &bars->act_full[as]);
                }
                TRACE(TR_PACT, ait);
                ++ait;
                ca.next();
            }
            if (!ok) raise_abort(abort, p.status);
            drain_ring(bars->raw_full, C::RAW, rit);
            drain_ring(bars->act_full, C::ACT, ait);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            uint32_t wit = 0, ait = 0, tcount = 0;
            uint32_t use[2] = {0, 0};
            bool ok = true;
            const uint32_t act_base = smem_u32(act), wdq_base = smem_u32(wdq);
            const uint32_t idesc = idesc_bf16_f32(kTokRows, kWRows);
            for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x, ++tcount) {
                const int buf = tcount & 1;
                if (!mbar_wait(&bars->tm_empty[buf], (use[buf] & 1) ^ 1, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t dcol = tmem + 256u * buf;
                for (int kb = 0; kb < KB && ok; ++kb) {
                    const int ws = wit % C::WDQ;
                    if (!mbar_wait(&bars->wdq_full[ws], (wit / C::WDQ) & 1, abort)) { ok = false; break; }
                    TRACE(TR_MWAIT, wit);
                    for (int part = 0; part < C::PARTS; ++part) {
                        const int as = ait % C::ACT;
                        if (!mbar_wait(&bars->act_full[as], (ait / C::ACT) & 1, abort)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t ad = sw128_desc(act_base + as * kActBytes + ks * 32);
                            const uint64_t bd = sw128_desc(wdq_base + ws * kWdqBytes + ks * 32);
                            tc_mma_bf16(dcol, ad, bd, idesc, (kb | part | ks) ? 1u : 0u);
                        }
                        tc_commit(&bars->act_empty[as]);
                        ++ait;
                    }
                    tc_commit(&bars->wdq_empty[ws]);
                    TRACE(TR_MDONE, wit);
                    ++wit;
                }
                if (!ok) break;
                tc_commit(&bars->tm_full[buf]);
                use[buf]++;
            }
            if (!ok) raise_abort(abort, p.status);
            tc_commit(&bars->drain);
            int never = 0;
            mbar_wait(&bars->drain, 0, &never);
        }
    } else if (warp < kDeqWarps) {
        // dequant: thread -> (weight row r of the 256-row tile, half hf); 32 weights per K block.
        // Rows 0..127 come from the first chunk of the pair, rows 128..255 from the second.
        // Every warp waits on its own (lock-stepping the 16 warps on a named barrier measured
        // slower: a warp may start the next K block while others finish this one).
        const int r = threadIdx.x & 255, hf = threadIdx.x >> 8;
        const int mat = r >> 7, rr = r & 127;
        const uint32_t code_off = mat * kChunkBytes + hf * 2048 + rr * 16;
        const uint32_t sb_off = mat * kChunkBytes + kChunkCodes + 2 * rr;
        const uint32_t row_off = (r >> 3) * 1024 + (r & 7) * 128;
        uint32_t rit = 0;
        bool ok = true;
        const int mode_r = *p.mode_routed, mode_s = *p.mode_shared;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            const bool denorm = (p.tiles[tile].x < p.E ? mode_r : mode_s) == kScaleDenorm;
            for (int kb = 0; kb < KB; ++kb) {
                const int rs = rit % C::RAW, ws = rit % C::WDQ;
                const bool got = mbar_wait(&bars->raw_full[rs], (rit / C::RAW) & 1, abort) &&
                                 mbar_wait(&bars->wdq_empty[ws], ((rit / C::WDQ) & 1) ^ 1, abort);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (threadIdx.x == 0) TRACE(TR_DWAIT, rit);
                const uint8_t* ch = raw + rs * kRawBytes;
                const uint4 cw = *reinterpret_cast<const uint4*>(ch + code_off);
                const uint32_t sv = *reinterpret_cast<const uint16_t*>(ch + sb_off);
                const uint32_t bv = *reinterpret_cast<const uint16_t*>(ch + sb_off + 256);
                if (denorm)
                    dequant_store4<true>(cw, sv * 0x10001u, bv * 0x10001u, wdq + ws * kWdqBytes + row_off, r, 4 * hf);
                else
                    dequant_store4<false>(cw, sv * 0x10001u, bv * 0x10001u, wdq + ws * kWdqBytes + row_off, r, 4 * hf);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) { mbar_arrive(&bars->raw_empty[rs]); mbar_arrive(&bars->wdq_full[ws]); }
                if (threadIdx.x == 0) TRACE(TR_DDONE, rit);
                ++rit;
            }
        }
        if (!ok && lane == 0) raise_abort(abort, p.status);
    } else {
        // epilogue: thread = token row (32 per warp, warp w % 4 = TMEM lane quadrant).  Its first
        // thread waits for the accumulator and releases the 4 warps through a named barrier.
        const int q = warp & 3;
        uint32_t use[2] = {0, 0}, tcount = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x, ++tcount) {
            const int4 t = p.tiles[tile];
            const int e = t.x, row0 = t.y, rows = t.z, wt = t.w;
            const int buf = tcount & 1;
            if (threadIdx.x == kDeqWarps * 32 && !mbar_wait(&bars->tm_full[buf], use[buf] & 1, abort))
                raise_abort(abort, p.status);
            named_bar_sync(2, kEpiWarps * 32);
            if (*abort) { ok = false; break; }
            tc_fence_after();
            if (warp == kDeqWarps && lane == 0) TRACE(TR_ETILE, tcount);
            const int tok = 32 * q + lane;                        // row within the tile
            const bool live = tok < rows;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + 256u * buf;
            if (!kDown) {
                // columns 0..127: g for i = 128*wt + c; columns 128..255: u for the same i
                const size_t hrow = e < p.E ? (size_t)row0 + tok : (size_t)p.k * p.T + row0 + tok;
                uint16_t* hp = p.H + hrow * 2 * p.I + (size_t)wt * 128;
                for (int c = 0; c < 8; ++c) {
                    uint32_t G[16], U[16];
                    tmem_ld16(taddr + 16 * c, G);
                    tmem_ld16(taddr + 128 + 16 * c, U);
                    tmem_ld_wait();
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {
                        float hv[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const float gv = __uint_as_float(G[jj + u]), uv = __uint_as_float(U[jj + u]);
                            hv[u] = gv / (1.0f + __expf(-gv)) * uv;
                        }
                        const uint32_t h2 = pack_bf16(hv[0], hv[1]);
                        hi[jj / 2] = h2;
                        lo[jj / 2] = pack_bf16(hv[0] - bf16lo(h2), hv[1] - bf16hi(h2));
                    }
                    if (live) {
                        uint4* dh = reinterpret_cast<uint4*>(hp + 16 * c);
                        uint4* dl = reinterpret_cast<uint4*>(hp + p.I + 16 * c);
                        dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                        dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                    }
                }
            } else {
                // 256 columns of d starting at 256*wt: acc[token][n] += w * y, 64 columns at a time
                // through the thread's staging row and one bulk reduce-add (TMA) per piece
                int tk = 0;
                float w = 0.f;
                if (live) {
                    if (e < p.E) {
                        const int asg = p.perm[row0 + tok];
                        tk = asg / p.k;
                        w = p.topk_w[asg];
                    } else {
                        tk = row0 + tok;
                        w = 1.0f;
                    }
                }
                float* ap = p.acc + (size_t)tk * p.d + (size_t)wt * kWRows;
                uint8_t* srow = smem + C::stage_off + (32 * q + lane) * kStageStride;
                for (int pc = 0; pc < 4; ++pc) {
                    bulk_wait_read0();   // the previous piece has left the staging row
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t Y[16];
                        tmem_ld16(taddr + 64 * pc + 16 * c, Y);
                        tmem_ld_wait();
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const uint32_t a = smem_u32(srow + 64 * c + 16 * v);
                            asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a),
                                         "f"(w * __uint_as_float(Y[4 * v])), "f"(w * __uint_as_float(Y[4 * v + 1])),
                                         "f"(w * __uint_as_float(Y[4 * v + 2])), "f"(w * __uint_as_float(Y[4 * v + 3]))
                                         : "memory");
                        }
                    }
                    fence_proxy_async_smem();
                    if (live) {
                        bulk_reduce_add_f32(ap + 64 * pc, srow, 256);
                        bulk_commit();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (warp == kDeqWarps && lane == 0) TRACE(TR_EDONE, tcount);
            if (lane == 0) mbar_arrive(&bars->tm_empty[buf]);
            use[buf]++;
        }
        if (!ok && lane == 0) raise_abort(abort, p.status);
        if (kDown) bulk_wait0();   // every bulk reduce-add of this thread has completed
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ======================================================================================
// combine: y = bf16(acc)
// ======================================================================================
// y = bf16(sum); the sum is left at zero (the one-launch decode kernel relies on that)
__global__ void combine_kernel(float4* __restrict__ acc, uint2* __restrict__ y, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[i];
        y[i] = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

FfnParams make_params(const FfnArgs& a, bool gate_up) {
    FfnParams p{};
    // packed buffer: header, gate/up pairs, down pairs
    const size_t gu_bytes = (size_t)(a.I / kTileRows) * (a.d / kBK) * kChunkPairBytes;
    p.w_routed = a.w_routed + kPackHeader + (gate_up ? 0 : (size_t)a.E * gu_bytes);
    p.w_shared = a.w_shared + kPackHeader + (gate_up ? 0 : gu_bytes);
    p.mode_routed = reinterpret_cast<const int*>(a.w_routed);
    p.mode_shared = reinterpret_cast<const int*>(a.w_shared);
    p.tiles = reinterpret_cast<const int4*>(a.ws + (gate_up ? a.L.gu_tiles : a.L.dn_tiles));
    p.num_tiles = reinterpret_cast<const int*>(a.ws + (gate_up ? a.L.gu_num : a.L.dn_num));
    p.H = reinterpret_cast<uint16_t*>(a.ws + a.L.H);
    p.acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    p.perm = a.perm;
    p.topk_w = a.topk_w;
    p.status = reinterpret_cast<int*>(a.ws + a.L.status);
#ifdef MOE_TRACE
    p.trace = reinterpret_cast<unsigned long long*>(a.ws + a.L.trace);
#endif
    p.T = a.T; p.d = a.d; p.I = a.I; p.E = a.E; p.k = a.k;
    return p;
}

template <bool kDown>
cudaError_t set_smem_attr() {
    static bool done = false;
    if (done) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(ffn_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           smem_bytes<kDown>());
    if (err == cudaSuccess) done = true;
    return err;
}

}  // namespace

cudaError_t launch_gate_up(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaError_t err = set_smem_attr<false>();
    if (err != cudaSuccess) return err;
    CUtensorMap tm_xs, tm_x;
    err = make_tmap_bf16_2d(&tm_xs, a.ws + a.L.xs, (uint64_t)a.k * a.T, a.d, (uint64_t)a.d * 2, kBK, kTokRows);
    if (err != cudaSuccess) return err;
    err = make_tmap_bf16_2d(&tm_x, a.x, a.T, a.d, (uint64_t)a.d * 2, kBK, kTokRows);
    if (err != cudaSuccess) return err;
    ffn_kernel<false><<<a.num_sms, kThreads, smem_bytes<false>(), st>>>(tm_xs, tm_x, make_params(a, true));
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_down(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaError_t err = set_smem_attr<true>();
    if (err != cudaSuccess) return err;
    CUtensorMap tm_h;
    err = make_tmap_bf16_2d(&tm_h, a.ws + a.L.H, (uint64_t)(a.k + 1) * a.T, 2 * (uint64_t)a.I, (uint64_t)a.I * 4,
                            kBK, kTokRows);
    if (err != cudaSuccess) return err;
    ffn_kernel<true><<<a.num_sms, kThreads, smem_bytes<true>(), st>>>(tm_h, tm_h, make_params(a, false));
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_combine(int T, int d, const float* acc, uint16_t* y, cudaStream_t st, unsigned long long* launches) {
    const size_t n4 = (size_t)T * d / 4;
    const int blocks = (int)((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
    combine_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<float4*>(const_cast<float*>(acc)), reinterpret_cast<uint2*>(y), n4);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
