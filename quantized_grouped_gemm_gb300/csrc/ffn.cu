// ffn.cu -- grouped SwiGLU FFN over packed 4-bit group-affine weights, sm_103a tcgen05.
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026), section "Dequantize
// weights during matrix multiplication": the grouped GEMM rebuilds one small bf16 weight tile
// at a time in on-chip memory, multiplies it with the routed activation rows, accumulates in
// fp32 and writes bf16; the expanded weight matrix never exists in memory.  Section "Reduce
// intermediate and state traffic": gate/up projections fused with the gated activation; the
// output projection fused with the routing score and the shared-expert result.
//
// GB300 design (one persistent CTA per SM, 18 warps):
//   warps 0-7   dequant: packed chunk (smem) -> bf16 A tile in the 128-byte-swizzled K-major
//               layout the tensor core reads (w = fma.rn.bf16x2(q, scale, bias): one rounding)
//   warps 8-15  epilogue: TMEM -> registers -> h (gate/up) or weighted fp32 adds (down)
//   warp 16     producer: cp.async.bulk of packed weight chunks, TMA tiles of activations
//   warp 17     MMA issuer (one thread) + TMEM owner
// Swap-AB: the weights are the M = 128 operand, the expert's token rows are N (16..256, in
// steps of 16, so small experts waste little), K steps of 64 = one quant group.
// All waits are bounded (MOE_STATUS_TIMEOUT, then the CTA unwinds).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 8;
constexpr int kProdWarp = kDeqWarps + kEpiWarps;   // 16
constexpr int kMmaWarp = kProdWarp + 1;            // 17
constexpr int kThreads = (kMmaWarp + 1) * 32;      // 576

constexpr int kBStageBytes = kMaxN * 128;          // 256 rows x 64 bf16
constexpr int kBoxRows = 64;
constexpr int kBoxBytes = kBoxRows * 128;
constexpr int kATileBytes = kTileRows * 128;       // 128 rows x 64 bf16

// gate/up ring depths
constexpr int kGuRaw = 6, kGuB = 3, kGuA = 2;
// down ring depths (B carries the hi and the lo half of h as separate K steps)
constexpr int kDnRaw = 6, kDnB = 4, kDnA = 2;

struct Bars {
    uint64_t raw_full[8], raw_empty[8], b_full[8], b_empty[8], a_full[4], a_empty[4];
    uint64_t tm_full[2], tm_empty[2], drain;
    uint32_t tmem_slot;
    int abort;
};

template <int RAW, int BST, int AST, int ABYTES, int RAWBYTES>
struct SmemPlan {
    static constexpr int b_off = 0;
    static constexpr int a_off = b_off + BST * kBStageBytes;
    static constexpr int raw_off = a_off + AST * ABYTES;
    static constexpr int bar_off = raw_off + RAW * RAWBYTES;
    static constexpr int bytes = bar_off + (int)sizeof(Bars) + 1024;   // + alignment slack
};
using GuPlan = SmemPlan<kGuRaw, kGuB, kGuA, 2 * kATileBytes, kChunkPairBytes>;
using DnPlan = SmemPlan<kDnRaw, kDnB, kDnA, kATileBytes, kChunkBytes>;
static_assert(GuPlan::bytes <= 232448, "gate/up smem");
static_assert(DnPlan::bytes <= 232448, "down smem");

struct FfnParams {
    const uint8_t* w_routed;   // packed stack (gate/up interleaved, or down)
    const uint8_t* w_shared;
    const int4* tiles;         // (expert, first row, rows, M tile); expert == E: shared
    const int* num_tiles;
    uint16_t* H;               // [(k+1)T][2I] bf16, hi | lo
    float* acc;                // [T][d] fp32 token-order sum
    const int32_t* perm;
    const float* topk_w;
    int* status;
    int T, d, I, E, k;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}

// every lane waits; the outcome is made warp-uniform
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
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

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// Walks this CTA's (tile, K block, part) sequence; part counts the B steps of one K block
// (1 for gate/up; 2 for down: the hi and the lo half of h).
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

// Weight chunks come from HBM and run up to kLead K blocks ahead of the activation tiles
// (from L2).  No deadlock: a wait on raw_empty for K step g needs the MMA of step
// g - RAW - AST, whose activation tile is already issued because kLead < RAW + AST.
constexpr int kLead = 5;


// Which TMEM buffers (256 columns each) a tile uses: N <= 128 -> one (alternating);
// N > 128 -> both.  Producer-side and consumer-side iterate identically.
struct TmemSched {
    int next = 0;
    uint32_t use[2] = {0, 0};
    __device__ __forceinline__ int pick(int N, int (&bufs)[2]) {
        if (N <= 128) { bufs[0] = next; next ^= 1; return 1; }
        bufs[0] = 0; bufs[1] = 1; return 2;
    }
};

// -------- dequant of one packed 128-row half-chunk into the swizzled A layout ---------
// w (16 B of codes, 32 weights) -> 4 output chunks of 8 bf16 at chunk index c0..c0+3.
__device__ __forceinline__ void dequant_store4(uint4 codes, uint32_t s2, uint32_t b2, uint8_t* row_dst, int r,
                                               int c0) {
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
    constexpr uint32_t kMagic = 0x43004300u;   // bf16 pair (128, 128); low nibble = mantissa
    constexpr uint32_t kOne = 0x3F803F80u;
    constexpr uint32_t kNeg128 = 0xC300C300u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w = words[q];
        uint32_t v[4];
        v[0] = (w & 0x000F000Fu) | kMagic;
        v[1] = ((w >> 4) & 0x000F000Fu) | kMagic;
        v[2] = ((w >> 8) & 0x000F000Fu) | kMagic;
        v[3] = ((w >> 12) & 0x000F000Fu) | kMagic;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t code = bf16x2_fma(v[u], kOne, kNeg128);   // exact: (128 + q) - 128
            v[u] = bf16x2_fma(code, s2, b2);                          // one rounding
        }
        const int c = c0 + q;
        const uint32_t addr = smem_u32(row_dst + ((c ^ (r & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                     "r"(v[3])
                     : "memory");
    }
}

// ======================================================================================
// gate/up + SwiGLU
// ======================================================================================
__global__ void __launch_bounds__(kThreads, 1)
    ffn_gate_up_kernel(const __grid_constant__ CUtensorMap tm_xs, const __grid_constant__ CUtensorMap tm_x,
                       FfnParams p) {
    extern __shared__ uint8_t smem_dyn[];
    const int num = *p.num_tiles;
    if ((int)blockIdx.x >= num) return;
    uint8_t* smem = align1024(smem_dyn);
    uint8_t* bstage = smem + GuPlan::b_off;
    uint8_t* astage = smem + GuPlan::a_off;
    uint8_t* raw = smem + GuPlan::raw_off;
    Bars* bars = reinterpret_cast<Bars*>(smem + GuPlan::bar_off);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = p.d / kBK, MT = p.I / kTileRows;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kGuRaw; ++i) { mbar_init(&bars->raw_full[i], 1); mbar_init(&bars->raw_empty[i], kDeqWarps); }
        for (int i = 0; i < kGuB; ++i) { mbar_init(&bars->b_full[i], 1); mbar_init(&bars->b_empty[i], 1); }
        for (int i = 0; i < kGuA; ++i) { mbar_init(&bars->a_full[i], kDeqWarps); mbar_init(&bars->a_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bars->tm_full[i], 1); mbar_init(&bars->tm_empty[i], kEpiWarps); }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kProdWarp && lane == 0) { prefetch_tmap(&tm_xs); prefetch_tmap(&tm_x); }
    if (warp == kMmaWarp) { tmem_alloc(&bars->tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    if (warp == kProdWarp) {
        if (lane == 0) {
            uint32_t rit = 0, bit = 0;
            bool ok = true;
            Cursor cr, cb;
            cr.init(p.tiles, num, KB, 1);
            cb.init(p.tiles, num, KB, 1);
            while (ok && !cb.done()) {
                while (ok && !cr.done() && rit < bit + kLead + 1) {
                    const int e = cr.t.x, mt = cr.t.w;
                    const uint8_t* wsrc = e < p.E ? p.w_routed + (size_t)(e * MT + mt) * KB * kChunkPairBytes
                                                  : p.w_shared + (size_t)mt * KB * kChunkPairBytes;
                    const int rs = rit % kGuRaw;
                    if (!mbar_wait(&bars->raw_empty[rs], ((rit / kGuRaw) & 1) ^ 1, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars->raw_full[rs], kChunkPairBytes);
                    bulk_g2s(raw + rs * kChunkPairBytes, wsrc + (size_t)cr.kb * kChunkPairBytes, kChunkPairBytes,
                             &bars->raw_full[rs]);
                    ++rit;
                    cr.next();
                }
                if (!ok) break;
                const int e = cb.t.x, row0 = cb.t.y, N = round16(cb.t.z);
                const int nbox = (N + kBoxRows - 1) / kBoxRows;
                const CUtensorMap* tm = e < p.E ? &tm_xs : &tm_x;
                const int bs = bit % kGuB;
                if (!mbar_wait(&bars->b_empty[bs], ((bit / kGuB) & 1) ^ 1, abort)) { ok = false; break; }
                mbar_arrive_expect_tx(&bars->b_full[bs], nbox * kBoxBytes);
                for (int bx = 0; bx < nbox; ++bx)
                    tma_load_2d(bstage + bs * kBStageBytes + bx * kBoxBytes, tm, cb.kb * kBK, row0 + bx * kBoxRows,
                                &bars->b_full[bs]);
                ++bit;
                cb.next();
            }
            if (!ok) raise_abort(abort, p.status);
            drain_ring(bars->raw_full, kGuRaw, rit);
            drain_ring(bars->b_full, kGuB, bit);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            uint32_t ait = 0, bit = 0;
            TmemSched ts;
            bool ok = true;
            const uint32_t a_base = smem_u32(astage), b_base = smem_u32(bstage);
            for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
                const int4 t = p.tiles[tile];
                const int N = round16(t.z);
                int bufs[2];
                const int nb = ts.pick(N, bufs);
                for (int q = 0; q < nb; ++q)
                    if (!mbar_wait(&bars->tm_empty[bufs[q]], (ts.use[bufs[q]] & 1) ^ 1, abort)) ok = false;
                if (!ok) break;
                tc_fence_after();
                const uint32_t gate_col = nb == 1 ? 256u * bufs[0] : 0u;
                const uint32_t up_col = nb == 1 ? gate_col + 128u : 256u;
                const uint32_t idesc = idesc_bf16_f32(128, N);
                for (int kb = 0; kb < KB; ++kb) {
                    const int as = ait % kGuA, bs = bit % kGuB;
                    if (!mbar_wait(&bars->a_full[as], (ait / kGuA) & 1, abort)) { ok = false; break; }
                    if (!mbar_wait(&bars->b_full[bs], (bit / kGuB) & 1, abort)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t aoff = a_base + as * 2 * kATileBytes + ks * 32;
                        const uint64_t bd = sw128_desc(b_base + bs * kBStageBytes + ks * 32);
                        const uint32_t accum = (kb | ks) ? 1u : 0u;
                        tc_mma_bf16(tmem + gate_col, sw128_desc(aoff), bd, idesc, accum);
                        tc_mma_bf16(tmem + up_col, sw128_desc(aoff + kATileBytes), bd, idesc, accum);
                    }
                    tc_commit(&bars->a_empty[as]);
                    tc_commit(&bars->b_empty[bs]);
                    ++ait;
                    ++bit;
                }
                if (!ok) break;
                for (int q = 0; q < nb; ++q) { tc_commit(&bars->tm_full[bufs[q]]); ts.use[bufs[q]]++; }
            }
            if (!ok) raise_abort(abort, p.status);
            tc_commit(&bars->drain);
            int never = 0;
            mbar_wait(&bars->drain, 0, &never);
        }
    } else if (warp < kDeqWarps) {
        // dequant: thread -> (matrix: 0 gate / 1 up, row r); 64 weights per K block
        const int mat = threadIdx.x >> 7, r = threadIdx.x & 127;
        uint32_t rit = 0, ait = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb) {
                const int rs = rit % kGuRaw, as = ait % kGuA;
                if (!warp_wait(&bars->raw_full[rs], (rit / kGuRaw) & 1, abort) ||
                    !warp_wait(&bars->a_empty[as], ((ait / kGuA) & 1) ^ 1, abort)) { ok = false; break; }
                const uint8_t* ch = raw + rs * kChunkPairBytes + mat * kChunkBytes;
                const uint4 c0 = *reinterpret_cast<const uint4*>(ch + r * 16);
                const uint4 c1 = *reinterpret_cast<const uint4*>(ch + 2048 + r * 16);
                const uint32_t s = *reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 2 * r);
                const uint32_t b = *reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 256 + 2 * r);
                uint8_t* row_dst = astage + as * 2 * kATileBytes + mat * kATileBytes + (r >> 3) * 1024 + (r & 7) * 128;
                dequant_store4(c0, s * 0x10001u, b * 0x10001u, row_dst, r, 0);
                dequant_store4(c1, s * 0x10001u, b * 0x10001u, row_dst, r, 4);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) { mbar_arrive(&bars->raw_empty[rs]); mbar_arrive(&bars->a_full[as]); }
                ++rit;
                ++ait;
            }
        }
        if (!ok && lane == 0) raise_abort(abort, p.status);
    } else {
        // epilogue: h = silu(g) * u, stored as the bf16 pair (hi, lo = h - hi)
        const int q = warp & 3, g = (warp - kDeqWarps) >> 2;
        TmemSched ts;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            const int4 t = p.tiles[tile];
            const int e = t.x, row0 = t.y, rows = t.z, N = round16(t.z), mt = t.w;
            int bufs[2];
            const int nb = ts.pick(N, bufs);
            for (int qq = 0; qq < nb; ++qq)
                if (!warp_wait(&bars->tm_full[bufs[qq]], ts.use[bufs[qq]] & 1, abort)) ok = false;
            if (!ok) break;
            tc_fence_after();
            const uint32_t gate_col = nb == 1 ? 256u * bufs[0] : 0u;
            const uint32_t up_col = nb == 1 ? gate_col + 128u : 256u;
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
            const int i = mt * kTileRows + 32 * q + lane;
            const size_t hrow0 = e < p.E ? (size_t)row0 : (size_t)p.k * p.T + row0;
            uint16_t* Hp = p.H + hrow0 * 2 * p.I + i;
            for (int c = g; c < N / 16; c += 2) {
                uint32_t G[16], U[16];
                tmem_ld16(tmem + lane_base + gate_col + 16 * c, G);
                tmem_ld16(tmem + lane_base + up_col + 16 * c, U);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = 16 * c + jj;
                    if (j < rows) {
                        const float gv = __uint_as_float(G[jj]), uv = __uint_as_float(U[jj]);
                        const float h = gv / (1.0f + __expf(-gv)) * uv;
                        const uint16_t hi = f32_to_bf16_rn(h);
                        const uint16_t lo = f32_to_bf16_rn(h - bf16f(hi));
                        Hp[(size_t)j * 2 * p.I] = hi;
                        Hp[(size_t)j * 2 * p.I + p.I] = lo;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                for (int qq = 0; qq < nb; ++qq) mbar_arrive(&bars->tm_empty[bufs[qq]]);
            for (int qq = 0; qq < nb; ++qq) ts.use[bufs[qq]]++;
        }
        if (!ok && lane == 0) raise_abort(abort, p.status);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ======================================================================================
// down projection + weighted fp32 accumulation into the token-order sum
// ======================================================================================
__global__ void __launch_bounds__(kThreads, 1)
    ffn_down_kernel(const __grid_constant__ CUtensorMap tm_h, FfnParams p) {
    extern __shared__ uint8_t smem_dyn[];
    const int num = *p.num_tiles;
    if ((int)blockIdx.x >= num) return;
    uint8_t* smem = align1024(smem_dyn);
    uint8_t* bstage = smem + DnPlan::b_off;
    uint8_t* astage = smem + DnPlan::a_off;
    uint8_t* raw = smem + DnPlan::raw_off;
    Bars* bars = reinterpret_cast<Bars*>(smem + DnPlan::bar_off);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = p.I / kBK, MT = p.d / kTileRows;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDnRaw; ++i) { mbar_init(&bars->raw_full[i], 1); mbar_init(&bars->raw_empty[i], kDeqWarps); }
        for (int i = 0; i < kDnB; ++i) { mbar_init(&bars->b_full[i], 1); mbar_init(&bars->b_empty[i], 1); }
        for (int i = 0; i < kDnA; ++i) { mbar_init(&bars->a_full[i], kDeqWarps); mbar_init(&bars->a_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bars->tm_full[i], 1); mbar_init(&bars->tm_empty[i], kEpiWarps); }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kProdWarp && lane == 0) prefetch_tmap(&tm_h);
    if (warp == kMmaWarp) { tmem_alloc(&bars->tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    if (warp == kProdWarp) {
        if (lane == 0) {
            uint32_t rit = 0, bit = 0;
            bool ok = true;
            Cursor cr, cb;
            cr.init(p.tiles, num, KB, 1);
            cb.init(p.tiles, num, KB, 2);
            while (ok && !cb.done()) {
                while (ok && !cr.done() && rit < bit / 2 + kLead + 1) {
                    const int e = cr.t.x, mt = cr.t.w;
                    const uint8_t* wsrc = e < p.E ? p.w_routed + (size_t)(e * MT + mt) * KB * kChunkBytes
                                                  : p.w_shared + (size_t)mt * KB * kChunkBytes;
                    const int rs = rit % kDnRaw;
                    if (!mbar_wait(&bars->raw_empty[rs], ((rit / kDnRaw) & 1) ^ 1, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bars->raw_full[rs], kChunkBytes);
                    bulk_g2s(raw + rs * kChunkBytes, wsrc + (size_t)cr.kb * kChunkBytes, kChunkBytes,
                             &bars->raw_full[rs]);
                    ++rit;
                    cr.next();
                }
                if (!ok) break;
                const int e = cb.t.x, row0 = cb.t.y, N = round16(cb.t.z);
                const int nbox = (N + kBoxRows - 1) / kBoxRows;
                const int hrow0 = e < p.E ? row0 : p.k * p.T + row0;
                const int bs = bit % kDnB;
                if (!mbar_wait(&bars->b_empty[bs], ((bit / kDnB) & 1) ^ 1, abort)) { ok = false; break; }
                mbar_arrive_expect_tx(&bars->b_full[bs], nbox * kBoxBytes);
                for (int bx = 0; bx < nbox; ++bx)
                    tma_load_2d(bstage + bs * kBStageBytes + bx * kBoxBytes, &tm_h, cb.part * p.I + cb.kb * kBK,
                                hrow0 + bx * kBoxRows, &bars->b_full[bs]);
                ++bit;
                cb.next();
            }
            if (!ok) raise_abort(abort, p.status);
            drain_ring(bars->raw_full, kDnRaw, rit);
            drain_ring(bars->b_full, kDnB, bit);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            uint32_t ait = 0, bit = 0, tcount = 0;
            uint32_t use[2] = {0, 0};
            bool ok = true;
            const uint32_t a_base = smem_u32(astage), b_base = smem_u32(bstage);
            for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x, ++tcount) {
                const int4 t = p.tiles[tile];
                const int N = round16(t.z);
                const int buf = tcount & 1;
                if (!mbar_wait(&bars->tm_empty[buf], (use[buf] & 1) ^ 1, abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t dcol = 256u * buf;
                const uint32_t idesc = idesc_bf16_f32(128, N);
                for (int kb = 0; kb < KB && ok; ++kb) {
                    const int as = ait % kDnA;
                    if (!mbar_wait(&bars->a_full[as], (ait / kDnA) & 1, abort)) { ok = false; break; }
                    for (int part = 0; part < 2; ++part) {
                        const int bs = bit % kDnB;
                        if (!mbar_wait(&bars->b_full[bs], (bit / kDnB) & 1, abort)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t ad = sw128_desc(a_base + as * kATileBytes + ks * 32);
                            const uint64_t bd = sw128_desc(b_base + bs * kBStageBytes + ks * 32);
                            tc_mma_bf16(tmem + dcol, ad, bd, idesc, (kb | part | ks) ? 1u : 0u);
                        }
                        tc_commit(&bars->b_empty[bs]);
                        ++bit;
                    }
                    tc_commit(&bars->a_empty[as]);
                    ++ait;
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
        // dequant: thread -> (row r, half hf); 32 weights per K block
        const int hf = threadIdx.x >> 7, r = threadIdx.x & 127;
        uint32_t rit = 0, ait = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb) {
                const int rs = rit % kDnRaw, as = ait % kDnA;
                if (!warp_wait(&bars->raw_full[rs], (rit / kDnRaw) & 1, abort) ||
                    !warp_wait(&bars->a_empty[as], ((ait / kDnA) & 1) ^ 1, abort)) { ok = false; break; }
                const uint8_t* ch = raw + rs * kChunkBytes;
                const uint4 cw = *reinterpret_cast<const uint4*>(ch + hf * 2048 + r * 16);
                const uint32_t s = *reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 2 * r);
                const uint32_t b = *reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 256 + 2 * r);
                uint8_t* row_dst = astage + as * kATileBytes + (r >> 3) * 1024 + (r & 7) * 128;
                dequant_store4(cw, s * 0x10001u, b * 0x10001u, row_dst, r, 4 * hf);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) { mbar_arrive(&bars->raw_empty[rs]); mbar_arrive(&bars->a_full[as]); }
                ++rit;
                ++ait;
            }
        }
        if (!ok && lane == 0) raise_abort(abort, p.status);
    } else {
        // epilogue: acc[t][n] += w * y for every row of the tile
        const int q = warp & 3, g = (warp - kDeqWarps) >> 2;
        uint32_t use[2] = {0, 0}, tcount = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num && ok; tile += gridDim.x, ++tcount) {
            const int4 t = p.tiles[tile];
            const int e = t.x, row0 = t.y, rows = t.z, N = round16(t.z), mt = t.w;
            const int buf = tcount & 1;
            if (!warp_wait(&bars->tm_full[buf], use[buf] & 1, abort)) { ok = false; break; }
            tc_fence_after();
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
            const int n = mt * kTileRows + 32 * q + lane;
            for (int c = g; c < N / 16; c += 2) {
                uint32_t Y[16];
                tmem_ld16(tmem + lane_base + 256u * buf + 16 * c, Y);
                // token and weight of the 16 rows: lane jj fetches row 16c + jj
                int my_t = 0;
                float my_w = 0.f;
                const int jl = 16 * c + (lane & 15);
                if (jl < rows) {
                    if (e < p.E) {
                        const int asg = p.perm[row0 + jl];
                        my_t = asg / p.k;
                        my_w = p.topk_w[asg];
                    } else {
                        my_t = row0 + jl;
                        my_w = 1.0f;
                    }
                }
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int tok = __shfl_sync(0xffffffffu, my_t, jj);
                    const float w = __shfl_sync(0xffffffffu, my_w, jj);
                    if (16 * c + jj < rows) atomicAdd(p.acc + (size_t)tok * p.d + n, w * __uint_as_float(Y[jj]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tm_empty[buf]);
            use[buf]++;
        }
        if (!ok && lane == 0) raise_abort(abort, p.status);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ======================================================================================
// combine: y = bf16(acc)
// ======================================================================================
__global__ void combine_kernel(const float4* __restrict__ acc, uint2* __restrict__ y, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[i];
        const uint32_t lo = (uint32_t)f32_to_bf16_rn(v.x) | ((uint32_t)f32_to_bf16_rn(v.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16_rn(v.z) | ((uint32_t)f32_to_bf16_rn(v.w) << 16);
        y[i] = make_uint2(lo, hi);
    }
}

FfnParams make_params(const FfnArgs& a, bool gate_up) {
    FfnParams p{};
    p.w_routed = a.w_routed;
    p.w_shared = a.w_shared;
    p.tiles = reinterpret_cast<const int4*>(a.ws + (gate_up ? a.L.gu_tiles : a.L.dn_tiles));
    p.num_tiles = reinterpret_cast<const int*>(a.ws + (gate_up ? a.L.gu_num : a.L.dn_num));
    p.H = reinterpret_cast<uint16_t*>(a.ws + a.L.H);
    p.acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    p.perm = a.perm;
    p.topk_w = a.topk_w;
    p.status = reinterpret_cast<int*>(a.ws + a.L.status);
    p.T = a.T; p.d = a.d; p.I = a.I; p.E = a.E; p.k = a.k;
    return p;
}

}  // namespace

cudaError_t launch_gate_up(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    static bool attr = false;
    if (!attr) {
        cudaError_t err = cudaFuncSetAttribute(ffn_gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               GuPlan::bytes);
        if (err != cudaSuccess) return err;
        attr = true;
    }
    CUtensorMap tm_xs, tm_x;
    cudaError_t err = make_tmap_bf16_2d(&tm_xs, a.ws + a.L.xs, (uint64_t)a.k * a.T, a.d, (uint64_t)a.d * 2, kBK, kBoxRows);
    if (err != cudaSuccess) return err;
    err = make_tmap_bf16_2d(&tm_x, a.x, a.T, a.d, (uint64_t)a.d * 2, kBK, kBoxRows);
    if (err != cudaSuccess) return err;
    ffn_gate_up_kernel<<<a.num_sms, kThreads, GuPlan::bytes, st>>>(tm_xs, tm_x, make_params(a, true));
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_down(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    static bool attr = false;
    if (!attr) {
        cudaError_t err =
            cudaFuncSetAttribute(ffn_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DnPlan::bytes);
        if (err != cudaSuccess) return err;
        attr = true;
    }
    CUtensorMap tm_h;
    cudaError_t err = make_tmap_bf16_2d(&tm_h, a.ws + a.L.H, (uint64_t)(a.k + 1) * a.T, 2 * (uint64_t)a.I,
                                        (uint64_t)a.I * 4, kBK, kBoxRows);
    if (err != cudaSuccess) return err;
    ffn_down_kernel<<<a.num_sms, kThreads, DnPlan::bytes, st>>>(tm_h, make_params(a, false));
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_combine(int T, int d, const float* acc, uint16_t* y, cudaStream_t st, unsigned long long* launches) {
    const size_t n4 = (size_t)T * d / 4;
    const int blocks = (int)((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
    combine_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc), reinterpret_cast<uint2*>(y), n4);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
