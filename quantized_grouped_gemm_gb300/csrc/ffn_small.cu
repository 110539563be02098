// ffn_small.cu -- grouped SwiGLU FFN for expert groups of at most 32 token rows (warp MMA).
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026), section "Dequantize
// weights during matrix multiplication" (the bf16 weight tile exists only on chip) and section
// "Match tile size to expert load" (small expert groups want a small row tile).
//
// When an expert receives few rows (a 512-token chunk gives each expert about 16), a
// tcgen05.mma tile of 128 token rows is mostly padding and its fixed cost per instruction
// dominates.  These kernels take the expert groups of at most kSmallRows rows from their own
// tile list instead: weights on the MMA's M side (16 rows per warp MMA), tokens on N (8 per
// MMA), so the tensor work follows the real row count.  The 4-bit weights are dequantised
// exactly (one bf16 FMA per two weights, as everywhere else) straight into MMA fragments;
// the bf16 weight tile never reaches shared memory.
//
// Two persistent CTAs per SM, each 8 compute warps + 1 producer warp.  A unit is a tile of the
// small list: (expert, first row, rows <= 32, weight tile).  The producer streams, per K block
// of 64, the packed chunk pair (one 9216-byte bulk copy) and the activation rows of the block
// (for the down projection the hi and lo halves of h) into a ring of shared-memory slots.  An
// activation block is two unswizzled 32-row x 32-column TMA boxes with 64-byte rows: the eight
// lanes of a quarter warp then read two whole rows, 128 contiguous bytes, with no bank
// conflict (a 64-column box in 128-byte swizzle puts rows 2p and 2p+1 of a quarter warp on the
// same banks).
//   gate/up: warp w owns i-rows 16w .. 16w+15 of the 128-row tile for both gate and up, so g
//            and u of the same (i, token) meet in one thread: h = silu(g) * u is written as a
//            bf16 hi/lo pair.
//   down:    warp w owns rows 32w .. 32w+31 of the 256-row output tile; h enters as hi + lo
//            (two MMAs); routing weight * y is added into the fp32 token-order sum.
// Both epilogues stage the warp's block in shared memory and write it with 16-byte stores or
// 4-wide vector adds.
// All waits are bounded (MOE_STATUS_TIMEOUT); copies in flight land before the CTA leaves.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kSmWarps = 8;                          // compute warps
constexpr int kSmThreads = (kSmWarps + 1) * 32;      // + producer warp
constexpr int kSmTok = kSmallRows;                   // token rows of an activation tile (TMA box)
constexpr int kSmActBytes = kSmTok * 128;            // 32 rows x 64 bf16: two 32-column boxes
constexpr int kSmHalfBytes = kSmActBytes / 2;        // one box, rows of 64 bytes
constexpr int kSmRingGU = 4, kSmRingDN = 3;   // per CTA; two CTAs per SM

template <bool kDown>
struct SmCfg {
    static constexpr int R = kDown ? kSmRingDN : kSmRingGU;
    static constexpr int ACTS = kDown ? 2 : 1;                   // activation tiles per K block
    static constexpr int w_off = 0;                              // R x 9216
    static constexpr int a_off = (R * kChunkPairBytes + 1023) / 1024 * 1024;
    static constexpr int stage_off = a_off + R * ACTS * kSmActBytes;
    // per warp: down 32 tokens x 33 floats (padded rows); gate/up 32 tokens x 16 (hi) + 16 (lo) bf16
    static constexpr int stage_warp = kDown ? kSmTok * 33 * 4 : kSmTok * 64;
    static constexpr int bar_off = stage_off + kSmWarps * stage_warp;
    static constexpr int smem = bar_off + 2 * R * 8 + 1024;      // + 1024-byte alignment slack
};

struct SmParams {
    const uint8_t* w_routed;   // packed stack of the projection (gate/up pairs or down pairs)
    const uint8_t* w_shared;
    const int* mode_routed;
    const int* mode_shared;
    const int4* tiles;         // (expert, first row, rows, weight tile); expert == E: shared
    const int* num_tiles;
    uint16_t* H;               // [(k+1)T][2I] bf16, hi | lo
    float* acc;                // [T][d] fp32 token-order sum
    const int32_t* perm;
    const float* topk_w;
    int* status;
    int T, d, I, E, k;
};

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t lds16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// Activation fragment of token row n of a 32 x 64 block: columns 8t..8t+7 (c4 = 0, first box)
// or 32+8t..32+8t+7 (c4 = 1, second box) as 8 bf16.
__device__ __forceinline__ uint4 act_frag(const uint8_t* tile, int n, int t, int c4) {
    return *reinterpret_cast<const uint4*>(tile + c4 * kSmHalfBytes + n * 64 + 16 * t);
}

// One activation block: columns x0 .. x0+63 of rows y0 .. y0+31 as two 32-column boxes.
__device__ __forceinline__ void load_act_block(uint8_t* dst, const CUtensorMap* tm, int x0, int y0, uint64_t* bar) {
    tma_load_2d(dst, tm, x0, y0, bar);
    tma_load_2d(dst + kSmHalfBytes, tm, x0 + 32, y0, bar);
}

// Dequantised A fragments of rows r0 = rb + g and r1 = r0 + 8 of one 128-row chunk: v[0..3]
// columns 8t..8t+7, v[4..7] columns 32+8t..32+8t+7 (pairs (2u, 2u+1) per register).
template <bool kDenorm>
__device__ __forceinline__ void deq_rows16(const uint8_t* ch, int rb, int lane, uint32_t (&a0)[8], uint32_t (&a1)[8]) {
    const int g = lane >> 2, t = lane & 3;
    const int r0 = rb + g, r1 = r0 + 8;
    const uint32_t w00 = lds32(ch + r0 * 16 + 4 * t), w01 = lds32(ch + 2048 + r0 * 16 + 4 * t);
    const uint32_t w10 = lds32(ch + r1 * 16 + 4 * t), w11 = lds32(ch + 2048 + r1 * 16 + 4 * t);
    const uint32_t s0 = lds16(ch + kChunkCodes + 2 * r0) * 0x10001u, b0 = lds16(ch + kChunkCodes + 256 + 2 * r0) * 0x10001u;
    const uint32_t s1 = lds16(ch + kChunkCodes + 2 * r1) * 0x10001u, b1 = lds16(ch + kChunkCodes + 256 + 2 * r1) * 0x10001u;
    uint32_t v[4];
    dequant_word<kDenorm>(w00, s0, b0, v); a0[0] = v[0]; a0[1] = v[1]; a0[2] = v[2]; a0[3] = v[3];
    dequant_word<kDenorm>(w01, s0, b0, v); a0[4] = v[0]; a0[5] = v[1]; a0[6] = v[2]; a0[7] = v[3];
    dequant_word<kDenorm>(w10, s1, b1, v); a1[0] = v[0]; a1[1] = v[1]; a1[2] = v[2]; a1[3] = v[3];
    dequant_word<kDenorm>(w11, s1, b1, v); a1[4] = v[0]; a1[5] = v[1]; a1[6] = v[2]; a1[7] = v[3];
}

// acc (16 rows x 8 tokens) += A (rows r0, r1 of a0/a1) . activations (x0 = cols 8t.., x1 = 32+8t..)
__device__ __forceinline__ void mma_rows16(float (&c)[4], const uint32_t (&a0)[8], const uint32_t (&a1)[8],
                                           const uint4& x0, const uint4& x1) {
    mma_bf16_16816(c, a0[0], a1[0], a0[1], a1[1], x0.x, x0.y);
    mma_bf16_16816(c, a0[2], a1[2], a0[3], a1[3], x0.z, x0.w);
    mma_bf16_16816(c, a0[4], a1[4], a0[5], a1[5], x1.x, x1.y);
    mma_bf16_16816(c, a0[6], a1[6], a0[7], a1[7], x1.z, x1.w);
}

__device__ __forceinline__ void red_add_v4_f32(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// One unit's K loop and epilogue for NT groups of 8 tokens.
template <bool kDown, int NT, bool kDenorm>
__device__ __forceinline__ void small_unit(const SmParams& p, const int4 t4, uint8_t* wring, uint8_t* aring,
                                           uint8_t* stage, uint64_t* full, uint64_t* empty, uint32_t& it, int KB,
                                           int warp, int lane, bool& ok, volatile int* abort) {
    using C = SmCfg<kDown>;
    const int g = lane >> 2, t = lane & 3;
    const int e = t4.x, row0 = t4.y, rows = t4.z, wt = t4.w;
    float acc[2][NT][4];
#pragma unroll
    for (int G = 0; G < 2; ++G)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[G][j][0] = acc[G][j][1] = acc[G][j][2] = acc[G][j][3] = 0.f;
    for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = it % C::R;
        if (!mbar_spin(&full[s], (it / C::R) & 1, abort)) ok = false;
        const uint8_t* pair = wring + s * kChunkPairBytes;
        const uint8_t* at = aring + s * C::ACTS * kSmActBytes;
        if (!kDown) {
            // gate rows 16w.. (first chunk) and up rows 16w.. (second chunk)
            uint32_t ga0[8], ga1[8], ua0[8], ua1[8];
            deq_rows16<kDenorm>(pair, 16 * warp, lane, ga0, ga1);
            deq_rows16<kDenorm>(pair + kChunkBytes, 16 * warp, lane, ua0, ua1);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const uint4 x0 = act_frag(at, 8 * j + g, t, 0), x1 = act_frag(at, 8 * j + g, t, 1);
                mma_rows16(acc[0][j], ga0, ga1, x0, x1);
                mma_rows16(acc[1][j], ua0, ua1, x0, x1);
            }
        } else {
            // rows 32w .. 32w+31 of the 256-row tile: chunk half = w >> 2
            const uint8_t* ch = pair + (warp >> 2) * kChunkBytes;
            const int rb = 32 * (warp & 3);
            uint32_t p0[8], p1[8], q0[8], q1[8];
            deq_rows16<kDenorm>(ch, rb, lane, p0, p1);
            deq_rows16<kDenorm>(ch, rb + 16, lane, q0, q1);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const uint4 h0 = act_frag(at, 8 * j + g, t, 0), h1 = act_frag(at, 8 * j + g, t, 1);
                const uint4 l0 = act_frag(at + kSmActBytes, 8 * j + g, t, 0);
                const uint4 l1 = act_frag(at + kSmActBytes, 8 * j + g, t, 1);
                mma_rows16(acc[0][j], p0, p1, h0, h1);
                mma_rows16(acc[0][j], p0, p1, l0, l1);
                mma_rows16(acc[1][j], q0, q1, h0, h1);
                mma_rows16(acc[1][j], q0, q1, l0, l1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        __syncwarp();
    }
    if (!ok) return;
    // D fragment: c0, c1 = (row g, tokens 8j + 2t, +1); c2, c3 = (row g + 8, same tokens).
    // The warp stages its block in shared memory, then writes it with 16-byte accesses.
    if (!kDown) {
        uint16_t* sh = reinterpret_cast<uint16_t*>(stage);   // [32 tokens][16 hi | 16 lo]
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int tok = 8 * j + 2 * t + u, r = g + 8 * hh;
                    const float gv = acc[0][j][2 * hh + u], uv = acc[1][j][2 * hh + u];
                    const float h = gv / (1.0f + __expf(-gv)) * uv;
                    const uint16_t hi = f32_to_bf16_rn(h);
                    sh[tok * 32 + r] = hi;
                    sh[tok * 32 + 16 + r] = f32_to_bf16_rn(h - __uint_as_float((uint32_t)hi << 16));
                }
        __syncwarp();
        // token tok, piece q (0, 1: hi columns 0-7, 8-15; 2, 3: lo): one 16-byte store
        for (int idx = lane; idx < 32 * 4; idx += 32) {
            const int tok = idx >> 2, q = idx & 3;
            if (tok < rows && tok < 8 * NT) {
                const size_t hrow = e < p.E ? (size_t)row0 + tok : (size_t)p.k * p.T + row0 + tok;
                const int col = wt * kTileRows + 16 * warp + 8 * (q & 1) + (q >> 1) * p.I;
                *reinterpret_cast<uint4*>(p.H + hrow * 2 * p.I + col) =
                    *reinterpret_cast<const uint4*>(sh + tok * 32 + 8 * q);
            }
        }
        __syncwarp();
    } else {
        float* sy = reinterpret_cast<float*>(stage);   // [32 tokens][33]: rows 0..31 of my 32
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int G = 0; G < 2; ++G)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        sy[(8 * j + 2 * t + u) * 33 + 16 * G + g + 8 * hh] = acc[G][j][2 * hh + u];
        __syncwarp();
        // token tok, rows 4q .. 4q+3: weight * y into the fp32 sum with one vector add
        for (int idx = lane; idx < 32 * 8; idx += 32) {
            const int tok = idx >> 3, q = idx & 7;
            if (tok < rows && tok < 8 * NT) {
                int tk;
                float w;
                if (e < p.E) {
                    const int asg = p.perm[row0 + tok];
                    tk = asg / p.k;
                    w = p.topk_w[asg];
                } else {
                    tk = row0 + tok;
                    w = 1.0f;
                }
                const float* v = sy + tok * 33 + 4 * q;
                red_add_v4_f32(p.acc + (size_t)tk * p.d + (size_t)wt * 256 + 32 * warp + 4 * q, w * v[0], w * v[1],
                               w * v[2], w * v[3]);
            }
        }
        __syncwarp();
    }
}

template <bool kDown>
__global__ void __launch_bounds__(kSmThreads, 2)
    ffn_small_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, SmParams p) {
    using C = SmCfg<kDown>;
    extern __shared__ uint8_t smem_dyn[];
    const int num = *p.num_tiles;
    if ((int)blockIdx.x >= num) return;
    uint8_t* smem = smem_dyn + ((1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u);
    uint8_t* wring = smem + C::w_off;
    uint8_t* aring = smem + C::a_off;
    uint8_t* stage = smem + C::stage_off + (threadIdx.x >> 5) * C::stage_warp;   // compute warps only
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::bar_off);
    uint64_t* empty = full + C::R;
    __shared__ int s_abort;
    volatile int* abort = &s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = (kDown ? p.I : p.d) / kBK;
    const int WT = (kDown ? p.d / 256 : p.I / kTileRows);      // weight tiles per expert
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::R; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kSmWarps); }
        s_abort = 0;
        fence_barrier_init();
    }
    __syncwarp();
    __syncthreads();

    if (warp == kSmWarps) {
        // producer: every (unit, K block) of this CTA in order
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num && ok; u += gridDim.x) {
                const int4 t4 = p.tiles[u];
                const int e = t4.x, row0 = t4.y, wt = t4.w;
                const uint8_t* wbase = e < p.E ? p.w_routed + (size_t)(e * WT + wt) * KB * kChunkPairBytes
                                               : p.w_shared + (size_t)wt * KB * kChunkPairBytes;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::R;
                    if (!mbar_spin(&empty[s], ((it / C::R) & 1) ^ 1, abort)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], kChunkPairBytes + C::ACTS * kSmActBytes);
                    bulk_g2s(wring + s * kChunkPairBytes, wbase + (size_t)kb * kChunkPairBytes, kChunkPairBytes, &full[s]);
                    uint8_t* at = aring + s * C::ACTS * kSmActBytes;
                    if (kDown) {
                        const int hrow0 = e < p.E ? row0 : p.k * p.T + row0;
                        load_act_block(at, &tm_a, kb * kBK, hrow0, &full[s]);
                        load_act_block(at + kSmActBytes, &tm_a, p.I + kb * kBK, hrow0, &full[s]);
                    } else {
                        load_act_block(at, e < p.E ? &tm_a : &tm_b, kb * kBK, row0, &full[s]);
                    }
                }
            }
            if (!ok) { *abort = 1; set_status(p.status, MOE_STATUS_TIMEOUT); }
            // the copies still in flight land before the CTA leaves
            int never = 0;
            const uint32_t first = it > (uint32_t)C::R ? it - C::R : 0;
            for (uint32_t i = first; i < it; ++i) mbar_spin(&full[i % C::R], (i / C::R) & 1, &never);
        }
        __syncwarp();
    } else {
        uint32_t it = 0;
        bool ok = true;
        const int mode_r = *p.mode_routed, mode_s = *p.mode_shared;
        for (int u = blockIdx.x; u < num; u += gridDim.x) {
            const int4 t4 = p.tiles[u];
            // warp votes keep the dispatch visibly warp-uniform
            const bool dn = __all_sync(0xffffffffu, (t4.x < p.E ? mode_r : mode_s) == kScaleDenorm);
            const int nt = __shfl_sync(0xffffffffu, (t4.z + 7) / 8, 0);
            if (dn) {
                if (nt <= 1) small_unit<kDown, 1, true>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
                else if (nt == 2) small_unit<kDown, 2, true>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
                else if (nt == 3) small_unit<kDown, 3, true>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
                else small_unit<kDown, 4, true>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
            } else {
                if (nt <= 1) small_unit<kDown, 1, false>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
                else if (nt == 2) small_unit<kDown, 2, false>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
                else if (nt == 3) small_unit<kDown, 3, false>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
                else small_unit<kDown, 4, false>(p, t4, wring, aring, stage, full, empty, it, KB, warp, lane, ok, abort);
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, ok)) break;
        }
        if (!ok && lane == 0) { *abort = 1; set_status(p.status, MOE_STATUS_TIMEOUT); }
    }
    __syncthreads();
}

SmParams make_small_params(const FfnArgs& a, bool gate_up) {
    SmParams p{};
    const size_t gu_bytes = (size_t)(a.I / kTileRows) * (a.d / kBK) * kChunkPairBytes;
    p.w_routed = a.w_routed + kPackHeader + (gate_up ? 0 : (size_t)a.E * gu_bytes);
    p.w_shared = a.w_shared + kPackHeader + (gate_up ? 0 : gu_bytes);
    p.mode_routed = reinterpret_cast<const int*>(a.w_routed);
    p.mode_shared = reinterpret_cast<const int*>(a.w_shared);
    p.tiles = reinterpret_cast<const int4*>(a.ws + (gate_up ? a.L.gu_small : a.L.dn_small));
    p.num_tiles = reinterpret_cast<const int*>(a.ws + (gate_up ? a.L.gu_small_num : a.L.dn_small_num));
    p.H = reinterpret_cast<uint16_t*>(a.ws + a.L.H);
    p.acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    p.perm = a.perm;
    p.topk_w = a.topk_w;
    p.status = reinterpret_cast<int*>(a.ws + a.L.status);
    p.T = a.T; p.d = a.d; p.I = a.I; p.E = a.E; p.k = a.k;
    return p;
}

template <bool kDown>
cudaError_t set_small_smem_attr() {
    static bool done = false;
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(ffn_small_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SmCfg<kDown>::smem);
    if (e == cudaSuccess) done = true;
    return e;
}

}  // namespace

cudaError_t launch_gate_up_small(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaError_t err = set_small_smem_attr<false>();
    if (err != cudaSuccess) return err;
    CUtensorMap tm_xs, tm_x;
    err = make_tmap_bf16_2d(&tm_xs, a.ws + a.L.xs, (uint64_t)a.k * a.T, a.d, (uint64_t)a.d * 2, 32, kSmTok, false);
    if (err != cudaSuccess) return err;
    err = make_tmap_bf16_2d(&tm_x, a.x, a.T, a.d, (uint64_t)a.d * 2, 32, kSmTok, false);
    if (err != cudaSuccess) return err;
    ffn_small_kernel<false><<<2 * a.num_sms, kSmThreads, SmCfg<false>::smem, st>>>(tm_xs, tm_x, make_small_params(a, true));
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_down_small(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaError_t err = set_small_smem_attr<true>();
    if (err != cudaSuccess) return err;
    CUtensorMap tm_h;
    err = make_tmap_bf16_2d(&tm_h, a.ws + a.L.H, (uint64_t)(a.k + 1) * a.T, 2 * (uint64_t)a.I, (uint64_t)a.I * 4, 32,
                            kSmTok, false);
    if (err != cudaSuccess) return err;
    ffn_small_kernel<true><<<2 * a.num_sms, kSmThreads, SmCfg<true>::smem, st>>>(tm_h, tm_h, make_small_params(a, false));
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
