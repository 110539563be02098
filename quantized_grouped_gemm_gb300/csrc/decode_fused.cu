// decode_fused.cu -- the one-token forward (routing, gate/up, SwiGLU, down, weighted combine)
// in a single launch.
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026): section "Optimize the
// single-row weight path" (a decode step reads every selected weight once; rows are split over
// threads that share the activation vector) and section "Reduce intermediate and state
// traffic" (the expert chain -- input projections, gated activation, output projection,
// routing score and shared-expert sum -- runs without round trips through memory).
//
// Work split.  A "unit" is (slot, h slice): slot 0..k-1 the routed experts in top-k order,
// slot k the shared expert; an h slice is 128 consecutive rows of the intermediate vector h
// (one 128-row tile of the gate and up matrices).  Each unit is a cluster of 4 CTAs; CTA c
//   * dots the 128 gate and 128 up rows of the slice with x over column quarter c (d/256 chunk
//     pairs of 128 rows x 64 columns);
//   * after the cluster exchange of the partial sums (distributed shared memory) computes
//     h = silu(g) * u for the slice and dots the down rows of its 256-row output tiles
//     (tiles c, c + 4, ...) with that slice of h (2 chunk pairs per tile);
//   * adds routing weight * partial rows into the fp32 sum (red.add); the last unit to finish an
//     output tile writes its bf16 rows and clears the sum.
// Routing runs in the same grid: warp w of CTA b computes the logit of expert b + w * grid in
// the fixed order of the router oracle and publishes it as a (call tag, value) word, in eight
// copies; the routed CTAs poll one copy each (bounded) until all E words carry this call's tag,
// take the top-k themselves and start their weight copies.  The tag is an epoch kept in the
// workspace and moved on by the last CTA past its read.  The shared-expert CTAs start their
// copies, and every CTA loads its router row, before the previous kernel on the stream has
// finished (programmatic dependent launch).
//
// Weights move with bulk copies (9216-byte chunk pairs) into a ring of shared-memory slots;
// the ALU dequantises them exactly as the prefill kernels do (one bf16 FMA per two weights)
// and the warp-level bf16 MMA, with fp32 accumulation, forms the dot products.  h enters the
// down MMA as a bf16 hi/lo pair, so h is not rounded to bf16.
//
// The grid waits on itself (the routing words and the cluster barriers), so it runs only when
// every cluster is resident at once: the launcher checks that with the occupancy API and
// otherwise reports cudaErrorNotSupported (the caller then runs the three-kernel decode path).
// Warp-collective code (MMA, shuffles, votes) sits outside branches the compiler cannot prove
// warp-uniform, and single-lane sections end with __syncwarp: a split warp ran such code
// several times slower.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kFzThreads = 256;
constexpr int kFzCluster = 4;         // CTAs per unit: the four column quarters of its gate/up rows
constexpr int kFzSlice = 128;         // h rows per unit (one 128-row tile of gate and up)
constexpr int kFzReplicas = 8;        // copies of the published logit words
constexpr int kFzMaxUnits = 72;       // (k + 1) * I / 128 for I <= 1024 (grids that fit the GPU at once)
constexpr int kFzRingMax = 16;        // chunk-pair slots
constexpr int kFzOneCtaSmem = 120000; // dynamic shared memory of a CTA: above half of an SM's
#ifndef MOE_POLL_SLEEP_NS
#define MOE_POLL_SLEEP_NS 200
#endif
constexpr unsigned kPollSleepNs = MOE_POLL_SLEEP_NS;   // back-off between polls of the logit words

// status words used here (the rest of the 64-int area belongs to the other decode kernels)
constexpr int kStPassed = 3;          // CTAs past their read of the epoch
constexpr int kStEpoch = 4;           // tag of the last call's published logits
constexpr int kStTiles = 8;           // per 256-row output tile: units finished

// Phase timestamps for tuning builds with MOE_TRACE: thread 0 of each CTA keeps SM clock
// readings in shared memory and writes them, with one global-timer reading to line CTAs up,
// to the unused tail of the decode scratch (after the partial outputs) when it ends.
#ifdef MOE_TRACE
#define FZ_STAMP(i)                                   \
    do {                                              \
        if (threadIdx.x == 0) s_trace[(i)] = clock64(); \
        __syncwarp();                                 \
    } while (0)
#define FZ_FLUSH()                                                                                      \
    do {                                                                                                \
        if (threadIdx.x == 0 && a.trace) {                                                              \
            unsigned long long* tr_ = a.trace + blockIdx.x * 20;                                        \
            for (int i_ = 0; i_ < 16; ++i_) tr_[i_] = s_trace[i_];                                      \
            tr_[16] = globaltimer_ns();                                                                 \
            unsigned smid_;                                                                             \
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                          \
            tr_[18] = smid_;                                                                            \
            tr_[17] = s_gt0;                                                                            \
        }                                                                                               \
    } while (0)
#else
#define FZ_STAMP(i) \
    do {            \
    } while (0)
#define FZ_FLUSH() \
    do {           \
    } while (0)
#endif

struct FzParams {
    FusedDecodeArgs a;
    int NS;         // h slices (I / 256)
    int ring;       // ring slots
};

__device__ __forceinline__ uint32_t lds_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t lds_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// 128 rows (eight m16 groups) x 64 columns of one 128-row chunk, dotted with activations
// given as bf16 pairs: a0 = columns 8t..8t+7, a1 = columns 32+8t..32+8t+7 (t = lane & 3); with
// kHiLo the activations are hi + lo and both halves go through the MMA.  Row 16 G + (lane >> 2)
// accumulates into acc[G][0], row 16 G + (lane >> 2) + 8 into acc[G][2].  The eight groups are
// independent accumulation chains.
template <bool kDenorm, bool kHiLo>
__device__ __forceinline__ void chunk_rows128(const uint8_t* ch, int lane, const uint4& a0, const uint4& a1,
                                              const uint4& l0, const uint4& l1, float (&acc)[8][4]) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int G = 0; G < 8; ++G) {
        const int r0 = 16 * G + g, r1 = r0 + 8;
        const uint32_t w00 = lds_u32(ch + r0 * 16 + 4 * t), w01 = lds_u32(ch + 2048 + r0 * 16 + 4 * t);
        const uint32_t w10 = lds_u32(ch + r1 * 16 + 4 * t), w11 = lds_u32(ch + 2048 + r1 * 16 + 4 * t);
        const uint32_t s0 = lds_u16(ch + kChunkCodes + 2 * r0) * 0x10001u;
        const uint32_t b0 = lds_u16(ch + kChunkCodes + 256 + 2 * r0) * 0x10001u;
        const uint32_t s1 = lds_u16(ch + kChunkCodes + 2 * r1) * 0x10001u;
        const uint32_t b1 = lds_u16(ch + kChunkCodes + 256 + 2 * r1) * 0x10001u;
        uint32_t v0[4], v1[4];
        dequant_word<kDenorm>(w00, s0, b0, v0);
        dequant_word<kDenorm>(w10, s1, b1, v1);
        mma_bf16_16816(acc[G], v0[0], v1[0], v0[1], v1[1], a0.x, a0.y);
        mma_bf16_16816(acc[G], v0[2], v1[2], v0[3], v1[3], a0.z, a0.w);
        if (kHiLo) {
            mma_bf16_16816(acc[G], v0[0], v1[0], v0[1], v1[1], l0.x, l0.y);
            mma_bf16_16816(acc[G], v0[2], v1[2], v0[3], v1[3], l0.z, l0.w);
        }
        dequant_word<kDenorm>(w01, s0, b0, v0);
        dequant_word<kDenorm>(w11, s1, b1, v1);
        mma_bf16_16816(acc[G], v0[0], v1[0], v0[1], v1[1], a1.x, a1.y);
        mma_bf16_16816(acc[G], v0[2], v1[2], v0[3], v1[3], a1.z, a1.w);
        if (kHiLo) {
            mma_bf16_16816(acc[G], v0[0], v1[0], v0[1], v1[1], l1.x, l1.y);
            mma_bf16_16816(acc[G], v0[2], v1[2], v0[3], v1[3], l1.z, l1.w);
        }
    }
}

// Top-k of the 256 logits held eight per lane (v[2 s + b] = expert 64 s + 2 lane + b) with warp
// max/min reductions, one place per round.  Lane j < k returns the expert and weight of place
// j: larger logit first, ties to the lower expert, NaN as -inf, -0 as +0; weight
// exp(l_j - l_0) / sum over the k kept logits.
__device__ __forceinline__ void warp_topk256_regs(const float (&v)[8], int k, int lane, int& out_e, float& out_w) {
    uint32_t key[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        float f = v[x];
        if (f != f) f = -INFINITY;
        if (f == 0.0f) f = 0.0f;
        const uint32_t u = __float_as_uint(f);
        key[x] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // order-preserving, never 0
    }
    int my_e = -1;
    float my_l = 0.f, l_first = 0.f;
    for (int j = 0; j < k; ++j) {
        uint32_t mx = key[0];
#pragma unroll
        for (int x = 1; x < 8; ++x) mx = max(mx, key[x]);
        const uint32_t top = __reduce_max_sync(0xffffffffu, mx);
        int cand = 0x7fffffff;
#pragma unroll
        for (int x = 7; x >= 0; --x)
            if (key[x] == top) cand = 64 * (x >> 1) + 2 * lane + (x & 1);
        const int e = __reduce_min_sync(0xffffffffu, cand);
#pragma unroll
        for (int x = 0; x < 8; ++x)
            if (64 * (x >> 1) + 2 * lane + (x & 1) == e) key[x] = 0u;
        const float l = __uint_as_float((top & 0x80000000u) ? (top & 0x7fffffffu) : ~top);
        if (j == 0) l_first = l;
        if (lane == j) { my_e = e; my_l = l; }
    }
    const float ex = lane < k ? expf(my_l - l_first) : 0.f;
    float den = ex;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) den += __shfl_xor_sync(0xffffffffu, den, m);
    out_e = my_e;
    out_w = ex / den;
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void ld_relaxed_v2u64(const unsigned long long* p, unsigned long long& a,
                                                 unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Routing results of the single token (warp-wide; lanes < k hold expert / weight of slot lane).
__device__ void write_routing_t1(const FusedDecodeArgs& a, int lane, int ee, float ww) {
    int es[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) es[j] = __shfl_sync(0xffffffffu, ee, j);
    if (lane < a.k) {
        int pos = 0;
        for (int j = 0; j < a.k; ++j) pos += es[j] < ee;   // the k experts are distinct
        a.topk_idx[lane] = ee;
        a.topk_w[lane] = ww;
        a.pos[lane] = pos;
        a.perm[pos] = lane;
        int32_t* tt = a.tiles + 3 * pos;   // one row per expert: tile i = i-th smallest expert
        tt[0] = ee; tt[1] = pos; tt[2] = 1;
    }
    for (int ex = lane; ex < a.E; ex += 32) {
        int off = 0, cnt = 0;
        for (int j = 0; j < a.k; ++j) { off += es[j] < ex; cnt += es[j] == ex; }
        a.offsets[ex] = off;
        a.counts[ex] = cnt;
    }
    if (lane == 0) { a.offsets[a.E] = a.k; *a.num_tiles = a.k; }
}

__global__ void __launch_bounds__(kFzThreads, 2) decode_fused(FzParams P) {
    const FusedDecodeArgs& a = P.a;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float s_wpart[4][2 * kTileRows];      // per-warp-pair partial sums
    __shared__ float s_part[2 * kTileRows];          // partial g (0..127) and u (128..255) of my rows
    __shared__ __align__(16) uint16_t s_hhi[kFzSlice], s_hlo[kFzSlice];   // h of my slice as bf16 hi + lo
    __shared__ uint64_t s_full[kFzRingMax], s_empty[kFzRingMax], s_xbar;
    __shared__ int s_expert, s_err;
    __shared__ float s_wgt;
    __shared__ unsigned int s_lastv[2];
    __shared__ int s_sel_e[8];
    __shared__ float s_sel_w[8];
#ifdef MOE_TRACE
    __shared__ long long s_trace[16];
    __shared__ unsigned long long s_gt0;
    if (threadIdx.x == 0) { for (int i_ = 0; i_ < 16; ++i_) s_trace[i_] = 0; s_gt0 = globaltimer_ns(); }
#endif

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = (int)cluster_ctarank();
    const int unit = blockIdx.x / kFzCluster;
    const int slot = unit / P.NS, slice = unit % P.NS;
    const bool is_shared = slot == a.k;
    const int d = a.d, E = a.E, R = P.ring;
    const int KB = d / kBK, MT = a.I / kTileRows, KQ = d / 256, ndt = d / 256, KBd = a.I / kBK;
    const int q = c;   // my column quarter of the gate/up rows
    const int my_dt = c < ndt ? (ndt - 1 - c) / kFzCluster + 1 : 0;   // 256-row output tiles c, c + 4, ...
    const int N = KQ + 2 * my_dt;
    const int units = gridDim.x / kFzCluster;
    uint8_t* ring = smem;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + (size_t)R * kChunkPairBytes);   // x [d]
    const uint16_t* xq = xs + (size_t)q * (d / 4);                                       // my column quarter
    unsigned int* st_u = reinterpret_cast<unsigned int*>(a.status);
    // warp roles in both phases: rows 128 rh .. +127 of the chunk pair, K part kp of four
    const int rh = warp & 1, kp = warp >> 1, t = lane & 3, g = lane >> 2;

    FZ_STAMP(0);
    if (tid == 0) {
        for (int i = 0; i < R; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 2); }
        mbar_init(&s_xbar, 1);
        fence_barrier_init();
        s_err = 0;
        s_expert = is_shared ? 0 : -1;
        s_wgt = 1.0f;
    }
    __syncwarp();   // (a CTA barrier does not reconverge a warp's lanes)
    __syncthreads();

    // chunk-pair address of item i for expert e of packed buffer pk (nE experts in it):
    // items 0..KQ-1 gate/up K blocks of my column quarter, then per output tile the 2 down K blocks
    // of my h slice
    auto item_addr = [&](const uint8_t* pk, int nE, int e, int i) -> const uint8_t* {
        if (i < KQ) {
            const int mt = slice, kb = q * KQ + i;
            return pk + kPackHeader + ((size_t)(e * MT + mt) * KB + kb) * kChunkPairBytes;
        }
        const int j = i - KQ, dt = c + kFzCluster * (j >> 1), kb = 2 * slice + (j & 1);
        const size_t gu_bytes = (size_t)nE * MT * KB * kChunkPairBytes;
        return pk + kPackHeader + gu_bytes + ((size_t)(e * ndt + dt) * KBd + kb) * kChunkPairBytes;
    };
    const uint8_t* pk = is_shared ? a.w_shared : a.w_routed;
    const int nE = is_shared ? 1 : E;
    auto issue = [&](int e, int i) {
        const int sl = i % R;
        mbar_arrive_expect_tx(&s_full[sl], kChunkPairBytes);
        bulk_g2s(ring + (size_t)sl * kChunkPairBytes, item_addr(pk, nE, e, i), kChunkPairBytes, &s_full[sl]);
    };
    const int first = N < R ? N : R;   // items issued at once (lane i of warp 0 issues item i)
    const int first_gu = first < KQ ? first : KQ;
    int issued = 0;                     // thread 0's count of issued items

    // ---- before the previous kernel's results are visible: weights only -------------------
    const int my_e = blockIdx.x + warp * gridDim.x;   // router row of this warp (if < E)
    uint4 wv[8];
    if (my_e < E && d <= 2048) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < d / 256) wv[i] = ld_nc_v4(a.w_router + (size_t)my_e * d + 256 * i + 8 * lane);
    }
    if (is_shared && warp == 0) {
        for (int i = lane; i < first; i += 32) issue(0, i);
        issued = first;
        __syncwarp();
    }
    pdl_wait();
    pdl_launch_dependents();
    // x (written by the previous kernel) in one bulk copy: every CTA reads all of it
    if (tid == 0) {
        mbar_arrive_expect_tx(&s_xbar, (uint32_t)d * 2);
        bulk_g2s(xs, a.x, (uint32_t)d * 2, &s_xbar);
    }
    __syncwarp();
    FZ_STAMP(1);
    // this call's tag for the published logits (the previous call's + 1)
    const unsigned int tag = ld_relaxed_u32(st_u + kStEpoch) + 1u;

    // ---- router logit(s) of this CTA, in the fixed order, published as (tag, value) words ------
    bool x_ok = true;
    if (my_e < E) {
        x_ok = mbar_spin(&s_xbar, 0, &s_err);
        float p = 0.f;
        for (int i0 = 0; i0 < d / 256; i0 += 8) {
            uint4 xv[8], wl[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i0 + i < d / 256) {
                    xv[i] = *reinterpret_cast<const uint4*>(xs + 256 * (i0 + i) + 8 * lane);
                    wl[i] = d <= 2048 ? wv[i] : ld_nc_v4(a.w_router + (size_t)my_e * d + 256 * (i0 + i) + 8 * lane);
                }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i0 + i < d / 256) {
                    p = fmaf(bf16lo(xv[i].x), bf16lo(wl[i].x), p);
                    p = fmaf(bf16hi(xv[i].x), bf16hi(wl[i].x), p);
                    p = fmaf(bf16lo(xv[i].y), bf16lo(wl[i].y), p);
                    p = fmaf(bf16hi(xv[i].y), bf16hi(wl[i].y), p);
                    p = fmaf(bf16lo(xv[i].z), bf16lo(wl[i].z), p);
                    p = fmaf(bf16hi(xv[i].z), bf16hi(wl[i].z), p);
                    p = fmaf(bf16lo(xv[i].w), bf16lo(wl[i].w), p);
                    p = fmaf(bf16hi(xv[i].w), bf16hi(wl[i].w), p);
                }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) p = p + __shfl_xor_sync(0xffffffffu, p, m);
        if (a.bias) p = p + a.bias[my_e];
        // eight copies of the word: each copy is polled by an eighth of the CTAs
        if (lane < kFzReplicas)
            st_relaxed_u64(a.logit_words + (size_t)lane * E + my_e, ((unsigned long long)tag << 32) | __float_as_uint(p));
#ifdef MOE_TRACE
        if (lane == 0 && a.trace)   // publish time per expert, after the per-CTA stamps
            a.trace[gridDim.x * 20 + my_e] = globaltimer_ns();
#endif
        __syncwarp();
    }
    FZ_STAMP(2);

    // ---- routed CTAs: wait until all E words of my copy carry this call's tag, take the top-k,
    // start the copies.  (Every CTA polling one shared copy of 16 lines made each poll take
    // microseconds; with eight copies each line has 16 pollers.)
    if (!is_shared && warp == 0) {
        const unsigned long long* words = a.logit_words + (size_t)(blockIdx.x % kFzReplicas) * E;
        float v[8];
        const long long t0 = clock64();
        bool ready = false;
#ifdef MOE_TRACE
        int npoll = 0;
#endif
        __nanosleep(kPollSleepNs);   // the logits of the other CTAs land about now
        while (true) {
#ifdef MOE_TRACE
            ++npoll;
#endif
            bool mine = true;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                unsigned long long w0, w1;
                ld_relaxed_v2u64(words + 64 * s4 + 2 * lane, w0, w1);
                mine &= (unsigned int)(w0 >> 32) == tag && (unsigned int)(w1 >> 32) == tag;
                v[2 * s4] = __uint_as_float((unsigned int)w0);
                v[2 * s4 + 1] = __uint_as_float((unsigned int)w1);
            }
            if (__all_sync(0xffffffffu, mine)) { ready = true; break; }
            if (__any_sync(0xffffffffu, clock64() - t0 > kWaitLimitCycles)) break;
            __nanosleep(kPollSleepNs);
        }
        __syncwarp();
        FZ_STAMP(3);
#ifdef MOE_TRACE
        if (lane == 0 && a.trace) {
            a.trace[gridDim.x * 20 + 256 + blockIdx.x] = globaltimer_ns();
            a.trace[gridDim.x * 20 + 512 + blockIdx.x] = (unsigned long long)npoll;
        }
        __syncwarp();
#endif
        // straight-line from here (the selection runs even after a timeout; nothing is issued then)
        int ee;
        float ww;
        warp_topk256_regs(v, a.k, lane, ee, ww);
        FZ_STAMP(12);
        const int e_slot = __shfl_sync(0xffffffffu, ee, slot);
        const float w_slot = __shfl_sync(0xffffffffu, ww, slot);
        if (ready) {
            // gate/up first: the down blocks follow once my first gate/up block has landed, so
            // that the gate/up stream (and the cluster exchange after it) finishes earlier
            for (int i = lane; i < first_gu; i += 32) issue(e_slot, i);
            issued = first_gu;
        }
        if (lane == 0) {
            if (ready) { s_expert = e_slot; s_wgt = w_slot; }
            else { s_err = 1; set_status(a.status, MOE_STATUS_TIMEOUT); }
        }
        __syncwarp();
        FZ_STAMP(4);
        if (blockIdx.x == 0 && lane < 8) { s_sel_e[lane] = ready ? ee : -1; s_sel_w[lane] = ww; }
        __syncwarp();
    }
    // every CTA has read the epoch once it gets here (routed ones have seen all tags, which
    // come after every CTA's read): the last one moves the epoch on
    if (tid == 0 && atomicAdd(st_u + kStPassed, 1u) == gridDim.x - 1) {
        atomicExch(st_u + kStEpoch, tag);
        atomicExch(st_u + kStPassed, 0u);
    }
    __syncwarp();
    __syncthreads();
    // warp votes: the branches below then are visibly warp-uniform
    const bool run = __all_sync(0xffffffffu, s_expert >= 0 && !s_err);
    const int e_me = s_expert;
    const bool denorm = __all_sync(0xffffffffu, *reinterpret_cast<const int*>(pk) == kScaleDenorm);

    // issue items < limit whose slot has been released by its two consumer warps (thread 0)
    auto refill = [&](int limit, bool block) {
        if (limit > N) limit = N;
        while (issued < limit) {
            const int sl = issued % R;
            const uint32_t par = (uint32_t)((issued / R - 1) & 1);
            if (block) {
                if (!mbar_spin(&s_empty[sl], par, &s_err)) { s_err = 1; set_status(a.status, MOE_STATUS_TIMEOUT); return; }
            } else if (!mbar_test_wait(&s_empty[sl], par)) {
                return;
            }
            issue(e_me, issued++);
        }
    };
    // Waits for item i.  The MMAs after it run whatever the outcome (a timeout only sets the
    // error flag; the sums are then discarded): warp-collective code under a branch that the
    // compiler cannot prove warp-uniform runs several times slower.
    bool ok = run;
    auto wait_item = [&](int i) {
        if (!mbar_spin(&s_full[i % R], (uint32_t)((i / R) & 1), &s_err)) {
            set_status(a.status, MOE_STATUS_TIMEOUT);
            s_err = 1;
            ok = false;
        }
    };
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);

    if (!mbar_spin(&s_xbar, 0, &s_err)) x_ok = false;
    if (!x_ok) { set_status(a.status, MOE_STATUS_TIMEOUT); ok = false; }
    // ---- gate / up: warp (rh, kp) -> matrix rh (gate, up), all 128 rows, items kp, kp + 4, ...
    {
        float acc[8][4] = {};
        for (int i = kp; i < KQ && run; i += 4) {
            wait_item(i);
            if (i == 0) FZ_STAMP(5);
            const uint8_t* ch = ring + (size_t)(i % R) * kChunkPairBytes + rh * kChunkBytes;
            const uint4 x0 = *reinterpret_cast<const uint4*>(xq + i * kBK + 8 * t);
            const uint4 x1 = *reinterpret_cast<const uint4*>(xq + i * kBK + 32 + 8 * t);
            if (denorm) chunk_rows128<true, false>(ch, lane, x0, x1, z4, z4, acc);
            else chunk_rows128<false, false>(ch, lane, x0, x1, z4, z4, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[i % R]);
            if (tid == 0) refill(N, false);
            __syncwarp();
        }
        if (t == 0) {
#pragma unroll
            for (int G = 0; G < 8; ++G) {
                s_wpart[kp][rh * kTileRows + 16 * G + g] = acc[G][0];
                s_wpart[kp][rh * kTileRows + 16 * G + g + 8] = acc[G][2];
            }
        }
        __syncwarp();
        if (tid == 0 && ok) refill(KQ, true);   // every gate/up item before the barrier below
        __syncwarp();
    }
    __syncthreads();
    s_part[tid] = s_wpart[0][tid] + s_wpart[1][tid] + s_wpart[2][tid] + s_wpart[3][tid];
    if (tid == 0 && ok) refill(KQ + R, true);    // slots freed by gate/up items
    __syncwarp();
    // ---- cluster exchange: g and u of the slice, summed over the 4 column quarters ------------
    FZ_STAMP(6);
    cluster_arrive();
    cluster_wait();
    FZ_STAMP(7);
    if (tid < kFzSlice) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int qq = 0; qq < kFzCluster; ++qq) {
            gs += ld_dsmem_f32(&s_part[tid], (uint32_t)qq);
            us += ld_dsmem_f32(&s_part[kTileRows + tid], (uint32_t)qq);
        }
        const float h = gs / (1.0f + __expf(-gs)) * us;
        const uint16_t hi = f32_to_bf16_rn(h);
        const float hif = __uint_as_float((uint32_t)hi << 16);
        s_hhi[tid] = hi;
        s_hlo[tid] = f32_to_bf16_rn(h - hif);
    }
    cluster_arrive();   // done reading the other CTAs' partials (waited for before exit)
    __syncthreads();
    FZ_STAMP(8);

    // ---- down: two output tiles per round; warp w -> tile 2 r + (w >> 2), K block kk = (w >> 1) & 1
    // of my h slice, rows 128 rh .. +127 ------------------------------------------------------
    const int kk = (warp >> 1) & 1, tp = warp >> 2;
    const uint4 h0 = *reinterpret_cast<const uint4*>(s_hhi + kk * kBK + 8 * t);
    const uint4 h1 = *reinterpret_cast<const uint4*>(s_hhi + kk * kBK + 32 + 8 * t);
    const uint4 l0 = *reinterpret_cast<const uint4*>(s_hlo + kk * kBK + 8 * t);
    const uint4 l1 = *reinterpret_cast<const uint4*>(s_hlo + kk * kBK + 32 + 8 * t);
    for (int r2 = 0; 2 * r2 < my_dt; ++r2) {
        if (tid == 0 && ok) refill(KQ + 4 * r2 + 4, true);
        __syncwarp();
        const int ti = 2 * r2 + tp;
        float acc[8][4] = {};
        if (run && ti < my_dt) {
            const int i = KQ + 2 * ti + kk;
            wait_item(i);
            const uint8_t* ch = ring + (size_t)(i % R) * kChunkPairBytes + rh * kChunkBytes;
            if (denorm) chunk_rows128<true, true>(ch, lane, h0, h1, l0, l1, acc);
            else chunk_rows128<false, true>(ch, lane, h0, h1, l0, l1, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[i % R]);
            __syncwarp();
        }
        if (t == 0) {
#pragma unroll
            for (int G = 0; G < 8; ++G) {
                s_wpart[2 * tp + kk][rh * kTileRows + 16 * G + g] = acc[G][0];
                s_wpart[2 * tp + kk][rh * kTileRows + 16 * G + g + 8] = acc[G][2];
            }
        }
        __syncwarp();
        if (tid == 0 && ok) refill(N, false);
        __syncwarp();
        __syncthreads();
        if (r2 == 0) FZ_STAMP(9);
        const int nt = my_dt - 2 * r2 < 2 ? my_dt - 2 * r2 : 2;   // tiles this pass
        // weight * partial rows go into the fp32 sum (order of the additions not fixed)
        for (int u2 = 0; u2 < nt; ++u2) {
            const int dt = c + kFzCluster * (2 * r2 + u2);
            const float v = s_wpart[2 * u2][tid] + s_wpart[2 * u2 + 1][tid];
            if (run) red_add_f32(a.acc + (size_t)dt * 256 + tid, s_wgt * v);
        }
        // the last unit to finish an output tile converts it to bf16 and clears the sum
        __threadfence();
        __syncthreads();
        if (tid < nt) s_lastv[tid] = atomicAdd(st_u + kStTiles + c + kFzCluster * (2 * r2 + tid), 1u) == (unsigned)(units - 1);
        __syncwarp();
        __syncthreads();
        for (int u2 = 0; u2 < nt; ++u2) {
            if (s_lastv[u2]) {
                __threadfence();
                const int dt = c + kFzCluster * (2 * r2 + u2), row = dt * 256 + tid;
                a.y[row] = f32_to_bf16_rn(__ldcg(a.acc + row));
                a.acc[row] = 0.f;
                if (tid == 0) st_u[kStTiles + dt] = 0u;
                __syncwarp();
            }
        }
        __syncthreads();   // s_wpart and s_lastv are reused by the next round
        if (r2 == 0) FZ_STAMP(10);
    }
    // copies still in flight after a failed wait land before the CTA leaves
    if (tid == 0 && run && s_err) {
        for (int i = 0; i < issued; ++i) {
            volatile int never = 0;
            (void)mbar_wait(&s_full[i % R], (uint32_t)((i / R) & 1), &never);
        }
    }
    // the routing results (read only after the kernel) leave the critical path: written last
    if (blockIdx.x == 0 && warp == 0) {
        const int ee = lane < 8 ? s_sel_e[lane] : -1;
        if (__all_sync(0xffffffffu, lane >= 8 || ee >= 0)) write_routing_t1(a, lane, ee, lane < 8 ? s_sel_w[lane] : 0.f);
        __syncwarp();
    }
    cluster_wait();
    FZ_STAMP(11);
    FZ_FLUSH();
}

// Per (device, shared-memory size, unit count): may the grid run (all clusters resident)?
struct FzCheck { int dev, smem, units, ok; };
std::mutex g_fz_mutex;
FzCheck g_fz_checks[32];
int g_fz_nchecks = 0;
int g_fz_smem_set[64] = {};

}  // namespace

cudaError_t launch_decode_fused(const FusedDecodeArgs& a, cudaStream_t st, unsigned long long* launches) {
    if (a.k != 8 || a.E != 256 || a.I % kFzSlice != 0 || a.d % 256 != 0) return cudaErrorNotSupported;
    const int NS = a.I / kFzSlice;
    const int units = (a.k + 1) * NS, grid = units * kFzCluster;
    if (units > kFzMaxUnits) return cudaErrorNotSupported;
    const int ndt = a.d / 256, max_items = a.d / 256 + 2 * ((ndt + kFzCluster - 1) / kFzCluster);
    if (grid < 32) return cudaErrorNotSupported;   // the grid's warps must cover the E router rows
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorNotSupported;

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kFzCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFzThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    // Can every cluster be resident at once with `smem` bytes per CTA (the grid waits on
    // itself)?  Checked once per (device, size, units).
    auto fits = [&](size_t smem, int& fit_ok) -> cudaError_t {
        std::lock_guard<std::mutex> lock(g_fz_mutex);
        fit_ok = -1;
        for (int i = 0; i < g_fz_nchecks; ++i)
            if (g_fz_checks[i].dev == dev && g_fz_checks[i].smem == (int)smem && g_fz_checks[i].units == units)
                fit_ok = g_fz_checks[i].ok;
        if (fit_ok >= 0) return cudaSuccess;
        if ((int)smem > g_fz_smem_set[dev]) {
            const cudaError_t er = cudaFuncSetAttribute(decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (er != cudaSuccess) return er;
            g_fz_smem_set[dev] = (int)smem;
        }
        cfg.dynamicSmemBytes = smem;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, decode_fused, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            nclusters = 0;
        }
        fit_ok = nclusters >= units ? 1 : 0;
        if (g_fz_nchecks < 32) g_fz_checks[g_fz_nchecks++] = FzCheck{dev, (int)smem, units, fit_ok};
        return cudaSuccess;
    };
    // ring of chunk-pair slots within `budget` bytes of shared memory per CTA (less the static
    // shared memory and x); the down rounds' refills need 5 slots unless every item fits at once
    auto ring_for = [&](size_t budget) {
        const int fit = (int)((budget - 8192 - 2 * (size_t)a.d) / kChunkPairBytes);
        int r = max_items < kFzRingMax ? max_items : kFzRingMax;
        if (r > fit) r = fit;
        return r < max_items && r < 5 ? 0 : r;
    };
    // First choice: one CTA of this grid per SM (a CTA that shared its SM with another of the
    // same layer ran ~1.5 us behind the others and held up the whole layer: 16.2 -> 15.5 us per
    // layer at d = 2048, I = 512); more than half of an SM's shared memory keeps a second one
    // out.  Grids with more clusters than fit that way take two CTAs per SM (116736 bytes each).
    int ring = 0, fit_ok = 0;
    size_t smem = 0;
    const int r1 = ring_for(232448);
    if (r1 > 0) {
        smem = (size_t)r1 * kChunkPairBytes + (size_t)a.d * 2;
        if (smem < (size_t)kFzOneCtaSmem) smem = kFzOneCtaSmem;
#ifdef MOE_FZ_MIN_SMEM
        if (smem < (size_t)(MOE_FZ_MIN_SMEM)) smem = MOE_FZ_MIN_SMEM;   // tuning builds
#endif
        if ((e = fits(smem, fit_ok)) != cudaSuccess) return e;
        ring = r1;
    }
    if (!fit_ok) {
        const int r2 = ring_for(116736);
        if (r2 == 0) return cudaErrorNotSupported;
        smem = (size_t)r2 * kChunkPairBytes + (size_t)a.d * 2;
        if ((e = fits(smem, fit_ok)) != cudaSuccess) return e;
        ring = r2;
    }
    if (!fit_ok) return cudaErrorNotSupported;
    FzParams P{a, NS, ring};
    cfg.dynamicSmemBytes = smem;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, decode_fused, P);
    *launches += 1;
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace moe
