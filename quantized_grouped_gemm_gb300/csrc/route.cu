// route.cu -- GPU-resident expert routing (no host round trip).
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026):
//   section "Qwen creates three different workload shapes": a router scores 256 experts per
//   token and keeps eight, plus one shared expert;
//   section "Keep expert routing on the GPU": a histogram counts assignments per expert, a
//   prefix scan turns counts into start offsets, a scatter places rows into their expert
//   groups, and a block map lists the fixed-size tiles for the grouped GEMM -- all enqueued
//   without a CPU stop inside the layer.
//
// Prefill (five launches):
//   router_wnorm       ||W_r[e]|| per expert (for the error bound below).
//   router_tc          approximate logits on the tensor cores (tcgen05, K-sliced partials).
//   route_certify_topk per token: an error bound picks the candidates that can be in the top-8
//                      of the fixed-order logits; only those are recomputed exactly (CUDA
//                      cores, fixed fp32 order) and ranked; weights; per-block counts.
//   route_scan         8 CTAs: per-block bases, counts, offsets, the exported block map
//                      and the GEMM tile lists (expert, first row, rows, weight tile).
//   route_scatter      one CTA per (block, slot): stable group positions (rank of the token among
//                      the block's tokens routed to the same expert, from a bitmask), perm /
//                      pos and the gathered rows xs.
// Decode (one launch): route_decode -- a warp per expert logit, the last CTA to finish
// does top-8 and the metadata for the few tokens.
#include <algorithm>
#include <vector>

#include "moe_internal.cuh"

namespace moe {
namespace {


// ---------------------------------------------------------------------------------------
// Exact logit of (token row xrow, expert row wrow) in the fixed order, computed by one warp:
// lane l is partial sum l (columns 256*i + 8*l + j, i ascending, j = 0..7, fmaf from 0); the
// xor-shuffle tree over 16, 8, 4, 2, 1 pairs the same lanes as s[i] += s[i+m].  Every lane
// returns the logit (+ bias).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_pinned_logit(const uint16_t* xrow, const uint16_t* wrow, int d, int lane,
                                                   const float* bias_e) {
    float p = 0.f;
    for (int i = 0; i < d / 256; ++i) {
        const int col = 256 * i + 8 * lane;
        const uint4 xv = ld_nc_v4(xrow + col);
        const uint4 wv = ld_nc_v4(wrow + col);
        p = fmaf(bf16lo(xv.x), bf16lo(wv.x), p);
        p = fmaf(bf16hi(xv.x), bf16hi(wv.x), p);
        p = fmaf(bf16lo(xv.y), bf16lo(wv.y), p);
        p = fmaf(bf16hi(xv.y), bf16hi(wv.y), p);
        p = fmaf(bf16lo(xv.z), bf16lo(wv.z), p);
        p = fmaf(bf16hi(xv.z), bf16hi(wv.z), p);
        p = fmaf(bf16lo(xv.w), bf16lo(wv.w), p);
        p = fmaf(bf16hi(xv.w), bf16hi(wv.w), p);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) p = p + __shfl_xor_sync(0xffffffffu, p, m);
    if (bias_e) p = p + *bias_e;
    return p;
}

// ---------------------------------------------------------------------------------------
// router_wnorm: ||W_r[e]||_2 (fp32) for every expert; one warp per expert.  It reads only the
// router weight, so it runs before waiting for the previous kernel on the stream (programmatic
// dependent launch); the wait comes before the result is written, so the launch order of the
// workspace writes is kept.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) router_wnorm(RouteArgs a) {
    const int lane = threadIdx.x & 31, e = blockIdx.x * 4 + (threadIdx.x >> 5);
    float s = 0.f;
    for (int c = 8 * lane; c < a.d; c += 256) {
        const uint4 v = ld_nc_v4(a.w_router + (size_t)e * a.d + c);
        const float f[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                            bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
#pragma unroll
        for (int j = 0; j < 8; ++j) s = fmaf(f[j], f[j], s);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0) reinterpret_cast<float*>(a.ws + a.L.wnorm)[e] = sqrtf(s);
}

// ---------------------------------------------------------------------------------------
// router_tc: approximate logits on the tensor cores.  grid = (ceil(T/128) token blocks,
// KS K-slices); CTA (b, s) computes the partial product of 128 tokens x all 256 experts over
// its K slice (tcgen05.mma M=128 x N=256 x K=16, operands by TMA with 128-byte swizzle, fp32
// accumulator in TMEM) and writes it to part[s][t][256].  Only used to pick candidates.
// Warps: 0 producer, 1 MMA + TMEM owner, 2..5 epilogue (one token row per thread).
// ---------------------------------------------------------------------------------------
constexpr int kRtStages = 4;
constexpr int kRtA = 128 * 128;   // 128 tokens x 64 bf16
constexpr int kRtB = 256 * 128;   // 256 experts x 64 bf16
constexpr int kRtSmem = kRtStages * (kRtA + kRtB) + 256 + 1024;
constexpr int kRtRowStride = 1040;   // epilogue staging: 128 rows of 1 KB partial logits, padded
static_assert(128 * kRtRowStride <= kRtStages * (kRtA + kRtB), "router_tc epilogue staging");

__global__ void __launch_bounds__(192, 1)
    router_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, RouteArgs a,
              int KS) {
    extern __shared__ uint8_t smem_dyn[];
    const uint32_t s0 = smem_u32(smem_dyn);
    uint8_t* smem = smem_dyn + ((1024u - (s0 & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRtStages * (kRtA + kRtB));
    uint64_t* empty = full + kRtStages;
    uint64_t* tmfull = empty + kRtStages;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(tmfull + 1);
    int* abortp = reinterpret_cast<int*>(tslot + 1);
    volatile int* abort = abortp;
    int* status = reinterpret_cast<int*>(a.ws + a.L.status);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.d / kBK, kb0 = blockIdx.y * KB / KS, kb1 = (blockIdx.y + 1) * KB / KS;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRtStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
        mbar_init(tmfull, 1);
        *abortp = 0;
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc(tslot, 256); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the router-weight tiles of the first stages do not depend on the previous kernel: they are
    // requested before the wait (the stage barrier expects their bytes, and the token tiles'
    // bytes and the producer's arrival after the wait)
    const int npre = kb1 - kb0 < kRtStages ? kb1 - kb0 : kRtStages;
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_w);
        for (int i = 0; i < npre; ++i) {
            mbar_expect_tx(&full[i], kRtB);
            tma_load_2d(smem + i * (kRtA + kRtB) + kRtA, &tm_w, (kb0 + i) * kBK, 0, &full[i]);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    // producer (warp 0) and MMA issuer (warp 1) walk their loops with the whole warp, so counters
    // and descriptors stay warp-uniform; one elected lane issues
    if (warp == 0) {
        const bool leader = elect_one();
        if (leader) prefetch_tmap(&tm_x);
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int st = it % kRtStages;
            if (!mbar_wait_warp(&empty[st], ((it / kRtStages) & 1) ^ 1, abort)) {
                if (leader) {
                    *abort = 1;
                    set_status(status, MOE_STATUS_TIMEOUT);
                }
                break;
            }
            if (leader) {
                uint8_t* dst = smem + st * (kRtA + kRtB);
                if ((int)it < npre) {   // router-weight tile already requested
                    mbar_arrive_expect_tx(&full[st], kRtA);
                } else {
                    mbar_arrive_expect_tx(&full[st], kRtA + kRtB);
                    tma_load_2d(dst + kRtA, &tm_w, kb * kBK, 0, &full[st]);
                }
                tma_load_2d(dst, &tm_x, kb * kBK, blockIdx.x * 128, &full[st]);
            }
            __syncwarp();
        }
        // every issued copy lands before the CTA can exit (including router-weight tiles
        // requested before the wait for stages the loop did not reach after a timeout)
        if (leader) {
            int never = 0;
            const uint32_t last = it > (uint32_t)npre ? it : (uint32_t)npre;
            const uint32_t first = last > (uint32_t)kRtStages ? last - kRtStages : 0;
            for (uint32_t i = first; i < last; ++i) mbar_wait(&full[i % kRtStages], (i / kRtStages) & 1, &never);
        }
        __syncwarp();
    } else if (warp == 1) {
        const bool leader = elect_one();
        const uint32_t idesc = idesc_bf16_f32(128, 256);
        const uint32_t base = smem_u32(smem);
        uint32_t it = 0;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int st = it % kRtStages;
            if (!mbar_wait_warp(&full[st], (it / kRtStages) & 1, abort)) { ok = false; break; }
            tc_fence_after();
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t sa = base + st * (kRtA + kRtB);
                    tc_mma_bf16(tmem, sw128_desc(sa + ks * 32), sw128_desc(sa + kRtA + ks * 32), idesc,
                                (kb > kb0 || ks) ? 1u : 0u);
                }
                tc_commit(&empty[st]);
            }
            __syncwarp();
        }
        if (leader) {
            if (!ok) { *abort = 1; set_status(status, MOE_STATUS_TIMEOUT); }
            tc_commit(tmfull);     // also drains every MMA before the epilogue / dealloc
        }
        __syncwarp();
    } else {
        // epilogue: thread -> token row 32 q + lane.  Its 256 partial logits go from TMEM into a
        // padded row of shared memory (the operand stages, free once every MMA has completed;
        // the 1040-byte row stride keeps the 16-byte stores of 8 consecutive threads on distinct
        // banks), then out as one 1 KB bulk copy per row.
        const int q = warp & 3, rl = 32 * q + lane;
        const bool got = mbar_wait(tmfull, 0, abort);
        if (__all_sync(0xffffffffu, got)) {
            tc_fence_after();
            const int t = blockIdx.x * 128 + rl;
            float* srow = reinterpret_cast<float*>(smem + (size_t)rl * kRtRowStride);
            for (int c = 0; c < 16; ++c) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 16 * c, v);
                tmem_ld_wait();
                float4* d4 = reinterpret_cast<float4*>(srow + 16 * c);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    d4[u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                        __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
            }
            if (t < a.T) {
                fence_proxy_async_smem();
                float* dst = reinterpret_cast<float*>(a.ws + a.L.rpart) + ((size_t)blockIdx.y * a.T + t) * 256;
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], 1024;" ::"l"(dst),
                             "r"(smem_u32(srow))
                             : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // before the CTA's smem goes
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------------------
// route_certify_topk (the bound): for each token, with l~[e] the tensor-core logit (sum of the
// K slices, + bias) and
//   delta[e] = c * ||x_t|| * ||W_r[e]||,  c = 2 * ((d + KS + 35) * 2^-23)  (+ a bias term),
// which bounds |l~[e] - l[e]| for the fixed-order logit l (any fp32 summation of d exact
// products errs by at most ~d*2^-23 * sum|x w| <= d*2^-23 ||x|| ||w||; the fixed order by
// 69*2^-24 of the same; factor 2 for margin):
//   lo = min over the 8 largest l~ of (l~[e] - delta[e]) <= the 8th largest l,
// so every expert of the exact top-8 has l~[f] + delta[f] >= lo.  Those candidates (usually
// ~10) are recomputed exactly (warp_pinned_logit) and ranked; over 32 candidates, all 256
// are recomputed.  The result equals top-8 over all 256 exact logits.
// Also writes the block's per-expert counts.
// ---------------------------------------------------------------------------------------
// p = fma(x.lo, w.lo, p), then p = fma(x.hi, w.hi, p), for the bf16 halves of two 32-bit words
// (bf16 -> fp32 is exact, so each step rounds once)
__device__ __forceinline__ float fma2_bf16(uint32_t x, uint32_t w, float p) {
    p = fmaf(bf16lo(x), bf16lo(w), p);
    return fmaf(bf16hi(x), bf16hi(w), p);
}

// Exact logits (fixed order, as warp_pinned_logit) of G experts for the token row held in
// registers, with all G rows' loads issued before the arithmetic.
template <int NI, int G>
__device__ __forceinline__ void warp_pinned_logits(const uint4 (&xv)[8], const uint16_t* const (&w)[G], int lane,
                                                   float (&l)[G]) {
    uint4 a[G][NI];
#pragma unroll
    for (int i = 0; i < NI; ++i)
#pragma unroll
        for (int g = 0; g < G; ++g) a[g][i] = ld_nc_v4(w[g] + 256 * i + 8 * lane);
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) p[g] = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            p[g] = fma2_bf16(xv[i].x, a[g][i].x, p[g]);
            p[g] = fma2_bf16(xv[i].y, a[g][i].y, p[g]);
            p[g] = fma2_bf16(xv[i].z, a[g][i].z, p[g]);
            p[g] = fma2_bf16(xv[i].w, a[g][i].w, p[g]);
        }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) p[g] = p[g] + __shfl_xor_sync(0xffffffffu, p[g], m);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) l[g] = p[g];
}

// Exact logits of G experts for one token: NI = d / 256 column groups with the token row in
// registers (NI <= 8), or NI = 0 for any other d (rows read from memory, one logit at a time).
template <int NI, int G>
__device__ __forceinline__ void pinned_logit_group(const uint4 (&xv)[8], const uint16_t* xrow, const uint16_t* w_router,
                                                   int d, const int (&e)[G], int lane, float (&l)[G]) {
    const uint16_t* w[G];
#pragma unroll
    for (int g = 0; g < G; ++g) w[g] = w_router + (size_t)e[g] * d;
    if constexpr (NI > 0) {
        warp_pinned_logits<NI, G>(xv, w, lane, l);
    } else {
#pragma unroll
        for (int g = 0; g < G; ++g) l[g] = warp_pinned_logit(xrow, w[g], d, lane, nullptr);
    }
}

// Sum of the KS K-slice partial logits of experts 8*lane .. 8*lane+7 (slice order).
template <int KS>
__device__ __forceinline__ void sum_kslices(const float* p, size_t qstride, float (&lt)[8]) {
    float4 v[KS][2];
#pragma unroll
    for (int q = 0; q < KS; ++q) {
        v[q][0] = ld_nc_f4(p + q * qstride);
        v[q][1] = ld_nc_f4(p + q * qstride + 4);
    }
#pragma unroll
    for (int q = 0; q < KS; ++q) {
        lt[0] += v[q][0].x; lt[1] += v[q][0].y; lt[2] += v[q][0].z; lt[3] += v[q][0].w;
        lt[4] += v[q][1].x; lt[5] += v[q][1].y; lt[6] += v[q][1].z; lt[7] += v[q][1].w;
    }
}

// Order key of a logit (NaN as -inf, -0 as +0); larger key = larger logit, never 0.
__device__ __forceinline__ uint32_t logit_key32(float f) {
    if (f != f) f = -INFINITY;
    if (f == 0.0f) f = 0.0f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key32_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ---------------------------------------------------------------------------------------
// route_certify_topk: one warp per token, kCertTokens tokens per CTA; lane l holds experts
// 8l .. 8l+7.  From the tensor-core partial logits l~ and the bound delta of each expert it
// keeps the candidates l~ + delta >= lo with lo = (8th largest l~) - max delta (at least eight
// experts have an exact logit >= lo, so no other expert can be in the exact top-8),
// recomputes their exact logits in the fixed order, kCertGroup at a time (each warp's time is
// a chain of L2 round trips, so every load of a group is in flight at once), and takes the
// top-k among them.  More than 32 candidates: all 256 are recomputed.  Per-block expert counts
// are added for the scan.
// ---------------------------------------------------------------------------------------
#ifndef MOE_CERT_TOKENS
#define MOE_CERT_TOKENS 8
#endif
// tokens (warps) per CTA: few, so that a small chunk still spreads over the SMs (each warp's
// exact recomputation is a chain of L2 loads; 2, 4, 8 and 16 measured within 10 % of each
// other at 512 tokens, 8 the fastest); divides the 32-token routing block
constexpr int kCertTokens = MOE_CERT_TOKENS;
static_assert(kRouteBlockTokens % kCertTokens == 0, "certify tokens per CTA");
#ifndef MOE_CERT_GROUP
#define MOE_CERT_GROUP 4
#endif
constexpr int kCertGroup = MOE_CERT_GROUP;   // exact logits per round
static_assert(kCertGroup >= 1 && 256 % kCertGroup == 0, "certify group");

template <int NI>
__global__ void __launch_bounds__(32 * kCertTokens, 2) route_certify_topk(RouteArgs a, int KS) {
    __shared__ uint32_t s_mask[256];
    __shared__ float s_all[kCertTokens][256];
    __shared__ int s_cand[kCertTokens][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tok = blockIdx.x * kCertTokens + warp;
    const float* part = reinterpret_cast<const float*>(a.ws + a.L.rpart);
    const float* wnorm = reinterpret_cast<const float*>(a.ws + a.L.wnorm);
    const float c = 2.0f * (float)(a.d + KS + 35) * 1.1920928955078125e-7f;   // 2^-23
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_mask[i] = 0;
    __syncthreads();
    if (tok < a.T) {
        const uint16_t* xrow = a.x + (size_t)tok * a.d;
        // the token row in registers (first 8 column groups) and ||x_t||
        uint4 xv[8];
        float nx = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xv[i] = make_uint4(0, 0, 0, 0);
            if (i < a.d / 256) xv[i] = ld_nc_v4(xrow + 256 * i + 8 * lane);
        }
        float lt[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, dl[8], wn[8];
        {
            const float* p = part + (size_t)tok * 256 + 8 * lane;
            const size_t qs = (size_t)a.T * 256;
            switch (KS) {
                case 1: sum_kslices<1>(p, qs, lt); break;
                case 2: sum_kslices<2>(p, qs, lt); break;
                case 4: sum_kslices<4>(p, qs, lt); break;
                case 8: sum_kslices<8>(p, qs, lt); break;
                case 16: sum_kslices<16>(p, qs, lt); break;
                default:
                    for (int q = 0; q < KS; ++q) sum_kslices<1>(p + q * qs, qs, lt);
            }
            const float4 w0 = ld_nc_f4(wnorm + 8 * lane), w1 = ld_nc_f4(wnorm + 8 * lane + 4);
            wn[0] = w0.x; wn[1] = w0.y; wn[2] = w0.z; wn[3] = w0.w;
            wn[4] = w1.x; wn[5] = w1.y; wn[6] = w1.z; wn[7] = w1.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float f[8] = {bf16lo(xv[i].x), bf16hi(xv[i].x), bf16lo(xv[i].y), bf16hi(xv[i].y),
                                bf16lo(xv[i].z), bf16hi(xv[i].z), bf16lo(xv[i].w), bf16hi(xv[i].w)};
#pragma unroll
            for (int j = 0; j < 8; ++j) nx = fmaf(f[j], f[j], nx);
        }
        for (int col = 2048 + 8 * lane; col < a.d; col += 256) {
            const uint4 v = ld_nc_v4(xrow + col);
            const float f[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                                bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
#pragma unroll
            for (int j = 0; j < 8; ++j) nx = fmaf(f[j], f[j], nx);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) nx += __shfl_xor_sync(0xffffffffu, nx, m);
        nx = sqrtf(nx);
        float dmax = 0.f;
        uint32_t key[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int e = 8 * lane + s;
            const float b = a.bias ? a.bias[e] : 0.f;
            lt[s] += b;
            dl[s] = c * nx * wn[s] + 4.7683716e-7f * (fabsf(lt[s]) + fabsf(b) + 1.0f);   // + 2^-21 (|l|+|b|+1)
            dmax = fmaxf(dmax, dl[s]);
            key[s] = logit_key32(lt[s]);
        }
        dmax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(dmax)));   // dmax >= 0
        // the 8th largest l~ (with multiplicity): each lane sorts its eight keys (descending,
        // Batcher's odd-even merge network), then eight rounds each remove the head of the lowest
        // lane holding the largest head
        {
            auto cx = [&](int i, int j) {   // key[i] >= key[j] afterwards
                const uint32_t hi = max(key[i], key[j]), lo = min(key[i], key[j]);
                key[i] = hi;
                key[j] = lo;
            };
            cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
            cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
            cx(1, 2); cx(5, 6);
            cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
            cx(2, 4); cx(3, 5);
            cx(1, 2); cx(3, 4); cx(5, 6);
        }
        uint32_t top = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            top = __reduce_max_sync(0xffffffffu, key[0]);
            const uint32_t holders = __ballot_sync(0xffffffffu, key[0] == top);
            if (lane == __ffs(holders) - 1) {
#pragma unroll
                for (int s = 0; s < 7; ++s) key[s] = key[s + 1];
                key[7] = 0u;
            }
        }
        const float lo = __fsub_rd(key32_logit(top), dmax);
        uint32_t cm[8];
        int ncand = 0;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const bool cand = !(__fadd_ru(lt[s], dl[s]) < lo);      // NaN-safe: NaN stays a candidate
            cm[s] = __ballot_sync(0xffffffffu, cand);
            ncand += __popc(cm[s]);
        }
        int e_out;
        float w_out;
        if (ncand <= 32) {
            // candidate j goes to lane j (listed by s, then lane)
            int before = 0;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if (cm[s] >> lane & 1u) s_cand[warp][before + __popc(cm[s] & ((1u << lane) - 1u))] = 8 * lane + s;
                before += __popc(cm[s]);
            }
            __syncwarp();
            int my_e = -1;
            float my_l = -INFINITY;
            // rounds of kCertGroup candidates, then the remaining one to three in rounds of 2 and 1
            // (every load of a round is in flight at once)
            auto round = [&](auto gsz, int j0) {
                constexpr int G = decltype(gsz)::value;
                int eg[G];
#pragma unroll
                for (int g = 0; g < G; ++g) eg[g] = s_cand[warp][j0 + g];
                float lg[G];
                pinned_logit_group<NI, G>(xv, xrow, a.w_router, a.d, eg, lane, lg);
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (lane == j0 + g) { my_e = eg[g]; my_l = a.bias ? lg[g] + a.bias[eg[g]] : lg[g]; }
            };
            int j0 = 0;
            for (; j0 + kCertGroup <= ncand; j0 += kCertGroup) round(std::integral_constant<int, kCertGroup>{}, j0);
            if (ncand - j0 >= 2) {
                round(std::integral_constant<int, 2>{}, j0);
                j0 += 2;
            }
            if (ncand - j0 == 1) round(std::integral_constant<int, 1>{}, j0);
            // top-k among the exact candidate logits, one per lane
            uint32_t k1 = my_e >= 0 ? logit_key32(my_l) : 0u;
            int sel_e = -1;
            float sel_l = 0.f, l0 = 0.f;
            for (int jj = 0; jj < a.k; ++jj) {
                const uint32_t best = __reduce_max_sync(0xffffffffu, k1);
                const int e = __reduce_min_sync(0xffffffffu, (k1 == best && my_e >= 0) ? my_e : 0x7fffffff);
                if (my_e == e) k1 = 0u;
                const float lc = key32_logit(best);
                if (jj == 0) l0 = lc;
                if (lane == jj) { sel_e = e; sel_l = lc; }
            }
            const float ex = lane < a.k ? expf(sel_l - l0) : 0.f;
            float den = ex;
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) den += __shfl_xor_sync(0xffffffffu, den, m);
            e_out = sel_e;
            w_out = ex / den;
        } else {
            for (int e0 = 0; e0 < 256; e0 += kCertGroup) {
                int eg[kCertGroup];
#pragma unroll
                for (int g = 0; g < kCertGroup; ++g) eg[g] = e0 + g;
                float lg[kCertGroup];
                pinned_logit_group<NI, kCertGroup>(xv, xrow, a.w_router, a.d, eg, lane, lg);
#pragma unroll
                for (int g = 0; g < kCertGroup; ++g)
                    if (lane == ((e0 + g) & 31)) s_all[warp][e0 + g] = a.bias ? lg[g] + a.bias[e0 + g] : lg[g];
            }
            __syncwarp();
            warp_topk256(s_all[warp], a.k, lane, e_out, w_out);
        }
        if (lane < a.k) {
            a.topk_idx[(size_t)tok * a.k + lane] = e_out;
            a.topk_w[(size_t)tok * a.k + lane] = w_out;
            atomicOr(&s_mask[e_out], 1u << warp);
        }
        __syncwarp();
    }
    __syncthreads();
    // per 32-token block counts (cleared by route_scatter once route_scan has read them)
    int32_t* blk_counts = reinterpret_cast<int32_t*>(a.ws + a.L.blk);
    const size_t blk = (size_t)blockIdx.x * kCertTokens / kRouteBlockTokens;
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (s_mask[i]) atomicAdd(&blk_counts[blk * 256 + i], __popc(s_mask[i]));
}

// ---------------------------------------------------------------------------------------
// route_scan: kScanCtas CTAs of 1024 threads.  In every CTA thread (e, part) sums the counts of
// expert e over a quarter of the token blocks, and the CTA computes the counts, offsets
// (exclusive scan over experts) and the per-expert tile scans; the writes are shared out: CTA c
// writes the per-block bases of experts [32c, 32c + 32) (kScanCtas = 8) and its contiguous
// share of the exported block map and of each GEMM tile list; CTA 0 writes counts, offsets and
// the list lengths.  (The per-block counts are cleared by route_scatter, which runs after every
// CTA here has read them.)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int block_exclusive_scan256(int v, int* s_tmp) {
    // called by the 256 threads of warps 0..7 only; s_tmp has 8 ints; uses named barrier 1
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, m);
        if (lane >= m) x += y;
    }
    named_bar_sync(1, 256);
    if (lane == 31) s_tmp[warp] = x;
    named_bar_sync(1, 256);
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_tmp[w];
    return base + x - v;
}

// The expert owning entry t of a list whose per-expert entry counts have the exclusive scan
// sc[0..256] (sc[256] = total, t < total): the largest e with sc[e] <= t, which has sc[e + 1] > t.
__device__ __forceinline__ int scan_owner(const int* sc, int t) {
    int lo = 0, hi = 256;
#pragma unroll
    for (int step = 0; step < 8; ++step) {
        const int mid = (lo + hi) >> 1;
        if (sc[mid] <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Entries j0 <= j < j1 of a GEMM tile list, written by the CTA's threads: position j holds the shared
// expert's entry j - from when from <= j < from + nsh * mt, else routed entry jj (jj = j before
// the shared block, j - nsh * mt after it) = (token block jj / mt, weight tile jj % mt) of the
// routed experts' blocks in expert order (sb: exclusive scan of their block counts).  An
// expert's cnt rows from off are cut into nb near-equal blocks: block i has q + (i < r) rows
// (q = cnt / nb, r = cnt % nb) and starts at off + i q + min(i, r); the shared expert cuts the
// T token rows the same way into nsh blocks.  Entry = (expert, first row, rows, weight tile).
__device__ void gemm_list_entries(int4* list, int j0, int j1, int mt, int nsh, int from, const int* sb,
                                  const int* cnt, const int* off, int T, int E) {
    const int nsh_e = nsh * mt;
    for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        int ex, i, m, rows, nb, r0;
        if (j >= from && j < from + nsh_e) {
            const int q = j - from;
            ex = E; i = q / mt; m = q % mt; rows = T; nb = nsh; r0 = 0;
        } else {
            const int jj = j < from ? j : j - nsh_e;
            const int blk = jj / mt;
            m = jj % mt;
            ex = scan_owner(sb, blk);
            i = blk - sb[ex];
            rows = cnt[ex]; nb = sb[ex + 1] - sb[ex]; r0 = off[ex];
        }
        const int q = rows / nb, r = rows % nb;
        list[j] = make_int4(ex, r0 + i * q + min(i, r), q + (i < r ? 1 : 0), m);
    }
}

constexpr int kScanCtas = 8;
__global__ void __launch_bounds__(1024) route_scan(RouteArgs a) {
    __shared__ int s_tmp[8];
    __shared__ int s_part[4][256];
    __shared__ int s_off[256];
    __shared__ int s_cnt[256];
    __shared__ int s_tb[257], s_gb[257], s_db[257];   // exclusive scans: block-map tiles, GEMM blocks
    pdl_wait();
    pdl_launch_dependents();
    const int E = 256, cta = blockIdx.x, S = gridDim.x;
    const int e = threadIdx.x & 255, part = threadIdx.x >> 8;
    const bool own_e = (e * S) / E == cta;   // this CTA writes the per-block bases of expert e
    int32_t* blk_counts = reinterpret_cast<int32_t*>(a.ws + a.L.blk);
    int32_t* blk_base = blk_counts + (size_t)a.L.nblk * E;
    const int nb = a.L.nblk, nq = (nb + 3) / 4;
    const int b0 = min(nb, part * nq), b1 = min(nb, b0 + nq);
    // Up to kScanRegs blocks per thread (T <= 4096) are loaded once, all in flight, and kept in
    // registers for the per-block bases; longer chunks read their counts twice in batches of 8.
    constexpr int kScanRegs = 32;
    const bool in_regs = nq <= kScanRegs;
    int creg[kScanRegs];
    int sum = 0;
    if (in_regs) {
#pragma unroll
        for (int u = 0; u < kScanRegs; ++u) creg[u] = b0 + u < b1 ? blk_counts[(size_t)(b0 + u) * E + e] : 0;
#pragma unroll
        for (int u = 0; u < kScanRegs; ++u) sum += creg[u];
    } else {
        int b = b0;
        for (; b + 8 <= b1; b += 8) {
            int c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = blk_counts[(size_t)(b + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) sum += c[u];
        }
        for (; b < b1; ++b) sum += blk_counts[(size_t)b * E + e];
    }
    s_part[part][e] = sum;
    __syncthreads();
    int pre = 0, run = 0;
    for (int q = 0; q < 4; ++q) {
        if (q < part) pre += s_part[q][e];
        run += s_part[q][e];
    }
    if (part == 0) {
        const int off = block_exclusive_scan256(run, s_tmp);
        s_off[e] = off;
        if (cta == 0) {
            a.counts[e] = run;
            a.offsets[e] = off;
            if (e == E - 1) a.offsets[E] = off + run;
        }
    }
    __syncthreads();
    // per-block bases: offsets[e] + counts of e in earlier blocks
    if (own_e && in_regs) {
        int r = s_off[e] + pre;
#pragma unroll
        for (int u = 0; u < kScanRegs; ++u) {
            if (b0 + u < b1) blk_base[(size_t)(b0 + u) * E + e] = r;
            r += creg[u];
        }
    } else if (own_e) {
        int r = s_off[e] + pre;
        int b = b0;
        for (; b + 8 <= b1; b += 8) {
            int c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = blk_counts[(size_t)(b + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                blk_base[(size_t)(b + u) * E + e] = r;
                r += c[u];
            }
        }
        for (; b < b1; ++b) {
            blk_base[(size_t)b * E + e] = r;
            r += blk_counts[(size_t)b * E + e];
        }
    }
    // per expert: tiles of the exported block map and token blocks of the two GEMM tile lists,
    // and their exclusive scans over the experts (warps 0..7, named barrier 1)
    if (part == 0) {
        s_cnt[e] = run;
        const int nt = (run + a.tile_rows - 1) / a.tile_rows;
        const int nn = (run + a.gu_rows - 1) / a.gu_rows;
        const int nd = (run + a.dn_rows - 1) / a.dn_rows;
        const int tb = block_exclusive_scan256(nt, s_tmp);
        s_tb[e] = tb;
        if (e == E - 1) s_tb[E] = tb + nt;
        named_bar_sync(1, 256);
        const int gb = block_exclusive_scan256(nn, s_tmp);
        s_gb[e] = gb;
        if (e == E - 1) s_gb[E] = gb + nn;
        named_bar_sync(1, 256);
        const int db = block_exclusive_scan256(nd, s_tmp);
        s_db[e] = db;
        if (e == E - 1) s_db[E] = db + nd;
    }
    __syncthreads();

    // Every entry of the three lists is a function of its position, so all threads write them
    // (an expert's entries are not left to one thread: a heavy expert has hundreds).
    // Exported block map: ceil(count / tile_rows) tiles per expert, expert-ascending.
    const int BM = a.tile_rows;
    const int ntile = s_tb[E];
    for (int t = (int)((long long)ntile * cta / S) + threadIdx.x; t < (int)((long long)ntile * (cta + 1) / S);
         t += blockDim.x) {
        const int ex = scan_owner(s_tb, t), i = t - s_tb[ex];
        int32_t* tt = a.tiles + 3 * (size_t)t;
        tt[0] = ex;
        tt[1] = s_off[ex] + i * BM;
        tt[2] = min(BM, s_cnt[ex] - i * BM);
    }
    // GEMM tile lists: an expert's rows split into near-equal token blocks of at most
    // a.gu_rows (gate/up) and a.dn_rows (down) rows (moe_options.gemm_rows); each block is
    // repeated for every weight tile (weight tile innermost, so the CTAs that run at the same
    // time share the block's activation rows in L2).  The shared expert (expert index E)
    // covers token rows 0..T-1 in full blocks; its entries sit at positions [from, from + its
    // count) -- where the persistent CTAs run one tile fewer (shared_tiles_at) -- and the
    // experts' entries follow in expert order around them.
    const int MTgu = a.I / kTileRows, MTdn = a.d / 256;   // 128 gate+up row pairs; 256-row down tiles
    const int nsh = (a.T + a.gu_rows - 1) / a.gu_rows;
    const int nshd = (a.T + a.dn_rows - 1) / a.dn_rows;
    const int ngu = (nsh + s_gb[E]) * MTgu, ndn = (nshd + s_db[E]) * MTdn;
    const int pg = shared_tiles_at(ngu, nsh * MTgu, a.num_sms);
    const int pd = shared_tiles_at(ndn, nshd * MTdn, a.num_sms);
    gemm_list_entries(reinterpret_cast<int4*>(a.ws + a.L.gu_tiles), (int)((long long)ngu * cta / S),
                      (int)((long long)ngu * (cta + 1) / S), MTgu, nsh, pg, s_gb, s_cnt, s_off, a.T, E);
    gemm_list_entries(reinterpret_cast<int4*>(a.ws + a.L.dn_tiles), (int)((long long)ndn * cta / S),
                      (int)((long long)ndn * (cta + 1) / S), MTdn, nshd, pd, s_db, s_cnt, s_off, a.T, E);
    if (cta == 0 && threadIdx.x == 0) {
        *a.num_tiles = ntile;
        *reinterpret_cast<int32_t*>(a.ws + a.L.gu_num) = ngu;
        *reinterpret_cast<int32_t*>(a.ws + a.L.dn_num) = ndn;
    }
}

// ---------------------------------------------------------------------------------------
// route_scatter: grid = (ceil(T/32) blocks, k slots), 256 threads.  Every CTA rebuilds the
// block's expert bitmasks (bit t set when token t of the block picked the expert), which
// give the stable rank of a token among the block's tokens routed to the same expert; CTA
// (b, j) then writes pos / perm of slot j and copies those 32 rows into expert order
// (xs[p] = x[t]); CTA (b, 0) also clears the block's per-expert counts for the next call.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) route_scatter(RouteArgs a) {
    __shared__ uint32_t s_mask[256];
    __shared__ int s_pos[kRouteBlockTokens];
    const int E = 256, k = a.k;
    const int t0 = blockIdx.x * kRouteBlockTokens, slot = blockIdx.y;
    const int ntok = min(kRouteBlockTokens, a.T - t0);
    const int32_t* blk_base = reinterpret_cast<const int32_t*>(a.ws + a.L.blk) + (size_t)a.L.nblk * E;
    int* status = reinterpret_cast<int*>(a.ws + a.L.status);
    pdl_wait();
    pdl_launch_dependents();
    s_mask[threadIdx.x] = 0;
    // the block's per-expert counts have been read by route_scan: clear them for the next call
    if (slot == 0) reinterpret_cast<int32_t*>(a.ws + a.L.blk)[(size_t)blockIdx.x * E + threadIdx.x] = 0;
    __syncthreads();
    const int tl = threadIdx.x / 8, j = threadIdx.x % 8;   // k == 8
    int e = -1;
    if (tl < ntok) {
        e = a.topk_idx[(size_t)(t0 + tl) * k + j];
        if (e < 0 || e >= E) { if (slot == 0) set_status(status, MOE_STATUS_BAD_EXPERT); e = -1; }
        else atomicOr(&s_mask[e], 1u << tl);
    }
    __syncthreads();
    if (j == slot) {
        int p = -1;
        if (e >= 0) {
            const int rank = __popc(s_mask[e] & ((1u << tl) - 1u));
            p = blk_base[(size_t)blockIdx.x * E + e] + rank;
            const int asg = (t0 + tl) * k + j;
            a.pos[asg] = p;
            a.perm[p] = asg;
        }
        s_pos[tl] = p;
    }
    __syncthreads();
    // gather this slot's rows into expert order: xs[p] = x[t]; a warp per row, eight 16-byte
    // loads in flight per lane before the stores
    uint16_t* xs = reinterpret_cast<uint16_t*>(a.ws + a.L.xs);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < ntok; r += blockDim.x / 32) {
        const int p = s_pos[r];
        if (p < 0) continue;
        const uint16_t* src = a.x + (size_t)(t0 + r) * a.d;
        uint16_t* dst = xs + (size_t)p * a.d;
        for (int c0 = 8 * lane; c0 < a.d; c0 += 8 * 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + 256 * u < a.d) v[u] = ld_nc_v4(src + c0 + 256 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + 256 * u < a.d) *reinterpret_cast<uint4*>(dst + c0 + 256 * u) = v[u];
        }
    }
    // (the fp32 token-order sum is zero here: a fresh workspace is, and moe_combine clears it)
}

// ---------------------------------------------------------------------------------------
// route_decode: few tokens (T <= 8).  grid = 64 CTAs x 128 threads: warp (4*blockIdx + w)
// computes the logit of that expert for every token, in the same fixed order (lane = partial
// sum, shuffle tree over 16, 8, 4, 2, 1).  The last CTA to finish (atomic counter) does
// top-k and writes all routing metadata; it also clears the decode accumulators.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) route_decode(RouteArgs a) {
    __shared__ int s_last;
    __shared__ int s_e[8 * 8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * 4 + warp;
    const int d = a.d;
    float* logits = reinterpret_cast<float*>(a.ws + a.L.dec);
    int* status = reinterpret_cast<int*>(a.ws + a.L.status);
    // Before the previous kernel's results are needed: this expert's router row (d <= 2048
    // in registers) and an L2 warm-up of weights known in advance (the shared expert).
    uint4 wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < d / 256) wv[i] = ld_nc_v4(a.w_router + (size_t)e * d + 256 * i + 8 * lane);
    if (a.pf_ptr) prefetch_l2_range(a.pf_ptr, a.pf_bytes, blockIdx.x * blockDim.x + threadIdx.x,
                                    (size_t)gridDim.x * blockDim.x);
    pdl_wait();
    pdl_launch_dependents();
    for (int t = 0; t < a.T; ++t) {
        const uint16_t* xrow = a.x + (size_t)t * d;
        float p = 0.f;
        if (d <= 2048) {
            uint4 xv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < d / 256) xv[i] = ld_nc_v4(xrow + 256 * i + 8 * lane);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < d / 256) {
                    p = fmaf(bf16lo(xv[i].x), bf16lo(wv[i].x), p);
                    p = fmaf(bf16hi(xv[i].x), bf16hi(wv[i].x), p);
                    p = fmaf(bf16lo(xv[i].y), bf16lo(wv[i].y), p);
                    p = fmaf(bf16hi(xv[i].y), bf16hi(wv[i].y), p);
                    p = fmaf(bf16lo(xv[i].z), bf16lo(wv[i].z), p);
                    p = fmaf(bf16hi(xv[i].z), bf16hi(wv[i].z), p);
                    p = fmaf(bf16lo(xv[i].w), bf16lo(wv[i].w), p);
                    p = fmaf(bf16hi(xv[i].w), bf16hi(wv[i].w), p);
                }
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) p = p + __shfl_xor_sync(0xffffffffu, p, m);
            if (a.bias) p = p + a.bias[e];
        } else {
            p = warp_pinned_logit(xrow, a.w_router + (size_t)e * d, d, lane, a.bias ? a.bias + e : nullptr);
        }
        if (lane == 0) logits[(size_t)t * 256 + e] = p;
    }
    __threadfence();
    __syncthreads();
    unsigned int* counter = reinterpret_cast<unsigned int*>(status + 1);
    if (threadIdx.x == 0) s_last = (atomicAdd(counter, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // top-k per token (warp t handles tokens t, t+4, ...)
    __shared__ float s_lg[4][256];
    for (int t = warp; t < a.T; t += 4) {
        int ee;
        float ww;
        // read through L2: written by other CTAs
        for (int s = 0; s < 8; ++s) s_lg[warp][lane + 32 * s] = __ldcg(logits + (size_t)t * 256 + lane + 32 * s);
        __syncwarp();
        warp_topk256(s_lg[warp], a.k, lane, ee, ww);
        if (lane < a.k) {
            a.topk_idx[(size_t)t * a.k + lane] = ee;
            a.topk_w[(size_t)t * a.k + lane] = ww;
            s_e[t * 8 + lane] = ee;
        }
        __syncwarp();
    }
    __syncthreads();
    // metadata for the n = T*k assignments, in parallel: expert e's group starts after every
    // assignment to a lower expert; rows of a group are in assignment (= token) order.
    __shared__ int s_cnt[256], s_tstart[256];
    const int n = a.T * a.k;
    for (int ex = threadIdx.x; ex < 256; ex += blockDim.x) {
        int off = 0, cnt = 0;
        for (int q = 0; q < n; ++q) { off += s_e[q] < ex; cnt += s_e[q] == ex; }
        a.offsets[ex] = off;
        a.counts[ex] = cnt;
        s_cnt[ex] = cnt;
    }
    if (threadIdx.x == 0) a.offsets[256] = n;
    __syncthreads();
    // block map: tiles of expert ex start after the tiles of lower experts
    if (threadIdx.x < 32) {
        int run = 0;
        for (int base = 0; base < 256; base += 32) {
            const int ex = base + threadIdx.x;
            const int nt = (s_cnt[ex] + a.tile_rows - 1) / a.tile_rows;
            int incl = nt;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, m);
                if ((int)threadIdx.x >= m) incl += y;
            }
            s_tstart[ex] = run + incl - nt;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (threadIdx.x == 0) *a.num_tiles = run;
    }
    __syncthreads();
    for (int ex = threadIdx.x; ex < 256; ex += blockDim.x) {
        int off = 0;
        for (int q = 0; q < n; ++q) off += s_e[q] < ex;
        for (int r = 0, i = 0; r < s_cnt[ex]; r += a.tile_rows, ++i) {
            int32_t* tt = a.tiles + 3 * (size_t)(s_tstart[ex] + i);
            tt[0] = ex; tt[1] = off + r; tt[2] = min(a.tile_rows, s_cnt[ex] - r);
        }
    }
    if (threadIdx.x < n) {
        const int q = threadIdx.x, ex = s_e[q];
        int p = 0;
        for (int q2 = 0; q2 < n; ++q2) p += (s_e[q2] < ex) || (s_e[q2] == ex && q2 < q);
        a.pos[q] = p;
        a.perm[p] = q;
    }
    if (threadIdx.x == 0) *counter = 0;
    // clear the decode accumulators (g/u per token and slot) and the token-order sum
    float* gu = logits + kDecodeMaxT * 256;
    for (int i = threadIdx.x; i < a.T * (a.k + 1) * 2 * a.I; i += blockDim.x) gu[i] = 0.f;
    float* acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    for (int i = threadIdx.x; i < a.T * d; i += blockDim.x) acc[i] = 0.f;
}

}  // namespace

// route_certify_topk instantiated for the token row in registers (d = 256, 512, 1024, 2048) or
// read from memory (other d)
static cudaError_t launch_certify(const RouteArgs& a, int KS, cudaStream_t st) {
    const dim3 grid((a.T + kCertTokens - 1) / kCertTokens), block(32 * kCertTokens);
    switch (a.d / 256) {
        case 1: return launch_with_pdl(route_certify_topk<1>, grid, block, 0, st, a, KS);
        case 2: return launch_with_pdl(route_certify_topk<2>, grid, block, 0, st, a, KS);
        case 4: return launch_with_pdl(route_certify_topk<4>, grid, block, 0, st, a, KS);
        case 8: return launch_with_pdl(route_certify_topk<8>, grid, block, 0, st, a, KS);
        default: return launch_with_pdl(route_certify_topk<0>, grid, block, 0, st, a, KS);
    }
}

cudaError_t launch_route_prefill(const RouteArgs& a, cudaStream_t st, unsigned long long* launches) {
    static bool attr = false;
    if (!attr) {
        cudaError_t err = cudaFuncSetAttribute(router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
        if (err != cudaSuccess) return err;
        attr = true;
    }
    const int nblk = a.L.nblk;
    const int KS = router_kslices(a.T, a.d);
    CUtensorMap tm_x, tm_w;
    cudaError_t err = make_tmap_bf16_2d(&tm_x, a.x, a.T, a.d, (uint64_t)a.d * 2, kBK, 128);
    if (err != cudaSuccess) return err;
    err = make_tmap_bf16_2d(&tm_w, a.w_router, 256, a.d, (uint64_t)a.d * 2, kBK, 256);
    if (err != cudaSuccess) return err;
    *launches += 5;
    if ((err = launch_with_pdl(router_wnorm, dim3(256 / 4), dim3(128), 0, st, a)) != cudaSuccess) return err;
    if ((err = launch_with_pdl(router_tc, dim3((a.T + 127) / 128, KS), dim3(192), kRtSmem, st, tm_x, tm_w, a, KS)) !=
        cudaSuccess)
        return err;
    if ((err = launch_certify(a, KS, st)) != cudaSuccess) return err;
    if ((err = launch_with_pdl(route_scan, dim3(kScanCtas), dim3(1024), 0, st, a)) != cudaSuccess) return err;
    return launch_with_pdl(route_scatter, dim3(nblk, a.k), dim3(256), 0, st, a);
}

namespace {
// ---------------------------------------------------------------------------------------
// router_logits_exact: every logit of every token with the exact recomputation's device code
// (pinned_logit_group, kCertGroup experts per round; NI = d / 256 as in route_certify_topk);
// one warp per (token, 32 experts).
// ---------------------------------------------------------------------------------------
template <int NI>
__global__ void __launch_bounds__(256) router_logits_exact(const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ w_router,
                                                           const float* __restrict__ bias, float* __restrict__ out,
                                                           int T, int d) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);   // (token, expert group of 32)
    const int t = gw >> 3, e0 = (gw & 7) * 32;
    if (t >= T) return;
    const uint16_t* xrow = x + (size_t)t * d;
    uint4 xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        xv[i] = make_uint4(0, 0, 0, 0);
        if (i < d / 256) xv[i] = ld_nc_v4(xrow + 256 * i + 8 * lane);
    }
    for (int g0 = 0; g0 < 32; g0 += kCertGroup) {
        int eg[kCertGroup];
#pragma unroll
        for (int g = 0; g < kCertGroup; ++g) eg[g] = e0 + g0 + g;
        float lg[kCertGroup];
        pinned_logit_group<NI, kCertGroup>(xv, xrow, w_router, d, eg, lane, lg);
#pragma unroll
        for (int g = 0; g < kCertGroup; ++g)
            if (lane == g0 + g) out[(size_t)t * 256 + eg[g]] = bias ? lg[g] + bias[eg[g]] : lg[g];
    }
}
}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_router, const float* bias, float* out, int T,
                                 int d, cudaStream_t st, unsigned long long* launches) {
    *launches += 1;
    const dim3 grid((unsigned)T), block(256);
    switch (d / 256) {
        case 1: return launch_with_pdl(router_logits_exact<1>, grid, block, 0, st, x, w_router, bias, out, T, d);
        case 2: return launch_with_pdl(router_logits_exact<2>, grid, block, 0, st, x, w_router, bias, out, T, d);
        case 4: return launch_with_pdl(router_logits_exact<4>, grid, block, 0, st, x, w_router, bias, out, T, d);
        case 8: return launch_with_pdl(router_logits_exact<8>, grid, block, 0, st, x, w_router, bias, out, T, d);
        default: return launch_with_pdl(router_logits_exact<0>, grid, block, 0, st, x, w_router, bias, out, T, d);
    }
}

// ---------------------------------------------------------------------------------------
// Host-round-trip routing (the ablation of "GPU-resident routing"): the same kernels up to
// the per-block counts; then the counts go to the host, the host computes what route_scan
// computes (counts, offsets, per-block bases, exported block map, GEMM tile lists), copies it
// back and the scatter runs.  One stream synchronisation per call.  Results are identical to
// launch_route_prefill's.
// ---------------------------------------------------------------------------------------
namespace {
struct HostScan {
    std::vector<int32_t> counts, offsets, base, tiles, gu, dn;
    int32_t num_tiles = 0, gu_num = 0, dn_num = 0;
};

// nb near-equal blocks of `rows` rows from r0, each repeated for the mt weight tiles (weight
// tile innermost); entry j = (first + i) * mt + m of its sequence goes to list position
// j + (j >= from ? by : 0), as route_scan places them
void host_split(std::vector<int32_t>& list, int mt, int first, int ex, int r0, int rows, int nb, int from, int by) {
    const int q = rows / nb, rem = rows % nb;
    for (int i = 0; i < nb; ++i) {
        const int n = q + (i < rem ? 1 : 0);
        for (int m = 0; m < mt; ++m) {
            const int j = (first + i) * mt + m;
            int32_t* t = &list[4 * (size_t)(j >= from ? j + by : j)];
            t[0] = ex; t[1] = r0; t[2] = n; t[3] = m;
        }
        r0 += n;
    }
}

HostScan host_scan(const RouteArgs& a, const std::vector<int32_t>& blk) {
    const int E = 256, nb = a.L.nblk, BM = a.tile_rows;
    HostScan h;
    h.counts.assign(E, 0);
    h.offsets.assign(E + 1, 0);
    h.base.assign((size_t)nb * E, 0);
    for (int b = 0; b < nb; ++b)
        for (int e = 0; e < E; ++e) h.counts[e] += blk[(size_t)b * E + e];
    for (int e = 0; e < E; ++e) h.offsets[e + 1] = h.offsets[e] + h.counts[e];
    for (int e = 0; e < E; ++e) {
        int r = h.offsets[e];
        for (int b = 0; b < nb; ++b) {
            h.base[(size_t)b * E + e] = r;
            r += blk[(size_t)b * E + e];
        }
    }
    for (int e = 0; e < E; ++e)
        for (int i = 0; i * BM < h.counts[e]; ++i) {
            h.tiles.push_back(e);
            h.tiles.push_back(h.offsets[e] + i * BM);
            h.tiles.push_back(std::min(BM, h.counts[e] - i * BM));
        }
    h.num_tiles = (int32_t)(h.tiles.size() / 3);
    const int MTgu = a.I / kTileRows, MTdn = a.d / 256;
    const int nsh = (a.T + a.gu_rows - 1) / a.gu_rows, nshd = (a.T + a.dn_rows - 1) / a.dn_rows;
    int ngu = nsh, ndn = nshd;
    for (int e = 0; e < E; ++e) {
        ngu += (h.counts[e] + a.gu_rows - 1) / a.gu_rows;
        ndn += (h.counts[e] + a.dn_rows - 1) / a.dn_rows;
    }
    h.gu.assign(4 * (size_t)ngu * MTgu, 0);
    h.dn.assign(4 * (size_t)ndn * MTdn, 0);
    const int shg = nsh * MTgu, shd = nshd * MTdn;
    const int pg = shared_tiles_at(ngu * MTgu, shg, a.num_sms), pd = shared_tiles_at(ndn * MTdn, shd, a.num_sms);
    for (int i = 0; i < nsh; ++i) {
        const int q = a.T / nsh, rem = a.T % nsh;
        host_split(h.gu, MTgu, i, E, i * q + std::min(i, rem), q + (i < rem ? 1 : 0), 1, 0, pg);
    }
    for (int i = 0; i < nshd; ++i) {
        const int q = a.T / nshd, rem = a.T % nshd;
        host_split(h.dn, MTdn, i, E, i * q + std::min(i, rem), q + (i < rem ? 1 : 0), 1, 0, pd);
    }
    int gb = 0, db = 0;
    for (int e = 0; e < E; ++e) {
        const int run = h.counts[e], nn = (run + a.gu_rows - 1) / a.gu_rows, nd = (run + a.dn_rows - 1) / a.dn_rows;
        if (nn > 0) host_split(h.gu, MTgu, gb, e, h.offsets[e], run, nn, pg, shg);
        if (nd > 0) host_split(h.dn, MTdn, db, e, h.offsets[e], run, nd, pd, shd);
        gb += nn;
        db += nd;
    }
    h.gu_num = ngu * MTgu;
    h.dn_num = ndn * MTdn;
    return h;
}
}  // namespace

cudaError_t launch_route_prefill_host(const RouteArgs& a, cudaStream_t st, unsigned long long* launches) {
    static bool attr = false;
    if (!attr) {
        cudaError_t err = cudaFuncSetAttribute(router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
        if (err != cudaSuccess) return err;
        attr = true;
    }
    const int nblk = a.L.nblk, E = 256;
    const int KS = router_kslices(a.T, a.d);
    CUtensorMap tm_x, tm_w;
    cudaError_t err = make_tmap_bf16_2d(&tm_x, a.x, a.T, a.d, (uint64_t)a.d * 2, kBK, 128);
    if (err != cudaSuccess) return err;
    err = make_tmap_bf16_2d(&tm_w, a.w_router, 256, a.d, (uint64_t)a.d * 2, kBK, 256);
    if (err != cudaSuccess) return err;
    *launches += 4;
    if ((err = launch_with_pdl(router_wnorm, dim3(256 / 4), dim3(128), 0, st, a)) != cudaSuccess) return err;
    if ((err = launch_with_pdl(router_tc, dim3((a.T + 127) / 128, KS), dim3(192), kRtSmem, st, tm_x, tm_w, a, KS)) !=
        cudaSuccess)
        return err;
    if ((err = launch_certify(a, KS, st)) != cudaSuccess) return err;
    // the round trip: per-block counts to the host, scan and block map there, results back
    int32_t* blk_dev = reinterpret_cast<int32_t*>(a.ws + a.L.blk);
    std::vector<int32_t> blk((size_t)nblk * E);
    if ((err = cudaMemcpyAsync(blk.data(), blk_dev, blk.size() * 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (err = cudaStreamSynchronize(st)) != cudaSuccess)
        return err;
    const HostScan h = host_scan(a, blk);
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        return bytes ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st) : cudaSuccess;
    };
    if ((err = cudaMemsetAsync(blk_dev, 0, blk.size() * 4, st)) != cudaSuccess ||   // the next call adds into zeros
        (err = h2d(blk_dev + (size_t)nblk * E, h.base.data(), h.base.size() * 4)) != cudaSuccess ||
        (err = h2d(a.counts, h.counts.data(), E * 4)) != cudaSuccess ||
        (err = h2d(a.offsets, h.offsets.data(), (E + 1) * 4)) != cudaSuccess ||
        (err = h2d(a.tiles, h.tiles.data(), h.tiles.size() * 4)) != cudaSuccess ||
        (err = h2d(a.num_tiles, &h.num_tiles, 4)) != cudaSuccess ||
        (err = h2d(a.ws + a.L.gu_tiles, h.gu.data(), h.gu.size() * 4)) != cudaSuccess ||
        (err = h2d(a.ws + a.L.gu_num, &h.gu_num, 4)) != cudaSuccess ||
        (err = h2d(a.ws + a.L.dn_tiles, h.dn.data(), h.dn.size() * 4)) != cudaSuccess ||
        (err = h2d(a.ws + a.L.dn_num, &h.dn_num, 4)) != cudaSuccess)
        return err;
    // pageable sources: every copy above has consumed its source when it returns
    *launches += 1;
    return launch_with_pdl(route_scatter, dim3(nblk, a.k), dim3(256), 0, st, a);
}

cudaError_t launch_route_decode(const RouteArgs& a, cudaStream_t st, unsigned long long* launches) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(64);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, route_decode, a);
    *launches += 1;
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace moe
