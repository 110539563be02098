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
// Prefill (four launches):
//   route_logits       CTA per (32-token block, 16 experts): router logits in the fixed
//                      fp32 order.
//   route_topk         one CTA per block: top-8 + weights, the block's per-expert counts.
//   route_scan         one CTA: per-block bases, counts, offsets, the exported block map
//                      and the GEMM tile lists (expert, first row, rows, 128-row M tile).
//   route_scatter      one CTA per (block, slot): stable group positions (rank of the token among
//                      the block's tokens routed to the same expert, from a bitmask), perm /
//                      pos, the gathered rows xs, and zeroing of the fp32 token-order sum.
// Decode (one launch): route_decode -- a warp per expert logit, the last CTA to finish
// does top-8 and the metadata for the few tokens.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;   // 8 warps; warp w owns tokens 4w..4w+3 of the block
constexpr int kExpPerPass = 16;

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

// ---------------------------------------------------------------------------------------
// route_logits: grid = (ceil(T/32) token blocks, 256/16 expert groups), 256 threads.
// Lane l of every warp is partial sum l of the fixed order: it takes columns
// k = 256*i + 8*l + j for i ascending, j = 0..7, with fmaf starting from 0.  Warp w holds
// tokens 4w..4w+3 of the block x the CTA's 16 experts (64 accumulators per lane); the 32
// partial sums of each logit are then added by a recursive-halving exchange over lane
// distances 16, 8, 4, 2, 1 -- the same pairing, hence the same value, as the tree
// s[i] += s[i+m].  Logits (+ bias) go to the workspace, [T][256] fp32.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouteThreads) route_logits(RouteArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * kRouteBlockTokens;
    const int e0 = blockIdx.y * kExpPerPass;
    const int d = a.d;
    const int nI = d / 256;
    float* logits = reinterpret_cast<float*>(a.ws + a.L.logits);

    float acc[4][kExpPerPass];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int e = 0; e < kExpPerPass; ++e) acc[t][e] = 0.f;
    for (int i = 0; i < nI; ++i) {
        const int col = 256 * i + 8 * lane;
        float xf[4][8];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int tok = t0 + 4 * warp + t;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tok < a.T) v = ld_nc_v4(a.x + (size_t)tok * d + col);
            xf[t][0] = bf16lo(v.x); xf[t][1] = bf16hi(v.x); xf[t][2] = bf16lo(v.y); xf[t][3] = bf16hi(v.y);
            xf[t][4] = bf16lo(v.z); xf[t][5] = bf16hi(v.z); xf[t][6] = bf16lo(v.w); xf[t][7] = bf16hi(v.w);
        }
#pragma unroll
        for (int e = 0; e < kExpPerPass; ++e) {
            uint4 v = ld_nc_v4(a.w_router + (size_t)(e0 + e) * d + col);
            float wf[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                           bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int t = 0; t < 4; ++t) acc[t][e] = fmaf(xf[t][j], wf[j], acc[t][e]);
        }
    }
    // recursive halving over 64 values (index o = 16*t + e); lane l ends with o = 2l, 2l+1
    float v[64];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int e = 0; e < kExpPerPass; ++e) v[16 * t + e] = acc[t][e];
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int m = 16 >> step;
        const int c = 64 >> step;        // live values before this step
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int q = 0; q < c / 2; ++q) {
            const float lo = v[q], hi = v[q + c / 2];
            const float send = upper ? lo : hi;
            const float keep = upper ? hi : lo;
            v[q] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int o = 2 * lane + r;
        const int t = o >> 4, e = e0 + (o & 15);
        const int tok = t0 + 4 * warp + t;
        float lg = v[r];
        if (a.bias) lg = lg + a.bias[e];
        if (tok < a.T) logits[(size_t)tok * 256 + e] = lg;
    }
}

// ---------------------------------------------------------------------------------------
// route_topk: grid = ceil(T/32) blocks, 256 threads: top-8 + weights per token (warp w does
// tokens 4w..4w+3) and the block's per-expert counts.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouteThreads) route_topk(RouteArgs a) {
    __shared__ uint32_t s_mask[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * kRouteBlockTokens;
    const float* logits = reinterpret_cast<const float*>(a.ws + a.L.logits);
    s_mask[threadIdx.x] = 0;
    __syncthreads();
    for (int t = 0; t < 4; ++t) {
        const int tl = 4 * warp + t, tok = t0 + tl;
        if (tok >= a.T) break;
        int e;
        float w;
        warp_topk256(logits + (size_t)tok * 256, a.k, lane, e, w);
        if (lane < a.k) {
            a.topk_idx[(size_t)tok * a.k + lane] = e;
            a.topk_w[(size_t)tok * a.k + lane] = w;
            atomicOr(&s_mask[e], 1u << tl);
        }
    }
    __syncthreads();
    int32_t* blk_counts = reinterpret_cast<int32_t*>(a.ws + a.L.blk);
    blk_counts[(size_t)blockIdx.x * 256 + threadIdx.x] = __popc(s_mask[threadIdx.x]);
}

// ---------------------------------------------------------------------------------------
// route_scan: one CTA of 256 threads (thread e = expert e).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_tmp) {
    // 256 threads; s_tmp has 8 ints
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, m);
        if (lane >= m) x += y;
    }
    __syncthreads();
    if (lane == 31) s_tmp[warp] = x;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_tmp[w];
    return base + x - v;
}

__global__ void __launch_bounds__(256) route_scan(RouteArgs a) {
    __shared__ int s_tmp[8];
    __shared__ int s_tot[4];
    const int e = threadIdx.x;
    const int E = 256;
    int32_t* blk_counts = reinterpret_cast<int32_t*>(a.ws + a.L.blk);
    int32_t* blk_base = blk_counts + (size_t)a.L.nblk * E;
    int run = 0;
    for (int b = 0; b < a.L.nblk; ++b) {
        const int c = blk_counts[(size_t)b * E + e];
        blk_base[(size_t)b * E + e] = run;
        run += c;
    }
    a.counts[e] = run;
    const int off = block_exclusive_scan(run, s_tmp);
    a.offsets[e] = off;
    if (e == E - 1) a.offsets[E] = off + run;
    for (int b = 0; b < a.L.nblk; ++b) blk_base[(size_t)b * E + e] += off;

    // exported block map: ceil(count / tile_rows) tiles per expert, expert-ascending
    const int BM = a.tile_rows;
    const int nt = (run + BM - 1) / BM;
    const int tbase = block_exclusive_scan(nt, s_tmp);
    for (int i = 0; i < nt; ++i) {
        int32_t* tt = a.tiles + 3 * (size_t)(tbase + i);
        tt[0] = e;
        tt[1] = off + i * BM;
        tt[2] = min(BM, run - i * BM);
    }
    if (e == E - 1) s_tot[0] = tbase + nt;

    // GEMM tile lists: an expert's rows split into ceil(rows / kMaxN) near-equal token blocks;
    // each block is repeated for every weight tile (weight tile innermost, so the CTAs that
    // run at the same time share the block's activation rows in L2).  The shared expert
    // (expert index E) comes first and covers token rows 0..T-1.
    const int MTgu = a.I / kTileRows, MTdn = a.d / 256;   // 128 gate+up row pairs; 256-row down tiles
    const int nn = (run + kMaxN - 1) / kMaxN;
    const int nsh = (a.T + kMaxN - 1) / kMaxN;
    const int nbase = block_exclusive_scan(nn, s_tmp);
    if (e == E - 1) s_tot[1] = nbase + nn;
    __syncthreads();
    int4* gu = reinterpret_cast<int4*>(a.ws + a.L.gu_tiles);
    int4* dn = reinterpret_cast<int4*>(a.ws + a.L.dn_tiles);
    auto emit = [&](int slot, int ex, int r0, int rows) {
        for (int m = 0; m < MTgu; ++m) gu[(size_t)slot * MTgu + m] = make_int4(ex, r0, rows, m);
        for (int m = 0; m < MTdn; ++m) dn[(size_t)slot * MTdn + m] = make_int4(ex, r0, rows, m);
    };
    if (nn > 0) {
        const int base_rows = run / nn, rem = run % nn;
        int r0 = off;
        for (int i = 0; i < nn; ++i) {
            const int rows = base_rows + (i < rem ? 1 : 0);
            emit(nsh + nbase + i, e, r0, rows);
            r0 += rows;
        }
    }
    for (int i = e; i < nsh; i += E) {   // shared expert N tiles
        const int base_rows = a.T / nsh, rem = a.T % nsh;
        const int r0 = i * base_rows + min(i, rem);
        emit(i, E, r0, base_rows + (i < rem ? 1 : 0));
    }
    __syncthreads();
    if (e == 0) {
        *a.num_tiles = s_tot[0];
        const int total_n = nsh + s_tot[1];
        *reinterpret_cast<int32_t*>(a.ws + a.L.gu_num) = total_n * MTgu;
        *reinterpret_cast<int32_t*>(a.ws + a.L.dn_num) = total_n * MTdn;
    }
}

// ---------------------------------------------------------------------------------------
// route_scatter: grid = (ceil(T/32) blocks, k slots), 256 threads.  Every CTA rebuilds the
// block's expert bitmasks (bit t set when token t of the block picked the expert), which
// give the stable rank of a token among the block's tokens routed to the same expert; CTA
// (b, j) then writes pos / perm of slot j, copies those 32 rows into expert order
// (xs[p] = x[t]) and clears 1/k of the block's rows of the fp32 token-order sum.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) route_scatter(RouteArgs a) {
    __shared__ uint32_t s_mask[256];
    __shared__ int s_pos[kRouteBlockTokens];
    const int E = 256, k = a.k;
    const int t0 = blockIdx.x * kRouteBlockTokens, slot = blockIdx.y;
    const int ntok = min(kRouteBlockTokens, a.T - t0);
    const int32_t* blk_base = reinterpret_cast<const int32_t*>(a.ws + a.L.blk) + (size_t)a.L.nblk * E;
    int* status = reinterpret_cast<int*>(a.ws + a.L.status);
    s_mask[threadIdx.x] = 0;
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
    // gather this slot's rows into expert order: xs[p] = x[t]
    uint16_t* xs = reinterpret_cast<uint16_t*>(a.ws + a.L.xs);
    const int cpr = a.d / 8;                       // 16-byte chunks per row
    const int total = ntok * cpr;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int r = idx / cpr, c = idx % cpr;
        const int p = s_pos[r];
        if (p < 0) continue;
        const uint4 v = ld_nc_v4(a.x + (size_t)(t0 + r) * a.d + 8 * c);
        *reinterpret_cast<uint4*>(xs + (size_t)p * a.d + 8 * c) = v;
    }
    // clear this CTA's share of the fp32 token-order sum of the block
    float4* acc = reinterpret_cast<float4*>(a.ws + a.L.acc) + (size_t)t0 * (a.d / 4);
    const int n4 = ntok * (a.d / 4);
    for (int idx = slot * blockDim.x + threadIdx.x; idx < n4; idx += k * blockDim.x)
        acc[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
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
    for (int t = 0; t < a.T; ++t) {
        float p = 0.f;
        for (int i = 0; i < d / 256; ++i) {
            const int col = 256 * i + 8 * lane;
            const uint4 xv = ld_nc_v4(a.x + (size_t)t * d + col);
            const uint4 wv = ld_nc_v4(a.w_router + (size_t)e * d + col);
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
        if (a.bias) p = p + a.bias[e];
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
    // metadata for T*k assignments (stable: token-ascending within an expert)
    if (threadIdx.x == 0) {
        const int n = a.T * a.k;
        // offsets: exclusive scan over experts of the counts
        int cnt[256];
        for (int ex = 0; ex < 256; ++ex) cnt[ex] = 0;
        for (int q = 0; q < n; ++q) cnt[s_e[q]]++;
        int run = 0, nt = 0;
        int start[256];
        for (int ex = 0; ex < 256; ++ex) {
            start[ex] = run;
            a.offsets[ex] = run;
            a.counts[ex] = cnt[ex];
            for (int r = 0; r < cnt[ex]; r += a.tile_rows) {
                int32_t* tt = a.tiles + 3 * (size_t)nt++;
                tt[0] = ex; tt[1] = run + r; tt[2] = min(a.tile_rows, cnt[ex] - r);
            }
            run += cnt[ex];
        }
        a.offsets[256] = run;
        *a.num_tiles = nt;
        for (int q = 0; q < n; ++q) {       // q = t*k + j ascending: token-ascending per expert
            const int p = start[s_e[q]]++;
            a.pos[q] = p;
            a.perm[p] = q;
        }
        *counter = 0;
    }
    // clear the decode accumulators (g/u per token and slot) and the token-order sum
    float* gu = logits + kDecodeMaxT * 256;
    for (int i = threadIdx.x; i < a.T * (a.k + 1) * 2 * a.I; i += blockDim.x) gu[i] = 0.f;
    float* acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    for (int i = threadIdx.x; i < a.T * d; i += blockDim.x) acc[i] = 0.f;
}

}  // namespace

cudaError_t launch_route_prefill(const RouteArgs& a, cudaStream_t st, unsigned long long* launches) {
    const int nblk = a.L.nblk;
    route_logits<<<dim3(nblk, 256 / kExpPerPass), kRouteThreads, 0, st>>>(a);
    route_topk<<<nblk, kRouteThreads, 0, st>>>(a);
    route_scan<<<1, 256, 0, st>>>(a);
    route_scatter<<<dim3(nblk, a.k), 256, 0, st>>>(a);
    *launches += 4;
    return cudaGetLastError();
}

cudaError_t launch_route_decode(const RouteArgs& a, cudaStream_t st, unsigned long long* launches) {
    route_decode<<<64, 128, 0, st>>>(a);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
