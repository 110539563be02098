// decode.cu -- batch-1 decode: HBM-bound GEMV kernels over the packed 4-bit weights.
//
// "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026): section "Optimize the
// single-row weight path" (row-parallel GEMV: threads cooperate on outputs while reading
// different parts of the weight matrix) and section "Reduce intermediate and state traffic"
// (fused chains: the two expert input projections with their gated activation; the output
// projection with its routing score and the shared-expert result).
//
// One token, 8 routed experts + the shared expert ("slots" 0..8):
//   decode_gate_up  grid (9 slots x I/128 row tiles x K/256 column groups): each thread owns
//                   one gate or up row of a packed chunk and dots 4 K blocks (256 columns) of
//                   it with x; partial sums go to the fp32 g/u accumulators with atomics.
//   decode_down     grid (9 slots x d/128 row tiles): h = silu(g) * u in fp32 (no rounding),
//                   each thread dots half of one down row with h; the result times the routing
//                   weight (1 for the shared expert) is added into the fp32 sum.  When y is
//                   given, the last CTA of a row tile writes those 128 outputs as bf16.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kKbPerCta = 4;

// 16 B of packed codes (32 weights, columns 0..31 of a half chunk) dequantised and dotted
// with 32 fp32 activations.
template <bool kDenorm>
__device__ __forceinline__ float dot32(uint4 codes, uint32_t s2, uint32_t b2, const float* xv, float acc) {
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t wv[4];
        dequant_word<kDenorm>(words[q], s2, b2, wv);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = 8 * q + 2 * u;
            acc = fmaf(bf16lo(wv[u]), xv[c], acc);
            acc = fmaf(bf16hi(wv[u]), xv[c + 1], acc);
        }
    }
    return acc;
}

__device__ __forceinline__ float dot32m(bool denorm, uint4 codes, uint32_t s2, uint32_t b2, const float* xv, float acc) {
    return denorm ? dot32<true>(codes, s2, b2, xv, acc) : dot32<false>(codes, s2, b2, xv, acc);
}

struct DecParams {
    const uint16_t* x;
    const int32_t* topk_idx;
    const float* topk_w;
    const uint8_t* w_gu_routed;
    const uint8_t* w_gu_shared;
    const uint8_t* w_dn_routed;
    const uint8_t* w_dn_shared;
    const int* mode_routed;    // scale encoding of each packed buffer
    const int* mode_shared;
    float* gu;          // [9][2][I]
    float* acc;         // [d]
    uint16_t* y;        // [d] or null
    unsigned int* tile_counters;   // [d/128]
    int* status;
    int d, I, E, k;
};

__global__ void __launch_bounds__(256) decode_gate_up(DecParams p) {
    __shared__ float xs[kKbPerCta * kBK];
    const int MT = p.I / kTileRows, KB = p.d / kBK, NKC = KB / kKbPerCta;
    const int s = blockIdx.x / (MT * NKC);
    const int mt = (blockIdx.x / NKC) % MT;
    const int kc = blockIdx.x % NKC;
    const int mat = threadIdx.x >> 7, r = threadIdx.x & 127;
    uint4 c[kKbPerCta][2];
    uint32_t sb[kKbPerCta][2];
    auto issue_loads = [&](const uint8_t* base) {
#pragma unroll
        for (int q = 0; q < kKbPerCta; ++q) {
            const uint8_t* ch = base + (size_t)(kc * kKbPerCta + q) * kChunkPairBytes + mat * kChunkBytes;
            c[q][0] = ld_nc_v4(ch + r * 16);
            c[q][1] = ld_nc_v4(ch + 2048 + r * 16);
            sb[q][0] = __ldg(reinterpret_cast<const uint16_t*>(ch + kChunkCodes) + r);
            sb[q][1] = __ldg(reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 256) + r);
        }
    };
    int e = p.E;
    if (s == p.k) {
        // the shared expert's weights do not depend on routing: load them before waiting
        issue_loads(p.w_gu_shared + (size_t)mt * KB * kChunkPairBytes);
        pdl_wait();
        pdl_launch_dependents();
    } else {
        pdl_wait();
        pdl_launch_dependents();
        e = p.topk_idx[s];
        if (e < 0 || e >= p.E) { if (threadIdx.x == 0) set_status(p.status, MOE_STATUS_BAD_EXPERT); return; }
        issue_loads(p.w_gu_routed + (size_t)(e * MT + mt) * KB * kChunkPairBytes);
        // warm L2 with this expert's down weights for the next kernel (a slice per CTA)
        const size_t dn_bytes = (size_t)(p.d / 256) * (p.I / kBK) * kChunkPairBytes;
        const int part = mt * NKC + kc, nparts = MT * NKC;
        const size_t lo = dn_bytes * part / nparts, hi = dn_bytes * (part + 1) / nparts;
        prefetch_l2_range(p.w_dn_routed + (size_t)e * dn_bytes + lo, hi - lo, threadIdx.x, blockDim.x);
    }
    const bool denorm = *(s < p.k ? p.mode_routed : p.mode_shared) == kScaleDenorm;
    xs[threadIdx.x] = bf16f(p.x[kc * kKbPerCta * kBK + threadIdx.x]);
    __syncthreads();
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kKbPerCta; ++q) {
        const uint32_t s2 = sb[q][0] * 0x10001u, b2 = sb[q][1] * 0x10001u;
        acc = dot32m(denorm, c[q][0], s2, b2, xs + q * kBK, acc);
        acc = dot32m(denorm, c[q][1], s2, b2, xs + q * kBK + 32, acc);
    }
    atomicAdd(p.gu + ((size_t)s * 2 + mat) * p.I + mt * kTileRows + r, acc);
}

__global__ void __launch_bounds__(256) decode_down(DecParams p) {
    extern __shared__ float hsm[];   // [I]
    __shared__ float part[kTileRows];
    __shared__ int s_last;
    const int MT = p.d / kTileRows, KB = p.I / kBK;
    const int s = blockIdx.x / MT, mt = blockIdx.x % MT;
    pdl_wait();
    pdl_launch_dependents();
    int e = p.E;
    float wgt = 1.0f;
    if (s < p.k) {
        e = p.topk_idx[s];
        wgt = p.topk_w[s];
        if (e < 0 || e >= p.E) e = -1;
    }
    const uint8_t* base = nullptr;
    // down stacks pair the two 128-row halves of each 256-row tile: chunk (mt, kb) sits at
    // ((mt / 2) * KB + kb) * 9216 + (mt % 2) * 4608
    if (e >= 0)
        base = (s < p.k ? p.w_dn_routed + (size_t)(e * (MT / 2)) * KB * kChunkPairBytes : p.w_dn_shared) +
               (size_t)(mt / 2) * KB * kChunkPairBytes + (mt % 2) * kChunkBytes;
    const int hf = threadIdx.x >> 7, r = threadIdx.x & 127;
    const int kb0 = hf * (KB / 2), nkb = KB / 2;
    const bool denorm = *(s < p.k ? p.mode_routed : p.mode_shared) == kScaleDenorm;
    float acc = 0.f;
    if (base) {
        // h = silu(g) * u for this slot
        const float* g = p.gu + (size_t)s * 2 * p.I;
        for (int i = threadIdx.x; i < p.I; i += blockDim.x) {
            const float gv = __ldcg(g + i), uv = __ldcg(g + p.I + i);
            hsm[i] = gv / (1.0f + __expf(-gv)) * uv;
        }
        __syncthreads();
        for (int q = 0; q < nkb; q += 4) {
            uint4 c[4][2];
            uint32_t sb[4][2];
            const int nq = min(4, nkb - q);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (u < nq) {
                    const uint8_t* ch = base + (size_t)(kb0 + q + u) * kChunkPairBytes;
                    c[u][0] = ld_nc_v4(ch + r * 16);
                    c[u][1] = ld_nc_v4(ch + 2048 + r * 16);
                    sb[u][0] = __ldg(reinterpret_cast<const uint16_t*>(ch + kChunkCodes) + r);
                    sb[u][1] = __ldg(reinterpret_cast<const uint16_t*>(ch + kChunkCodes + 256) + r);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (u < nq) {
                    const int kb = kb0 + q + u;
                    const uint32_t s2 = sb[u][0] * 0x10001u, b2 = sb[u][1] * 0x10001u;
                    acc = dot32m(denorm, c[u][0], s2, b2, hsm + kb * kBK, acc);
                    acc = dot32m(denorm, c[u][1], s2, b2, hsm + kb * kBK + 32, acc);
                }
            }
        }
    } else {
        __syncthreads();
        if (threadIdx.x == 0) set_status(p.status, MOE_STATUS_BAD_EXPERT);
    }
    if (hf == 1) part[r] = acc;
    __syncthreads();
    if (hf == 0 && base) atomicAdd(p.acc + mt * kTileRows + r, wgt * (acc + part[r]));
    if (p.y == nullptr) return;
    // last CTA of this row tile writes the 128 outputs
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(p.tile_counters + mt, 1u) == (unsigned)(p.k + 1) - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < kTileRows) {
        const float v = __ldcg(p.acc + mt * kTileRows + threadIdx.x);
        p.y[mt * kTileRows + threadIdx.x] = f32_to_bf16_rn(v);
        p.acc[mt * kTileRows + threadIdx.x] = 0.f;   // leave the sum at zero
    }
    if (threadIdx.x == 0) p.tile_counters[mt] = 0;
}

DecParams make_dec_params(const FfnArgs& a, uint16_t* y) {
    DecParams p{};
    p.x = a.x;
    p.topk_idx = a.topk_idx;
    p.topk_w = a.topk_w;
    // packed buffer: header, gate/up pairs, down pairs
    const size_t gu_sh = (size_t)(a.I / kTileRows) * (a.d / kBK) * kChunkPairBytes;
    const size_t gu_bytes = (size_t)a.E * gu_sh;
    p.w_gu_routed = a.w_routed + kPackHeader;
    p.w_dn_routed = a.w_routed + kPackHeader + gu_bytes;
    p.w_gu_shared = a.w_shared + kPackHeader;
    p.w_dn_shared = a.w_shared + kPackHeader + gu_sh;
    p.mode_routed = reinterpret_cast<const int*>(a.w_routed);
    p.mode_shared = reinterpret_cast<const int*>(a.w_shared);
    p.gu = reinterpret_cast<float*>(a.ws + a.L.dec) + kDecodeMaxT * 256;
    p.acc = reinterpret_cast<float*>(a.ws + a.L.acc);
    p.y = y;
    p.status = reinterpret_cast<int*>(a.ws + a.L.status);
    p.tile_counters = reinterpret_cast<unsigned int*>(p.status + 8);
    p.d = a.d; p.I = a.I; p.E = a.E; p.k = a.k;
    return p;
}

}  // namespace

template <typename K>
cudaError_t launch_pdl(K kernel, int grid, int block, size_t smem, cudaStream_t st, const DecParams& prm) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_decode_gate_up(const FfnArgs& a, cudaStream_t st, unsigned long long* launches) {
    const int MT = a.I / kTileRows, NKC = a.d / kBK / kKbPerCta;
    *launches += 1;
    return launch_pdl(decode_gate_up, (a.k + 1) * MT * NKC, 256, 0, st, make_dec_params(a, nullptr));
}

cudaError_t launch_decode_down(const FfnArgs& a, uint16_t* y, cudaStream_t st, unsigned long long* launches) {
    const int MT = a.d / kTileRows;
    *launches += 1;
    return launch_pdl(decode_down, (a.k + 1) * MT, 256, a.I * sizeof(float), st, make_dec_params(a, y));
}

}  // namespace moe
