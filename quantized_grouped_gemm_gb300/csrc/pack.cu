// pack.cu -- load-time relayout of 4-bit weight stacks into the packed chunk format.
//
// Input: the checkpoint layout of "Optimizing on-device inference for Apple Silicon"
// (section "Dequantize weights during matrix multiplication"): 4-bit codes, 64 weights per
// bf16 scale and bias.  Output: one contiguous 4608-byte chunk per (expert, 128-row tile,
// 64-column K block) holding codes (nibbles reordered so that a shift and a mask give two
// consecutive codes in the mantissa of a bf16 pair), then the 128 scales and 128 biases.
// The buffer starts with a 256-byte header holding the scale encoding (kScaleDenorm when every
// scale of the stack has |s| < 2^-5: scales stored as s * 2^133; else kScaleMagic).
// Chunks are stored in pairs of 9216 bytes: the gate and the up chunk of the same rows, or
// (down stacks) the two 128-row halves of a 256-row tile.
// Still 4 bits per weight: no bf16 copy of the weights is made.
#include "moe_internal.cuh"

namespace moe {
namespace {

// Sets *mode to kScaleMagic if any scale is non-finite or has |s| >= 2^-5 (bf16 0x3D00).
__global__ void scale_check_kernel(size_t n, const uint16_t* __restrict__ scales, int* mode) {
    bool bad = false;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        bad |= (scales[i] & 0x7FFFu) >= 0x3D00u;
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(mode, kScaleMagic);
}

// bf16 bits of s * 2^133 (exact for |s| < 2^-5, the only case it is used for)
__device__ __forceinline__ uint16_t scale_to_denorm(uint16_t s) {
    float f = __uint_as_float((uint32_t)s << 16);
    f = f * 0x1p64f;
    f = f * 0x1p69f;
    return (uint16_t)(__float_as_uint(f) >> 16);
}

__global__ void pack_kernel(int E, int N, int K, const uint8_t* __restrict__ codes,
                            const uint16_t* __restrict__ scales, const uint16_t* __restrict__ biases, int slot,
                            int nslots, uint8_t* __restrict__ dst, const int* __restrict__ mode) {
    const int MT = N / kTileRows, KB = K / kBK;
    const size_t total = (size_t)E * MT * KB * kTileRows;
    const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int r = (int)(idx % kTileRows);
    size_t rest = idx / kTileRows;
    const int kb = (int)(rest % KB);
    rest /= KB;
    const int mt = (int)(rest % MT);
    const int e = (int)(rest / MT);
    const int row = mt * kTileRows + r;
    const uint8_t* src = codes + ((size_t)e * N + row) * (K / 2) + (size_t)kb * (kBK / 2);
    // nslots == 2, slot < 0: the two 128-row halves of a 256-row tile form the pair (down stacks)
    const int tile = slot < 0 ? mt / 2 : mt, s = slot < 0 ? mt % 2 : slot, ntile = slot < 0 ? MT / 2 : MT;
    uint8_t* chunk = dst + ((((size_t)e * ntile + tile) * KB + kb) * nslots + s) * kChunkBytes;
    constexpr int kPerm[8] = {0, 2, 4, 6, 1, 3, 5, 7};   // nibble p <- column offset kPerm[p]
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint8_t* sb = src + 16 * h + 4 * w;
            const uint32_t S = (uint32_t)sb[0] | ((uint32_t)sb[1] << 8) | ((uint32_t)sb[2] << 16) |
                               ((uint32_t)sb[3] << 24);   // column c at nibble c
            uint32_t D = 0;
#pragma unroll
            for (int p = 0; p < 8; ++p) D |= ((S >> (4 * kPerm[p])) & 0xFu) << (4 * p);
            *reinterpret_cast<uint32_t*>(chunk + h * 2048 + r * 16 + 4 * w) = D;
        }
    const size_t gi = ((size_t)e * N + row) * (K / kBK) + kb;
    const uint16_t sc = scales[gi];
    reinterpret_cast<uint16_t*>(chunk + kChunkCodes)[r] = *mode == kScaleDenorm ? scale_to_denorm(sc) : sc;
    reinterpret_cast<uint16_t*>(chunk + kChunkCodes + 256)[r] = biases[gi];
}

}  // namespace

cudaError_t launch_scale_check(size_t n, const uint16_t* scales, int* mode, cudaStream_t st,
                               unsigned long long* launches) {
    const size_t blocks = (n + 255) / 256 < 2048 ? (n + 255) / 256 : 2048;
    scale_check_kernel<<<(unsigned)blocks, 256, 0, st>>>(n, scales, mode);
    *launches += 1;
    return cudaGetLastError();
}

cudaError_t launch_pack(int E, int N, int K, const moe_q4& m, int slot, int nslots, uint8_t* dst, const int* mode,
                        cudaStream_t st, unsigned long long* launches) {
    const size_t total = (size_t)E * (N / kTileRows) * (K / kBK) * kTileRows;
    const int threads = 256;
    const size_t blocks = (total + threads - 1) / threads;
    pack_kernel<<<(unsigned)blocks, threads, 0, st>>>(E, N, K, m.codes_dev, m.scales_dev, m.biases_dev, slot, nslots,
                                                       dst, mode);
    *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
