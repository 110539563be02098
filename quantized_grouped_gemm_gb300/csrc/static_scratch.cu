// static_scratch.cu -- batch-1 decode forward that allocates nothing and takes no workspace.
//
// Some callers cannot hand the library a workspace: a plugin that receives only its input and
// output device pointers from a host program that owns every allocation, or a service loop
// that must not allocate once it has started.  moe_forward_decode_static serves them: its
// scratch (status word and counters, router logits, gate/up accumulators, the fp32 output sum)
// is a fixed array in this file's device memory.  It runs the same kernels as moe_forward with
// T = 1 (the fused one-launch kernel when it fits, else the three decode kernels).
//
// The array is shared by every call on a device and keeps the previous call's contents; each
// call clears the part that must start at zero (status word and counters) with an async memset
// on the caller's stream, and the router kernel clears the accumulators.  Calls whose kernels
// overlap on the GPU (two streams at once) race on the array.
#include <atomic>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

void count_launches(unsigned long long n);

namespace {

static __device__ __align__(256) uint8_t g_decode_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
uint8_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device; looked up once per device (the
// name is only a host-side stand-in for the array).
uint8_t* scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
    }
    return g_scratch_ptr[dev];
}

// Scratch layout inside the array: status word and counters, the fp32 output sum [d] (both
// decode paths add into it), the GEMV path's router logits [8][E] and g/u sums [k+1][2][I],
// then the fused kernel's eight copies of the tagged logits [8][E].
WsLayout static_layout(const moe_shape& s) {
    WsLayout L{};
    size_t o = 0;
    L.status = o; o = align_up(o + 64 * 4, 256);
    L.acc = o; o = align_up(o + (size_t)s.d * 4, 256);
    L.dec = o; o = align_up(o + (size_t)kDecodeMaxT * s.E * 4 + (size_t)(s.k + 1) * 2 * s.I * 4, 256);
    L.fzlog = o; o = align_up(o + (size_t)8 * s.E * 8, 256);
    L.total = o;
    L.nblk = 1;
    return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_forward_decode_static(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                                         const float* logit_bias, const void* packed_routed,
                                         const void* packed_shared, const moe_routing* rt, uint16_t* y,
                                         void* stream) {
    // the shape and its scratch size first: a shape that cannot run is refused whatever the
    // pointers are
    int rc = moe_check_shape(s);
    if (rc != MOE_OK) return rc;
    if (s->T != 1) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = static_layout(*s);
    if (L.total > (size_t)MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    if (!rt || !rt->topk_idx_dev || !rt->topk_w_dev || !rt->counts_dev || !rt->offsets_dev || !rt->perm_dev ||
        !rt->pos_dev || !rt->tiles_dev || !rt->num_tiles_dev)
        return MOE_ERR_INVALID_ARG;
    if (!x || !w_router || !packed_routed || !packed_shared || !y || !aligned16(x) || !aligned16(w_router) ||
        !aligned16(y) || (reinterpret_cast<uintptr_t>(packed_routed) & 255) ||
        (reinterpret_cast<uintptr_t>(packed_shared) & 255) || (logit_bias && (reinterpret_cast<uintptr_t>(logit_bias) & 3)))
        return MOE_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    uint8_t* ws = scratch_address(dev);
    if (!ws) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // status word and every counter must start at zero; word 4 (the fused kernel's epoch of its
    // tagged logits) must not go back to an earlier value, so it is left alone
    if (cudaMemsetAsync(ws + L.status, 0, 4 * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(ws + L.status + 5 * 4, 0, 59 * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    // and the fp32 sum (zero after every completed call; cleared here all the same)
    if (cudaMemsetAsync(ws + L.acc, 0, (size_t)s->d * 4, st) != cudaSuccess) return MOE_ERR_CUDA;

    {   // one launch for the whole token when it fits (as moe_forward)
        FusedDecodeArgs fa{};
        fa.d = s->d; fa.E = s->E; fa.k = s->k; fa.I = s->I;
        fa.x = x; fa.w_router = w_router; fa.bias = logit_bias;
        fa.w_routed = static_cast<const uint8_t*>(packed_routed);
        fa.w_shared = static_cast<const uint8_t*>(packed_shared);
        fa.topk_idx = rt->topk_idx_dev; fa.topk_w = rt->topk_w_dev; fa.counts = rt->counts_dev;
        fa.offsets = rt->offsets_dev; fa.perm = rt->perm_dev; fa.pos = rt->pos_dev; fa.tiles = rt->tiles_dev;
        fa.num_tiles = rt->num_tiles_dev;
        fa.status = reinterpret_cast<int*>(ws + L.status);
        fa.logit_words = reinterpret_cast<unsigned long long*>(ws + L.fzlog);
        fa.acc = reinterpret_cast<float*>(ws + L.acc);
        fa.y = y;
        unsigned long long nf = 0;
        const cudaError_t ef = launch_decode_fused(fa, st, &nf);
        count_launches(nf);
        if (ef != cudaErrorNotSupported) return ef == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }

    RouteArgs ra{};
    ra.T = 1; ra.d = s->d; ra.E = s->E; ra.k = s->k; ra.I = s->I; ra.tile_rows = 32;
    ra.gu_rows = kGemmRowsDefault;
    ra.dn_rows = kDnMaxRows;
    ra.x = x; ra.w_router = w_router; ra.bias = logit_bias;
    ra.topk_idx = rt->topk_idx_dev; ra.topk_w = rt->topk_w_dev; ra.counts = rt->counts_dev;
    ra.offsets = rt->offsets_dev; ra.perm = rt->perm_dev; ra.pos = rt->pos_dev; ra.tiles = rt->tiles_dev;
    ra.num_tiles = rt->num_tiles_dev;
    ra.ws = ws;
    ra.L = L;
    ra.pf_ptr = static_cast<const uint8_t*>(packed_shared);   // warm L2 with the shared expert while routing
    ra.pf_bytes = moe_packed_bytes(s, 1, s->I_shared);
    FfnArgs fa{};
    fa.T = 1; fa.d = s->d; fa.E = s->E; fa.k = s->k; fa.I = s->I;
    fa.x = x; fa.topk_idx = rt->topk_idx_dev; fa.topk_w = rt->topk_w_dev; fa.perm = rt->perm_dev;
    fa.w_routed = static_cast<const uint8_t*>(packed_routed);
    fa.w_shared = static_cast<const uint8_t*>(packed_shared);
    fa.ws = ws;
    fa.L = L;
    unsigned long long n = 0;
    cudaError_t e = launch_route_decode(ra, st, &n);
    if (e == cudaSuccess) e = launch_decode_gate_up(fa, st, &n);
    if (e == cudaSuccess) e = launch_decode_down(fa, y, st, &n);
    count_launches(n);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
