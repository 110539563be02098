// api.cu -- host side of the C ABI declared in include/moe.h: argument checks, workspace
// layout, tensor maps and kernel launches.  Nothing here allocates device memory or
// synchronises a stream (except moe_read_status, a debug call).
#include <atomic>
#include <cstring>

#include "moe_internal.cuh"

namespace moe {

static std::atomic<unsigned long long> g_launches{0};

void count_launches(unsigned long long n) { g_launches += n; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load();
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f);
    }
    return f;
}

cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    EncodeTiledFn f = encode_fn();
    if (!f) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = f(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static int num_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int v = cache[dev].load();
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(v);
    }
    return v;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Opts {
    int tile_rows = 32;
    int decode_max_tokens = 1;
    int decode_path = MOE_DECODE_AUTO;
    bool deterministic = false;
    bool host_routing = false;
    bool unfused_dequant = false;
    int gemm_rows = kGemmRowsDefault;
};

static int get_opts(const moe_options* o, Opts* out) {
    Opts r;
    if (o) {
        if (o->tile_rows < 0 || o->decode_max_tokens < 0) return MOE_ERR_INVALID_ARG;
        if (o->tile_rows > 0) r.tile_rows = o->tile_rows;
        if (o->decode_max_tokens > 1) return MOE_ERR_UNSUPPORTED;
        r.decode_max_tokens = o->decode_max_tokens;
        if (o->decode_path != MOE_DECODE_AUTO && o->decode_path != MOE_DECODE_GEMV) return MOE_ERR_INVALID_ARG;
        r.decode_path = o->decode_path;
        if (o->deterministic != 0 && o->deterministic != 1) return MOE_ERR_INVALID_ARG;
        r.deterministic = o->deterministic == 1;
        if (o->host_routing != 0 && o->host_routing != 1) return MOE_ERR_INVALID_ARG;
        r.host_routing = o->host_routing == 1;
        if (o->unfused_dequant != 0 && o->unfused_dequant != 1) return MOE_ERR_INVALID_ARG;
        r.unfused_dequant = o->unfused_dequant == 1;
        if (o->gemm_rows != 0 && !gemm_rows_valid(o->gemm_rows)) return MOE_ERR_INVALID_ARG;
        if (o->gemm_rows != 0) r.gemm_rows = o->gemm_rows;
    }
    *out = r;
    return MOE_OK;
}

static int check_routing(const moe_routing* rt) {
    if (!rt || !rt->topk_idx_dev || !rt->topk_w_dev || !rt->counts_dev || !rt->offsets_dev || !rt->perm_dev ||
        !rt->pos_dev || !rt->tiles_dev || !rt->num_tiles_dev)
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

static size_t ws_bytes_for(const moe_shape& s, const Opts& o) {
    const WsLayout L = ws_layout(s);
    return o.unfused_dequant && !(s.T >= 1 && s.T <= o.decode_max_tokens) ? L.total_unfused : L.total;
}

static int check_ws(const moe_shape* s, void* ws, size_t bytes, const Opts& o) {
    if (!ws || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    if (bytes < ws_bytes_for(*s, o)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

static size_t gate_up_bytes(const moe_shape& s, int I) { return (size_t)(I / kTileRows) * (s.d / kBK) * kChunkPairBytes; }
static size_t down_bytes(const moe_shape& s, int I) { return (size_t)(s.d / kTileRows) * (I / kBK) * kChunkBytes; }

static RouteArgs route_args(const moe_shape* s, const uint16_t* x, const uint16_t* wr, const float* bias,
                            const moe_routing* rt, void* ws, const Opts& o) {
    RouteArgs a{};
    a.T = s->T; a.d = s->d; a.E = s->E; a.k = s->k; a.I = s->I; a.tile_rows = o.tile_rows;
    a.gu_rows = o.gemm_rows; a.dn_rows = o.gemm_rows < kDnMaxRows ? o.gemm_rows : kDnMaxRows;
    a.x = x; a.w_router = wr; a.bias = bias;
    a.topk_idx = rt->topk_idx_dev; a.topk_w = rt->topk_w_dev; a.counts = rt->counts_dev;
    a.offsets = rt->offsets_dev; a.perm = rt->perm_dev; a.pos = rt->pos_dev; a.tiles = rt->tiles_dev;
    a.num_tiles = rt->num_tiles_dev;
    a.ws = static_cast<uint8_t*>(ws);
    a.L = ws_layout(*s);
    a.num_sms = num_sms();
    return a;
}

static FfnArgs ffn_args(const moe_shape* s, const uint16_t* x, const moe_routing* rt, const void* wr,
                        const void* wsh, void* ws) {
    FfnArgs a{};
    a.T = s->T; a.d = s->d; a.E = s->E; a.k = s->k; a.I = s->I;
    a.x = x;
    a.topk_idx = rt->topk_idx_dev; a.topk_w = rt->topk_w_dev; a.perm = rt->perm_dev;
    a.w_routed = static_cast<const uint8_t*>(wr);
    a.w_shared = static_cast<const uint8_t*>(wsh);
    a.ws = static_cast<uint8_t*>(ws);
    a.L = ws_layout(*s);
    a.num_sms = num_sms();
    return a;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static bool is_decode(const moe_shape* s, const Opts& o) { return s->T >= 1 && s->T <= o.decode_max_tokens; }

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_error_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_STATUS: return "device reported bad routing data";
        case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_WORKSPACE: return "workspace or packed buffer too small";
        default: return "unknown error";
    }
}

int moe_check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->d <= 0 || s->E <= 0 || s->k <= 0 || s->I <= 0 || s->I_shared <= 0 || s->group <= 0)
        return MOE_ERR_INVALID_ARG;
    if (s->E != 256 || s->k != 8 || s->group != 64) return MOE_ERR_UNSUPPORTED;
    if (s->d % 256 != 0 || s->I % 128 != 0 || s->I_shared != s->I) return MOE_ERR_UNSUPPORTED;
    if (s->T > 65536 || s->d > 7168 || s->I > 8192) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

size_t moe_workspace_bytes(const moe_shape* s, const moe_options* o) {
    Opts op;
    if (moe_check_shape(s) != MOE_OK || get_opts(o, &op) != MOE_OK) return 0;
    return ws_bytes_for(*s, op);
}

size_t moe_max_tiles(int T, int k, int E, int tile_rows) {
    if (T < 0 || k <= 0 || E <= 0) return 0;
    if (tile_rows <= 0) tile_rows = 32;
    return ((size_t)k * T + tile_rows - 1) / tile_rows + E;
}

size_t moe_packed_bytes(const moe_shape* s, int num_experts, int I) {
    if (moe_check_shape(s) != MOE_OK || num_experts <= 0 || I <= 0 || I % 128 != 0) return 0;
    return kPackHeader + (size_t)num_experts * (gate_up_bytes(*s, I) + down_bytes(*s, I));
}

int moe_pack_weights(const moe_shape* s, const moe_expert_weights* src, int I, void* dst, size_t dst_bytes,
                     void* stream) {
    int rc = moe_check_shape(s);
    if (rc != MOE_OK) return rc;
    if (!src || !dst || !aligned(dst, 256) || I <= 0 || I % 128 != 0 || src->num_experts <= 0)
        return MOE_ERR_INVALID_ARG;
    const moe_q4* mats[3] = {&src->gate, &src->up, &src->down};
    for (const moe_q4* m : mats)
        if (!m->codes_dev || !m->scales_dev || !m->biases_dev || !aligned(m->codes_dev, 4) ||
            !aligned(m->scales_dev, 2) || !aligned(m->biases_dev, 2))
            return MOE_ERR_INVALID_ARG;
    const int E = src->num_experts;
    if (dst_bytes < moe_packed_bytes(s, E, I)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* hdr = static_cast<uint8_t*>(dst);
    int* mode = reinterpret_cast<int*>(hdr);
    uint8_t* d8 = hdr + kPackHeader;
    unsigned long long n = 0;
    cudaError_t e = cudaMemsetAsync(hdr, 0, kPackHeader, st);
    const size_t ngu = (size_t)E * I * (s->d / 64), ndn = (size_t)E * s->d * (I / 64);
    if (e == cudaSuccess) e = launch_scale_check(ngu, src->gate.scales_dev, mode, st, &n);
    if (e == cudaSuccess) e = launch_scale_check(ngu, src->up.scales_dev, mode, st, &n);
    if (e == cudaSuccess) e = launch_scale_check(ndn, src->down.scales_dev, mode, st, &n);
    if (e == cudaSuccess) e = launch_pack(E, I, s->d, src->gate, 0, 2, d8, mode, st, &n);
    if (e == cudaSuccess) e = launch_pack(E, I, s->d, src->up, 1, 2, d8, mode, st, &n);
    if (e == cudaSuccess)
        e = launch_pack(E, s->d, I, src->down, -1, 2, d8 + (size_t)E * gate_up_bytes(*s, I), mode, st, &n);
    // a memset last: a kernel launched next with programmatic dependent launch (the decode
    // kernels read weights before their wait) is then ordered after the packs, not overlapped
    if (e == cudaSuccess) e = cudaMemsetAsync(hdr + 4, 0, 4, st);
    g_launches += n;
    return cuda_status(e);
}

static int route_impl(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
                      const moe_routing* rt, void* ws, size_t ws_bytes, const moe_options* o, void* stream,
                      const void* packed_shared) {
    int rc = moe_check_shape(s);
    if (rc != MOE_OK) return rc;
    Opts op;
    if ((rc = get_opts(o, &op)) != MOE_OK) return rc;
    if (s->T == 0) return MOE_OK;
    if ((rc = check_routing(rt)) != MOE_OK) return rc;
    if ((rc = check_ws(s, ws, ws_bytes, op)) != MOE_OK) return rc;
    if (!x || !w_router || !aligned(x, 16) || !aligned(w_router, 16) || (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    RouteArgs a = route_args(s, x, w_router, bias, rt, ws, op);
    if (packed_shared) {   // decode: warm L2 with the shared expert's weights while routing
        a.pf_ptr = static_cast<const uint8_t*>(packed_shared);
        a.pf_bytes = moe_packed_bytes(s, 1, s->I_shared);
    }
    unsigned long long n = 0;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = is_decode(s, op)     ? launch_route_decode(a, st, &n)
                    : op.host_routing ? launch_route_prefill_host(a, st, &n)
                                      : launch_route_prefill(a, st, &n);
    g_launches += n;
    return cuda_status(e);
}

int moe_router_logits(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
                      float* logits, void* stream) {
    int rc = moe_check_shape(s);
    if (rc != MOE_OK) return rc;
    if (s->T == 0) return MOE_OK;
    if (!x || !w_router || !logits || !aligned(x, 16) || !aligned(w_router, 16) || !aligned(logits, 16) ||
        (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    unsigned long long n = 0;
    const cudaError_t e = launch_router_logits(x, w_router, bias, logits, s->T, s->d, static_cast<cudaStream_t>(stream), &n);
    g_launches += n;
    return cuda_status(e);
}

int moe_route(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias,
              const moe_routing* rt, void* ws, size_t ws_bytes, const moe_options* o, void* stream) {
    return route_impl(s, x, w_router, bias, rt, ws, ws_bytes, o, stream, nullptr);
}

static int ffn_common(const moe_shape* s, const uint16_t* x, const moe_routing* rt, const void* wr, const void* wsh,
                      void* ws, size_t ws_bytes, const moe_options* o, Opts* op, bool need_x) {
    int rc = moe_check_shape(s);
    if (rc != MOE_OK) return rc;
    if ((rc = get_opts(o, op)) != MOE_OK) return rc;
    if (s->T == 0) return 1;
    if ((rc = check_routing(rt)) != MOE_OK) return rc;
    if ((rc = check_ws(s, ws, ws_bytes, *op)) != MOE_OK) return rc;
    if (!wr || !wsh || !aligned(wr, 256) || !aligned(wsh, 256)) return MOE_ERR_INVALID_ARG;
    if (need_x && (!x || !aligned(x, 16))) return MOE_ERR_INVALID_ARG;
    if (num_sms() <= 0) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_ffn_gate_up(const moe_shape* s, const uint16_t* x, const moe_routing* rt, const void* wr, const void* wsh,
                    void* ws, size_t ws_bytes, const moe_options* o, void* stream) {
    Opts op;
    int rc = ffn_common(s, x, rt, wr, wsh, ws, ws_bytes, o, &op, true);
    if (rc != MOE_OK) return rc == 1 ? MOE_OK : rc;
    FfnArgs a = ffn_args(s, x, rt, wr, wsh, ws);
    a.unfused = op.unfused_dequant;
    unsigned long long n = 0;
    cudaError_t e;
    if (is_decode(s, op)) {
        e = launch_decode_gate_up(a, static_cast<cudaStream_t>(stream), &n);
    } else {
        e = launch_gate_up_tm(a, static_cast<cudaStream_t>(stream), &n);
    }
    g_launches += n;
    return cuda_status(e);
}

int moe_ffn_down(const moe_shape* s, const moe_routing* rt, const void* wr, const void* wsh, void* ws,
                 size_t ws_bytes, const moe_options* o, void* stream) {
    Opts op;
    int rc = ffn_common(s, nullptr, rt, wr, wsh, ws, ws_bytes, o, &op, false);
    if (rc != MOE_OK) return rc == 1 ? MOE_OK : rc;
    FfnArgs a = ffn_args(s, nullptr, rt, wr, wsh, ws);
    a.rows_out = ffn_rows_output(s->T, s->d, s->k, op.deterministic);
    a.unfused = op.unfused_dequant;
    unsigned long long n = 0;
    cudaError_t e;
    if (is_decode(s, op)) {
        e = launch_decode_down(a, nullptr, static_cast<cudaStream_t>(stream), &n);
    } else {
        e = launch_down_tm(a, static_cast<cudaStream_t>(stream), &n);
    }
    g_launches += n;
    return cuda_status(e);
}

int moe_grouped_ffn(const moe_shape* s, const uint16_t* x, const moe_routing* rt, const void* wr, const void* wsh,
                    void* ws, size_t ws_bytes, const moe_options* o, void* stream) {
    int rc = moe_ffn_gate_up(s, x, rt, wr, wsh, ws, ws_bytes, o, stream);
    if (rc != MOE_OK) return rc;
    return moe_ffn_down(s, rt, wr, wsh, ws, ws_bytes, o, stream);
}

int moe_combine(const moe_shape* s, const moe_routing* rt, void* ws, size_t ws_bytes, uint16_t* y,
                const moe_options* o, void* stream) {
    int rc = moe_check_shape(s);
    if (rc != MOE_OK) return rc;
    Opts op;
    if ((rc = get_opts(o, &op)) != MOE_OK) return rc;
    if (s->T == 0) return MOE_OK;
    if ((rc = check_ws(s, ws, ws_bytes, op)) != MOE_OK) return rc;
    if (!y || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(*s);
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    unsigned long long n = 0;
    cudaError_t e;
    if (!is_decode(s, op) && ffn_rows_output(s->T, s->d, s->k, op.deterministic)) {
        // prefill: the down projection left weighted rows in Y; sum each token's rows
        if ((rc = check_routing(rt)) != MOE_OK) return rc;
        e = launch_combine_rows(s->T, s->d, s->k, reinterpret_cast<const float*>(w8 + L.Y), rt->pos_dev, y,
                                static_cast<cudaStream_t>(stream), &n);
    } else {
        e = launch_combine(s->T, s->d, reinterpret_cast<const float*>(w8 + L.acc), y, static_cast<cudaStream_t>(stream),
                           &n);
    }
    g_launches += n;
    return cuda_status(e);
}

int moe_forward(const moe_shape* s, const uint16_t* x, const uint16_t* w_router, const float* bias, const void* wr,
                const void* wsh, const moe_routing* rt, void* ws, size_t ws_bytes, uint16_t* y, const moe_options* o,
                void* stream) {
    Opts op;
    int rc = get_opts(o, &op);
    if (rc != MOE_OK) return rc;
    if (s && s->T == 1 && is_decode(s, op) && op.decode_path == MOE_DECODE_AUTO) {
        // one launch for the whole token when the shape and the GPU allow it
        if ((rc = moe_check_shape(s)) != MOE_OK) return rc;
        if ((rc = check_routing(rt)) != MOE_OK) return rc;
        if ((rc = check_ws(s, ws, ws_bytes, op)) != MOE_OK) return rc;
        if (!x || !w_router || !wr || !wsh || !y || !aligned(x, 16) || !aligned(w_router, 16) ||
            (bias && !aligned(bias, 4)) || !aligned(wr, 256) || !aligned(wsh, 256) || !aligned(y, 16))
            return MOE_ERR_INVALID_ARG;
        const WsLayout L = ws_layout(*s);
        uint8_t* w8 = static_cast<uint8_t*>(ws);
        FusedDecodeArgs fa{};
        fa.d = s->d; fa.E = s->E; fa.k = s->k; fa.I = s->I;
        fa.x = x; fa.w_router = w_router; fa.bias = bias;
        fa.w_routed = static_cast<const uint8_t*>(wr);
        fa.w_shared = static_cast<const uint8_t*>(wsh);
        fa.topk_idx = rt->topk_idx_dev; fa.topk_w = rt->topk_w_dev; fa.counts = rt->counts_dev;
        fa.offsets = rt->offsets_dev; fa.perm = rt->perm_dev; fa.pos = rt->pos_dev; fa.tiles = rt->tiles_dev;
        fa.num_tiles = rt->num_tiles_dev;
        fa.status = reinterpret_cast<int*>(w8 + L.status);
        fa.logit_words = reinterpret_cast<unsigned long long*>(w8 + L.fzlog);
        fa.acc = reinterpret_cast<float*>(w8 + L.acc);
        fa.y = y;
#ifdef MOE_TRACE
        fa.trace = reinterpret_cast<unsigned long long*>(w8 + L.trace);
#endif
        unsigned long long n = 0;
        cudaError_t e = launch_decode_fused(fa, static_cast<cudaStream_t>(stream), &n);
        g_launches += n;
        if (e != cudaErrorNotSupported) return cuda_status(e);
        // otherwise the three decode kernels below
    }
    const bool dec = s && is_decode(s, op) && wsh && aligned(wsh, 256);
    rc = route_impl(s, x, w_router, bias, rt, ws, ws_bytes, o, stream, dec ? wsh : nullptr);
    if (rc != MOE_OK || s->T == 0) return rc;
    if (is_decode(s, op)) {
        // decode: the down GEMV also writes y (its last CTA per row tile converts to bf16)
        rc = moe_ffn_gate_up(s, x, rt, wr, wsh, ws, ws_bytes, o, stream);
        if (rc != MOE_OK) return rc;
        if (!y || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
        FfnArgs a = ffn_args(s, x, rt, wr, wsh, ws);
        unsigned long long n = 0;
        cudaError_t e = launch_decode_down(a, y, static_cast<cudaStream_t>(stream), &n);
        g_launches += n;
        return cuda_status(e);
    }
    rc = moe_grouped_ffn(s, x, rt, wr, wsh, ws, ws_bytes, o, stream);
    if (rc != MOE_OK) return rc;
    return moe_combine(s, rt, ws, ws_bytes, y, o, stream);
}

int moe_read_status(void* ws, void* stream, int* status_out) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (status_out) *status_out = v;
    if (v & MOE_STATUS_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
    if (v) return MOE_ERR_DEVICE_STATUS;
    return MOE_OK;
}

unsigned long long moe_launch_count(void) { return g_launches.load(); }

}  // extern "C"
