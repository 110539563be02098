/* moe.h -- C ABI of the GB300 (sm_103a) sparse-MoE expert path.
 *
 * The path (one MoE layer of a hybrid MoE language model; "Optimizing on-device inference
 * for Apple Silicon", Perplexity Engineering 2026):
 *   route        router logits over E = 256 experts, top-8, routing weights, per-expert
 *                histogram, exclusive prefix scan to group offsets, stable scatter of the
 *                token rows into expert groups, block map of fixed-size row tiles
 *                (sections "Qwen creates three different workload shapes" and "Keep expert
 *                routing on the GPU"; tile rows: "Match tile size to expert load").
 *   grouped_ffn  per expert group: SwiGLU FFN whose 4-bit group-affine weights are rebuilt
 *                in bf16 tile by tile on chip (64 weights share one bf16 scale and bias,
 *                w = scale*q + bias), fp32 accumulation; the output projection is weighted by
 *                the routing score (1 for the always-on shared expert) in fp32 (sections
 *                "Dequantize weights during matrix multiplication" and "Reduce intermediate
 *                and state traffic").
 *   combine      each token's k weighted routed rows and its shared row are summed in fp32
 *                (a fixed order: routing slot 0..k-1, then the shared expert) and written
 *                out as bf16.
 * Batch-1 decode (T <= options.decode_max_tokens) runs the same calls on GEMV kernels
 * (section "Optimize the single-row weight path").
 *
 * Conventions
 *   - Every pointer argument named *_dev is CUDA device memory owned by the caller; the
 *     library never allocates, frees, or keeps pointers between calls.  bf16 values are
 *     passed as their 16-bit patterns (uint16_t).  All device buffers must be 16-byte
 *     aligned (256-byte for the workspace).
 *   - stream is a cudaStream_t passed as void*.  Calls are asynchronous on that stream,
 *     never synchronise it, and do no device-to-host copies; results are valid when the
 *     stream reaches them.  The three path calls of one layer must share a stream.
 *   - Return values: MOE_OK or a negative MOE_ERR_*.  Argument errors are found on the host
 *     before anything is launched.  Errors found on the device (a routing index out of
 *     range, a bounded wait that ran out) set bits of the status word kept in the workspace;
 *     read it with moe_read_status (a synchronising debug call).
 *   - Supported shapes: E = 256, k = 8, group = 64, d % 256 == 0, I % 128 == 0,
 *     I_shared == I, 0 <= T <= 65536, d <= 7168, I <= 8192.  T = 0 is a no-op.
 *     I % 128 (not only a whole number of 64-weight groups) is a deliberate restriction:
 *     every gate/up weight tile is one 128-row tensor-core operand (M = 128, one TMEM lane
 *     per row) and the packed layout cuts rows in 128s; an I with a 64-row remainder would
 *     need zero-padded rows in the packed weights and masked writes of h.  Other shapes
 *     return MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG -1    /* null pointer, negative or inconsistent size, misalignment */
#define MOE_ERR_UNSUPPORTED -2    /* a shape outside the supported set above */
#define MOE_ERR_CUDA -3           /* a CUDA runtime call failed (launch, attribute, tensor map) */
#define MOE_ERR_DEVICE_STATUS -4  /* moe_read_status: the device flagged bad routing data */
#define MOE_ERR_DEVICE_TIMEOUT -5 /* moe_read_status: a bounded wait inside a kernel ran out */
#define MOE_ERR_WORKSPACE -6      /* workspace or packed-weight buffer smaller than required */

/* Device status bits (moe_read_status) */
#define MOE_STATUS_BAD_EXPERT 0x1   /* an expert index outside [0, E) reached the FFN */
#define MOE_STATUS_TIMEOUT 0x2      /* a pipeline wait gave up */

/* Problem sizes: T tokens, hidden d, E routed experts, top-k, expert intermediate I,
 * shared-expert intermediate I_shared, quant group (weights per scale/bias). */
typedef struct moe_shape {
    int T, d, E, k, I, I_shared, group;
} moe_shape;

/* One stack of 4-bit group-affine matrices in the checkpoint layout, expert outermost:
 *   codes  uint8 [n_experts][N][K/2]; code k of a row is the low nibble of byte k/2 for
 *          even k and the high nibble for odd k; unsigned values 0..15
 *   scales bf16  [n_experts][N][K/64]   (group g covers weights 64g .. 64g+63 of the row)
 *   biases bf16  [n_experts][N][K/64]
 * Weight (n, k) = bf16_round_nearest_even(scale * code + bias) (one rounding). */
typedef struct moe_q4 {
    const uint8_t* codes_dev;
    const uint16_t* scales_dev;
    const uint16_t* biases_dev;
} moe_q4;

/* The three projections of num_experts SwiGLU experts.  gate/up: N = I, K = d;
 * down: N = d, K = I.  h = silu(x.gate) * (x.up); y = h.down. */
typedef struct moe_expert_weights {
    moe_q4 gate, up, down;
    int num_experts;
} moe_expert_weights;

/* Routing results, all caller-owned device buffers (sizes for T tokens, E experts, top-k):
 *   topk_idx  int32 [T][k]   expert of slot j (slots in rank order, ties -> lower index)
 *   topk_w    fp32  [T][k]   routing weights: softmax over the E logits renormalised
 *                            over the kept k (sum to 1 per token)
 *   counts    int32 [E]      rows routed to each expert
 *   offsets   int32 [E+1]    exclusive prefix scan of counts; offsets[E] = k*T
 *   perm      int32 [k*T]    group row p -> assignment t*k + j (rows of a group ascend in t)
 *   pos       int32 [T][k]   assignment -> group row (the inverse of perm)
 *   tiles     int32 [moe_max_tiles(T, tile_rows)][3]  block map (expert, first row, rows),
 *                            expert-ascending, tile_rows rows each but the last of a group
 *   num_tiles int32 [1]      number of valid tiles */
typedef struct moe_routing {
    int32_t* topk_idx_dev;
    float* topk_w_dev;
    int32_t* counts_dev;
    int32_t* offsets_dev;
    int32_t* perm_dev;
    int32_t* pos_dev;
    int32_t* tiles_dev;
    int32_t* num_tiles_dev;
} moe_routing;

/* Options.  Zero-initialise and set what you need; zero fields take the defaults. */
/* Values of moe_options.decode_path. */
#define MOE_DECODE_AUTO 0   /* moe_forward with T = 1: one fused launch when it fits the GPU */
#define MOE_DECODE_GEMV 1   /* always the three decode kernels (route, gate/up GEMV, down GEMV) */

typedef struct moe_options {
    int tile_rows;          /* rows per exported block-map tile; default 32 */
    int decode_max_tokens;  /* T at or below this runs the decode (GEMV) kernels; default 1 */
    int decode_path;        /* MOE_DECODE_AUTO (default) or MOE_DECODE_GEMV */
    int deterministic;      /* 0 (default): prefill adds each token's weighted rows into an fp32
                               sum with bulk reduce-adds (addition order not fixed, so the last
                               bits may differ between calls); 1: the rows are stored and summed
                               per token in a fixed order, so repeated calls give identical bits
                               (slower: the rows make a round trip through L2, or HBM at large T) */
    int host_routing;       /* 0 (default): the routing scan and block map stay on the GPU.
                               1: an ablation of that design ("GPU-resident routing" on the
                               page): moe_route copies the per-block expert counts to the host,
                               computes counts, offsets, block map and GEMM tile lists there,
                               copies them back and then scatters.  It synchronises the stream
                               once per call (so it cannot be captured in a CUDA graph) and gives
                               results identical to 0.  Ignored by the decode path. */
    int unfused_dequant;    /* 0 (default): weights are dequantised on chip inside the grouped
                               GEMMs.  1: an ablation of that design ("Dequantize weights during
                               matrix multiplication" on the page): each FFN call first writes
                               every expert's weights of that projection as bf16 into the
                               workspace (about 6 MB per expert at d=2048, I=512; the workspace
                               grows accordingly, see moe_workspace_bytes) and the GEMM then
                               streams those.  Same bf16 weights, same results bit for bit.
                               Ignored by the decode path. */
    int gemm_rows;          /* prefill: largest number of token rows in one grouped-GEMM block, 16, 32,
                               64 or 128 (default 128; 0 takes the default, other values are an
                               argument error).  Each expert's rows are cut into near-equal blocks
                               of at most this many rows (the down projection caps its blocks at
                               96 rows), and every block streams its expert's weights once per
                               projection ("Match tile size to expert load" on the page).  Used by moe_route, which writes the GEMM tile lists that
                               moe_grouped_ffn reads.  Every value gives the same routing and the
                               same outputs up to fp32 summation order.  Ignored by the decode
                               path. */
    int reserved[1];
} moe_options;

/* Human-readable text for a return code. */
const char* moe_error_string(int code);

/* Check a shape against the supported set: MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED. */
int moe_check_shape(const moe_shape* shape);

/* Bytes of the caller-provided workspace for this shape (0 if the shape is unsupported).
 * The workspace holds routing scratch, the gathered rows, the intermediate h, the fp32
 * weighted output rows ((k+1) T x d), the fp32 token-order sum of the decode kernels and the
 * device status word.  One workspace serves one stream at a time. */
size_t moe_workspace_bytes(const moe_shape* shape, const moe_options* options);

/* Number of int32 triples the block map (moe_routing.tiles) can need: ceil(k*T/tile_rows) + E. */
size_t moe_max_tiles(int T, int k, int E, int tile_rows);

/* Bytes of the device-friendly 4-bit layout of a weight stack (see moe_pack_weights). */
size_t moe_packed_bytes(const moe_shape* shape, int num_experts, int intermediate);

/* Load-time relayout of one expert-weight stack into the library's packed 4-bit form:
 * per (expert, 128-row tile, 64-wide K block) one contiguous chunk of codes (nibbles
 * reordered for register-level unpacking), scales and biases; gate and up chunks are
 * interleaved.  The packed form is still 4 bits per weight plus the bf16 scale and bias
 * per group; no bf16 copy of the weights is made.  `intermediate` is I for the routed
 * stack and I_shared for the shared one.  dst_dev (packed_bytes bytes, caller-owned) is
 * written asynchronously on stream.  Call once per weight stack, outside any timed region. */
int moe_pack_weights(const moe_shape* shape, const moe_expert_weights* src, int intermediate, void* dst_dev,
                     size_t dst_bytes, void* stream);

/* Step a1-a6: router logits (x [T][d] bf16, w_router [E][d] bf16, optional fp32 logit_bias
 * [E] added after the dot product), top-k with weights, histogram, prefix scan, stable
 * scatter, block map.  Also gathers the routed rows into expert order inside the workspace
 * for moe_grouped_ffn.
 * The logit of (t, e) is fixed bit-exactly: 32 partial fp32 sums, sum l taking
 * k = 256*i + 8*l + j (i ascending, j = 0..7) with fused multiply-adds from 0, then the
 * tree s[i] += s[i+m] for m = 16, 8, 4, 2, 1, then + logit_bias[e].
 * Prefill kernels are launched with programmatic dependent launch; the first two read
 * w_router_dev before the previous kernel on the stream has finished (everything else only
 * after it), so w_router_dev must not be written by the kernel launched just before this call
 * on the same stream. */
int moe_route(const moe_shape* shape, const uint16_t* x_dev, const uint16_t* w_router_dev,
              const float* logit_bias_dev, const moe_routing* routing, void* workspace_dev,
              size_t workspace_bytes, const moe_options* options, void* stream);

/* Step a1 on its own: every router logit of every token, exactly as moe_route defines them
 * (the fixed fp32 order above, then + logit_bias[e]), computed by the same device code that
 * moe_route uses for its exact recomputation.  logits_dev: fp32 [T][E], caller-owned, written
 * asynchronously on stream.  x_dev and w_router_dev 16-byte aligned, logit_bias_dev (nullable)
 * 4-byte aligned, logits_dev 16-byte aligned; no workspace.  For inspection and tests: moe_route
 * itself does not materialise all logits. */
int moe_router_logits(const moe_shape* shape, const uint16_t* x_dev, const uint16_t* w_router_dev,
                      const float* logit_bias_dev, float* logits_dev, void* stream);

/* Steps a7-a9: for every expert group and the shared expert, gate/up projections with
 * SwiGLU (h kept to 16 bits as a bf16 pair), output projection, and the fp32 weighting
 * (routing weight topk_w for routed rows, 1 for the shared expert).  Prefill writes every
 * weighted output row into the workspace (rows in expert-group order, then the shared
 * expert's rows); decode shapes (T <= options.decode_max_tokens) add into the fp32 token-order
 * sum instead.  Weights are the packed stacks written by moe_pack_weights (routed: E experts
 * with I; shared: 1 expert with I_shared).  Requires moe_route on the same workspace and
 * stream first. */
int moe_grouped_ffn(const moe_shape* shape, const uint16_t* x_dev, const moe_routing* routing,
                    const void* packed_routed_dev, const void* packed_shared_dev, void* workspace_dev,
                    size_t workspace_bytes, const moe_options* options, void* stream);

/* Sub-steps of moe_grouped_ffn, in this order (exposed so callers can time them apart):
 * gate/up + SwiGLU into h, then output projection + weighted accumulation. */
int moe_ffn_gate_up(const moe_shape* shape, const uint16_t* x_dev, const moe_routing* routing,
                    const void* packed_routed_dev, const void* packed_shared_dev, void* workspace_dev,
                    size_t workspace_bytes, const moe_options* options, void* stream);
int moe_ffn_down(const moe_shape* shape, const moe_routing* routing, const void* packed_routed_dev,
                 const void* packed_shared_dev, void* workspace_dev, size_t workspace_bytes,
                 const moe_options* options, void* stream);

/* Step a10: y [T][d] bf16 (round to nearest even).  Prefill: the sum, in fp32 and in a fixed
 * order, of each token's k weighted routed rows (found through routing.pos) and its shared
 * row, as moe_grouped_ffn left them.  Decode shapes: the fp32 token-order sum, which it then
 * clears: the decode kernels add into a sum that a fresh (zeroed) workspace or the previous
 * moe_combine / moe_forward left at zero. */
int moe_combine(const moe_shape* shape, const moe_routing* routing, void* workspace_dev, size_t workspace_bytes,
                uint16_t* y_dev, const moe_options* options, void* stream);

/* The whole layer: moe_route, moe_grouped_ffn, moe_combine in one call.
 * One token (T = 1, decode): with options.decode_path = MOE_DECODE_AUTO the layer is one
 * kernel launch (routing, both projections and the combine) when it has at most 72 units of
 * work -- a unit is one 128-row slice of h of one of the k+1 experts, so (k+1) * I/128 <= 72,
 * i.e. I <= 1024 -- and all of its (k+1) * I/128 clusters of 4 CTAs (256 threads each) are
 * resident on the GPU at once (cudaOccupancyMaxActiveClusters, checked once per shape);
 * otherwise the three decode kernels run.  Decode kernels are launched with programmatic dependent launch: they read
 * w_router_dev, logit_bias_dev and the packed weights before the previous kernel on the
 * stream has finished (x_dev and the workspace only after), so those inputs must not be
 * written by the kernel launched just before this call on the same stream (moe_pack_weights
 * ends with a memset, which orders a following launch after it).
 * The one-launch kernel adds into the workspace's fp32 sum, which every completed moe_forward
 * and moe_combine leaves at zero (moe_ffn_down without moe_combine does not).
 * After a MOE_ERR_DEVICE_TIMEOUT the workspace counters are undefined: zero it again. */
int moe_forward(const moe_shape* shape, const uint16_t* x_dev, const uint16_t* w_router_dev,
                const float* logit_bias_dev, const void* packed_routed_dev, const void* packed_shared_dev,
                const moe_routing* routing, void* workspace_dev, size_t workspace_bytes, uint16_t* y_dev,
                const moe_options* options, void* stream);

/* Synchronise stream, read and clear the device status word of a workspace.
 * Returns MOE_OK, MOE_ERR_DEVICE_STATUS or MOE_ERR_DEVICE_TIMEOUT; *status_out (if not
 * null) gets the raw MOE_STATUS_* bits.  A debug/test call: it blocks the host. */
int moe_read_status(void* workspace_dev, void* stream, int* status_out);

/* Number of kernels this library has launched in this process (diagnostics). */
unsigned long long moe_launch_count(void);

/* Size of the device scratch array behind moe_forward_decode_static. */
#define MOE_STATIC_SCRATCH_BYTES 131072

/* Batch-1 decode forward (T = 1) that allocates nothing and takes no workspace.
 * This call has no counterpart on the pages; it is here for callers that cannot provide
 * scratch memory: a plugin that is handed only its input and output device pointers by a
 * host program owning every allocation, or a service loop that must not allocate once it
 * runs.  It computes what moe_forward computes for one token (routing into *routing, the
 * layer output into y_dev [d] bf16) with its scratch in a fixed array of
 * MOE_STATIC_SCRATCH_BYTES in the library's device memory, which every GPU that loads the
 * library holds until the process exits.
 * - Shapes whose scratch (256 + d*4 + 8*E*4 + 18*I*4 + 64*E bytes, each part rounded up to
 *   256) exceeds the array are rejected with MOE_ERR_WORKSPACE; T != 1 gives
 *   MOE_ERR_UNSUPPORTED.  Both are checked before any pointer argument and before any CUDA
 *   call.  Other checks as moe_forward; the one-launch kernel runs when moe_forward would run
 *   it, else the three decode kernels (e.g. I = 1152, whose 81 units do not fit at once).
 * - No cudaMalloc/cudaFree or allocating library call is made.  The first call on a device
 *   looks up the array's device address (cudaGetSymbolAddress); make that first call before
 *   any stream capture.
 * - All calls share the array and it keeps the last call's contents; each call clears the
 *   part that must start at zero.  Calls that overlap on the GPU (e.g. two streams at once)
 *   race on it: serialise them.
 * - Device-side status bits are not reported by this call (use moe_forward with a workspace
 *   and moe_read_status for diagnostics). */
int moe_forward_decode_static(const moe_shape* shape, const uint16_t* x_dev, const uint16_t* w_router_dev,
                              const float* logit_bias_dev, const void* packed_routed_dev,
                              const void* packed_shared_dev, const moe_routing* routing, uint16_t* y_dev,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
