// moe_oracle.cpp -- plain CPU oracle of the sparse-MoE expert path.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline leg of
// the benchmark may load this library.  It shares no code, header, table or helper with
// the CUDA path; the two meet only through the seeded inputs of moe_workload.
//
// What it computes follows "Optimizing on-device inference for Apple Silicon"
// (Perplexity Engineering, 2026):
//   * router: a router scores 256 expert subnetworks per token and keeps eight, plus one
//     shared expert that sees every token  (section "Qwen creates three different
//     workload shapes");
//   * weights: 4-bit codes, groups of 64 weights sharing one bf16 scale and one bf16 bias,
//     reconstructed as bf16 before the matmul; fp32 accumulation  (section "Dequantize
//     weights during matrix multiplication");
//   * routing metadata: per-expert histogram, prefix scan to start offsets, scatter of rows
//     into expert groups, block map of fixed-size tiles  (section "Keep expert routing on
//     the GPU"; tile rows in section "Match tile size to expert load");
//   * the expert FFN is gate/up projections with their gated activation, then the output
//     projection weighted by the routing score plus the shared-expert result  (section
//     "Reduce intermediate and state traffic", its first two fused chains).
//
// Readings where the pages are silent (each is listed in the design notes):
//   R1 router logit order: 32 lane chains, chain l accumulates k = 256*i + 8*l + j
//      (i ascending, j = 0..7) with fmaf from 0.0f; then the fixed tree
//      s[i] += s[i+m] for m = 16, 8, 4, 2, 1; then + bias[e] (fp32, round to nearest).
//   R2 top-8: sort by (logit descending, expert index ascending); NaN counts as -inf;
//      slot j holds rank j.
//   R3 routing weights: softmax over the 256 logits renormalised over the 8 kept ones,
//      which equals exp(l_j - l_0) / sum_i exp(l_i - l_0) over the kept logits (fp64).
//   R4 group order: within an expert group rows are ordered by ascending token; offsets
//      are exclusive and unpadded; tiles go expert-ascending then row-ascending; experts
//      with no rows get no tile.
//   R5 dequant: w = bf16_rne(scale * q + bias), ONE rounding of the exact value; q is the
//      unsigned code in [0, 15]; code k of a row is the low nibble of byte k/2 for even k
//      and the high nibble for odd k; group of weight k is k / 64.
//   R6 FFN: g = x . Wg_i, u = x . Wu_i, h_i = silu(g) * u with silu(z) = z / (1 + e^-z),
//      y = h . Wd_n, all in fp64; h is NOT rounded (the CUDA path carries h as a bf16
//      pair to 16 bits; see the design notes for why one bf16 rounding cannot meet the
//      elementwise tolerance).
//   R7 combine: out = sum_j w_j * y_j (j ascending) + y_shared, fp64, shared weight 1.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// ---------------------------------------------------------------------------------
// bf16 helpers (decode and round); bf16 values are passed as their 16-bit patterns.
// ---------------------------------------------------------------------------------

static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

static double bf16_to_double(uint16_t b) { return (double)bf16_to_float(b); }

// Round the real number hi + lo to bf16, round-to-nearest-even.  Requires hi = fl64(hi+lo)
// (so |lo| is at most half a double ulp of hi).  neg_zero_hint is the sign IEEE gives an
// exact zero sum (both addends -0).
static uint16_t bf16_round_pair(double hi, double lo, bool neg_zero_hint) {
    if (std::isnan(hi)) return 0x7FC0;
    if (hi == 0.0 && lo == 0.0) return neg_zero_hint ? 0x8000 : 0x0000;
    if (std::isinf(hi)) return hi > 0 ? 0x7F80 : 0xFF80;
    const bool neg = hi < 0;
    double a = std::fabs(hi);
    double l = neg ? -lo : lo;               // correction in the direction of |x|
    int e;
    std::frexp(a, &e);                        // a = m * 2^e, m in [0.5, 1)
    int qexp = e - 8;                         // quantum: 8 significant bits
    if (qexp < -133) qexp = -133;             // bf16 subnormal quantum 2^-133
    double r = std::ldexp(a, -qexp);          // exact (power-of-two scaling)
    double n = std::floor(r);
    double f = r - n;                         // exact
    bool up;
    if (f > 0.5) up = true;
    else if (f < 0.5) up = false;
    else up = (l > 0) || (l == 0 && std::fmod(n, 2.0) != 0.0);   // tie: lo decides, else even
    if (up) n += 1.0;
    double v = std::ldexp(n, qexp);
    if (v > 3.3895313892515355e38) return neg ? 0xFF80 : 0x7F80;  // overflow to inf
    float fv = (float)v;                      // exact: <= 8 significant bits
    uint32_t u;
    std::memcpy(&u, &fv, 4);
    uint16_t b = (uint16_t)(u >> 16);
    return neg ? (uint16_t)(b | 0x8000) : b;
}

uint16_t oracle_bf16_round(double x) { return bf16_round_pair(x, 0.0, std::signbit(x)); }

// R5: one dequantised weight, bf16 bits.
uint16_t oracle_dequant_one(uint16_t scale_bits, uint16_t bias_bits, int q) {
    double s = bf16_to_double(scale_bits), b = bf16_to_double(bias_bits);
    double p = s * (double)q;                 // exact: at most 12 significant bits
    double hi = p + b;                        // TwoSum: hi + lo == p + b exactly
    double bb = hi - p;
    double lo = (p - (hi - bb)) + (b - bb);
    bool negz = std::signbit(p) && std::signbit(b);
    return bf16_round_pair(hi, lo, negz);
}

static inline int code_at(const uint8_t* row, int k) {
    uint8_t byte = row[k >> 1];
    return (k & 1) ? (byte >> 4) : (byte & 0x0F);
}

// Weight (n, k) of one [N, K] Q4 matrix as a double (the bf16 value).
static inline double q4_weight(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                               int K, int n, int k) {
    const uint8_t* row = codes + (size_t)n * (K / 2);
    int g = k / 64;
    size_t gi = (size_t)n * (K / 64) + g;
    return bf16_to_double(oracle_dequant_one(scales[gi], biases[gi], code_at(row, k)));
}

// Dequantise a whole [N, K] Q4 matrix to bf16 bits (pins and ablation references).
void oracle_dequant_matrix(int N, int K, const uint8_t* codes, const uint16_t* scales,
                           const uint16_t* biases, uint16_t* out_bf16) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            const uint8_t* row = codes + (size_t)n * (K / 2);
            size_t gi = (size_t)n * (K / 64) + k / 64;
            out_bf16[(size_t)n * K + k] = oracle_dequant_one(scales[gi], biases[gi], code_at(row, k));
        }
}

// Bytes of one [N, K] Q4 matrix in the checkpoint format: K/2 code bytes per row plus one
// bf16 scale and one bf16 bias per 64 weights (0.5625 bytes per weight).
double oracle_q4_bytes(double N, double K) { return N * (K / 2.0) + N * (K / 64.0) * 4.0; }

// ---------------------------------------------------------------------------------
// R1: router logits, bit-exact fp32 contract.
// ---------------------------------------------------------------------------------
float oracle_router_logit(int d, const uint16_t* x_row, const uint16_t* w_row, const float* bias_e) {
    float p[32];
    for (int l = 0; l < 32; ++l) p[l] = 0.0f;
    for (int i = 0; i < d / 256; ++i)
        for (int l = 0; l < 32; ++l)
            for (int j = 0; j < 8; ++j) {
                int k = 256 * i + 8 * l + j;
                p[l] = std::fmaf(bf16_to_float(x_row[k]), bf16_to_float(w_row[k]), p[l]);
            }
    for (int m = 16; m >= 1; m /= 2)
        for (int i = 0; i < m; ++i) p[i] = p[i] + p[i + m];
    float v = p[0];
    if (bias_e) v = v + *bias_e;
    return v;
}

void oracle_router_logits(int T, int d, int E, const uint16_t* x, const uint16_t* w_router,
                          const float* logit_bias, float* logits) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e)
            logits[(size_t)t * E + e] = oracle_router_logit(d, x + (size_t)t * d, w_router + (size_t)e * d,
                                                            logit_bias ? logit_bias + e : nullptr);
}

// ---------------------------------------------------------------------------------
// R2, R3: top-k and routing weights.
// ---------------------------------------------------------------------------------
void oracle_topk(int T, int E, int k, const float* logits, int32_t* topk_idx, double* topk_w) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float* lg = logits + (size_t)t * E;
        auto key = [&](int e) { float v = lg[e]; return std::isnan(v) ? -INFINITY : v; };
        std::vector<int> order(E);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
            float va = key(a), vb = key(b);
            if (va != vb) return va > vb;
            return a < b;
        });
        double l0 = key(order[0]);
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += std::exp((double)key(order[j]) - l0);
        for (int j = 0; j < k; ++j) {
            topk_idx[(size_t)t * k + j] = order[j];
            topk_w[(size_t)t * k + j] = std::exp((double)key(order[j]) - l0) / den;
        }
    }
}

// ---------------------------------------------------------------------------------
// R4: histogram, exclusive prefix scan, stable scatter, block map.
// tiles is [max_tiles][3] = (expert, first row, rows); returns the number of tiles.
// ---------------------------------------------------------------------------------
int oracle_route_meta(int T, int E, int k, int tile_rows, const int32_t* topk_idx, int32_t* counts,
                      int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* tiles, int max_tiles) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int a = 0; a < T * k; ++a) counts[topk_idx[a]] += 1;            // histogram
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];  // exclusive scan
    std::vector<int32_t> cursor(offsets, offsets + E);
    for (int t = 0; t < T; ++t)                                          // stable scatter
        for (int j = 0; j < k; ++j) {
            int a = t * k + j;
            int p = cursor[topk_idx[a]]++;
            pos[a] = p;
            perm[p] = a;
        }
    int nt = 0;                                                          // block map
    for (int e = 0; e < E; ++e)
        for (int r = 0; r < counts[e]; r += tile_rows) {
            if (nt < max_tiles) {
                tiles[3 * nt + 0] = e;
                tiles[3 * nt + 1] = offsets[e] + r;
                tiles[3 * nt + 2] = std::min(tile_rows, counts[e] - r);
            }
            ++nt;
        }
    return nt;
}

// ---------------------------------------------------------------------------------
// R6, R7: expert FFN and combine.
// ---------------------------------------------------------------------------------
struct oracle_q4 {
    const uint8_t* codes;     // [E][N][K/2]
    const uint16_t* scales;   // [E][N][K/64]
    const uint16_t* biases;   // [E][N][K/64]
};

struct oracle_experts {
    oracle_q4 gate, up, down;  // gate/up: N = I, K = d; down: N = d, K = I
};

static const uint8_t* q4_codes(const oracle_q4& m, int e, int N, int K) { return m.codes + (size_t)e * N * (K / 2); }
static const uint16_t* q4_scales(const oracle_q4& m, int e, int N, int K) { return m.scales + (size_t)e * N * (K / 64); }
static const uint16_t* q4_biases(const oracle_q4& m, int e, int N, int K) { return m.biases + (size_t)e * N * (K / 64); }

static double silu(double z) { return z / (1.0 + std::exp(-z)); }

// y[d] = FFN of expert e on one token row x[d]; h_out[I] optional.
void oracle_expert_ffn(int d, int I, const oracle_experts* W, int e, const uint16_t* x_row, double* y,
                       double* h_out) {
    std::vector<double> h(I);
    const uint8_t* gc = q4_codes(W->gate, e, I, d);
    const uint16_t* gs = q4_scales(W->gate, e, I, d);
    const uint16_t* gb = q4_biases(W->gate, e, I, d);
    const uint8_t* uc = q4_codes(W->up, e, I, d);
    const uint16_t* us = q4_scales(W->up, e, I, d);
    const uint16_t* ub = q4_biases(W->up, e, I, d);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int k = 0; k < d; ++k) {
            double xv = bf16_to_double(x_row[k]);
            g += xv * q4_weight(gc, gs, gb, d, i, k);
            u += xv * q4_weight(uc, us, ub, d, i, k);
        }
        h[i] = silu(g) * u;
        if (h_out) h_out[i] = h[i];
    }
    const uint8_t* dc = q4_codes(W->down, e, d, I);
    const uint16_t* ds = q4_scales(W->down, e, d, I);
    const uint16_t* db = q4_biases(W->down, e, d, I);
    for (int n = 0; n < d; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += h[i] * q4_weight(dc, ds, db, I, n, i);
        y[n] = acc;
    }
}

// out[ntok][d] (fp64) for the tokens listed in tok (indices into x / topk arrays).
void oracle_moe_tokens(int d, int k, int I, int I_shared, const oracle_experts* routed,
                       const oracle_experts* shared, int ntok, const int32_t* tok, const uint16_t* x,
                       const int32_t* topk_idx, const double* topk_w, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int a = 0; a < ntok; ++a) {
        int t = tok[a];
        const uint16_t* xr = x + (size_t)t * d;
        std::vector<double> y(d), acc(d, 0.0);
        for (int j = 0; j < k; ++j) {
            oracle_expert_ffn(d, I, routed, topk_idx[(size_t)t * k + j], xr, y.data(), nullptr);
            double w = topk_w[(size_t)t * k + j];
            for (int n = 0; n < d; ++n) acc[n] += w * y[n];
        }
        if (shared) {
            oracle_expert_ffn(d, I_shared, shared, 0, xr, y.data(), nullptr);
            for (int n = 0; n < d; ++n) acc[n] += y[n];
        }
        std::memcpy(out + (size_t)a * d, acc.data(), sizeof(double) * d);
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

}  // extern "C"
