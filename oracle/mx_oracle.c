/*
 * mx_oracle.c -- plain, slow, fp64 CPU oracle for the fused MXFP4-weight
 * mixture-of-experts layer (route -> permute -> MXFP8 activation quant ->
 * gated FC1 -> SwiGLU -> MXFP8 requant -> FC2 -> top-k weighted combine).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; neither includes the other.
 *
 * Sources of the definitions:
 *  - "[MXFP4 layerwise prefill] SM 8.6 (Ampere) excluded by capability
 *    whitelist" (KTransformers issue 2172), Environment: DeepSeek-V4-Flash
 *    MoE with 256 experts, top-6 routing and native MXFP4 expert weights.
 *  - "Kimi-K3 SM120 FlashInfer MXFP4 MoE", Goal: an MXFP8-activation x
 *    MXFP4-weight fused MoE; on-device evidence: the gated FC1 has twice the
 *    FC2 inter size (256 vs 128 in the official test shape); Phase 0 audit
 *    conclusions, item 4: the SwiGLU gated activation.
 *  - OCP Microscaling Formats (MX) Specification v1.0 (a public standard the
 *    pages name through "MXFP4"/"MXFP8"): e2m1 element values, e8m0 shared
 *    scales, e4m3 (E4M3FN) element values, 32-element blocks, and the
 *    shared-exponent rule X = floor(log2(amax)) - emax_elem.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - e2m1 nibble order: element 2i in bits 0-3 of byte i, element 2i+1 in
 *    bits 4-7.
 *  - routing: experts ordered by (logit descending, index ascending); the
 *    weights are the softmax over the k selected logits (renormalize = 1) or
 *    the full softmax over all E logits taken at the selected experts.
 *  - permutation: rows grouped by expert, stable in slot order s = t*k + j.
 *  - w13 rows [0, I) are the gate projection, rows [I, 2I) the up projection;
 *    SwiGLU h = silu(gate) * up with no clamp, alpha or bias.  As an option,
 *    the gate/up rows interleave (row 2i gate, row 2i+1 up) and the gated
 *    activation is the clamped SwiGLU of GPT-OSS-format checkpoints ("Kimi-K3
 *    SM120 FlashInfer MXFP4 MoE", Phase 0 audit conclusions, item 4, names
 *    that model's SwiGLU weight layout and parameters without stating them;
 *    the definition below is the published GPT-OSS one).
 *  - FC1 accumulators and h are not rounded before the MXFP8 requant.
 *  - the routing weight multiplies the FC2 output (not folded into A2).
 *  - all arithmetic is fp64; the output is rounded once to bf16 (RNE).
 *
 * Every routine is written for clarity, not speed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MXO_OK 0
#define MXO_ERR_ARG (-1)
#define MXO_ERR_SHAPE (-2)
#define MXO_ERR_NAN_SCALE (-3)
#define MXO_ERR_NOMEM (-4)

/* ------------------------------------------------------------------ */
/* Element formats (OCP MX v1.0, element data types and scale type).  */
/* ------------------------------------------------------------------ */

/* e2m1 (FP4): 1 sign bit (bit 3), 2 exponent bits, 1 mantissa bit, bias 1.
 * The eight magnitudes follow from the bit fields: exponent field 0 is the
 * subnormal 0 / 0.5, exponent fields 1..3 give 1.0, 1.5, 2, 3, 4, 6. */
double mxo_e2m1_value(unsigned nibble)
{
    unsigned e = (nibble >> 1) & 3u, m = nibble & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return (nibble & 8u) ? -mag : mag;
}

/* e8m0 shared scale: 2^(s - 127); s = 255 is NaN. */
double mxo_e8m0_value(unsigned s)
{
    if (s == 255u) return NAN;
    return ldexp(1.0, (int)s - 127);
}

/* e4m3 (OCP E4M3FN): bias 7, exponent field 0 is subnormal (m/8 * 2^-6),
 * S.1111.111 is NaN, no infinities; largest finite magnitude 448. */
double mxo_e4m3_value(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* Round-half-to-even of a non-negative value that is an exact double. */
static double rne_nonneg(double v)
{
    double f = floor(v), r = v - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Encode a finite double into e4m3 with round-to-nearest-even and
 * saturation to +-448 (the "satfinite" conversion).  NaN maps to 0x7F.
 * The sign bit is kept, so negative values that round to zero give 0x80. */
unsigned mxo_e4m3_encode(double x)
{
    unsigned sign = signbit(x) ? 0x80u : 0u;
    double a = fabs(x), q;
    int e;
    if (isnan(x)) return 0x7Fu;
    if (a >= 448.0) return sign | 0x7Eu;            /* 1.75 * 2^8 */
    if (a < ldexp(1.0, -6)) {                        /* subnormal grid, step 2^-9 */
        q = rne_nonneg(ldexp(a, 9));                 /* 0..8 (8 == 2^-6, first normal) */
        return sign | (unsigned)q;                   /* code 8 is exponent 1, mantissa 0 */
    }
    frexp(a, &e);                                    /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                          /* a in [2^e, 2^(e+1)) */
    q = rne_nonneg(ldexp(a, 3 - e));                 /* mantissa with implicit 1: 8..16 */
    if (q >= 16.0) { q = 8.0; e += 1; }
    if (e > 8 || (e == 8 && q > 14.0)) return sign | 0x7Eu;
    return sign | ((unsigned)(e + 7) << 3) | ((unsigned)q - 8u);
}

/* Shared exponent of one block: floor(log2(amax)) - emax_elem, clamped to
 * the e8m0 range [-127, 127]; an all-zero block takes -127 (scale byte 0).
 * emax_elem is 8 for e4m3 (448 = 1.75 * 2^8) and 2 for e2m1 (6 = 1.5 * 2^2). */
int mxo_mx_block_exponent(double amax, int emax_elem)
{
    int e, x;
    if (!(amax > 0.0)) return -127;
    frexp(amax, &e);
    x = (e - 1) - emax_elem;
    if (x < -127) x = -127;
    if (x > 127) x = 127;
    return x;
}

/* MXFP8 quantisation of n values (n a multiple of 32): per 32-block the
 * shared scale byte X + 127 and the e4m3 codes of x * 2^-X. */
int mxo_quant_mxfp8(const double* x, int n, uint8_t* codes, uint8_t* scales)
{
    int b, i;
    if (n % 32) return MXO_ERR_SHAPE;
    for (b = 0; b < n / 32; ++b) {
        double amax = 0.0;
        int X;
        for (i = 0; i < 32; ++i) {
            double a = fabs(x[32 * b + i]);
            if (a > amax) amax = a;
        }
        X = mxo_mx_block_exponent(amax, 8);
        scales[b] = (uint8_t)(X + 127);
        for (i = 0; i < 32; ++i) codes[32 * b + i] = (uint8_t)mxo_e4m3_encode(ldexp(x[32 * b + i], -X));
    }
    return MXO_OK;
}

/* bf16 bits -> value (exact). */
double mxo_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* value -> bf16 bits with round-to-nearest-even, computed directly from the
 * double (no intermediate float rounding).  Overflow goes to +-inf. */
uint16_t mxo_bf16_round(double x)
{
    double a = fabs(x), q;
    int e;
    float f;
    uint32_t u;
    if (isnan(x)) return 0x7FC0u;
    if (a == 0.0) return signbit(x) ? 0x8000u : 0u;
    frexp(a, &e);
    e -= 1;                                  /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;                  /* subnormal step 2^-133 */
    q = ldexp(rne_nonneg(ldexp(a, 7 - e)), e - 7);
    if (q >= ldexp(1.0, 128)) q = INFINITY;  /* beyond the largest finite bf16 */
    f = (float)(signbit(x) ? -q : q);        /* exact: q is on the bf16 grid */
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

int mxo_quant_rows_bf16(const uint16_t* x, int rows, int cols, uint8_t* codes, uint8_t* scales)
{
    int r, c, rc = MXO_OK;
    double* buf;
    if (cols % 32) return MXO_ERR_SHAPE;
    buf = (double*)malloc(sizeof(double) * (size_t)(cols > 0 ? cols : 1));
    if (!buf) return MXO_ERR_NOMEM;
    for (r = 0; r < rows && rc == MXO_OK; ++r) {
        for (c = 0; c < cols; ++c) buf[c] = mxo_bf16_value(x[(size_t)r * cols + c]);
        rc = mxo_quant_mxfp8(buf, cols, codes + (size_t)r * cols, scales + (size_t)r * (cols / 32));
    }
    free(buf);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Routing and permutation.                                           */
/* ------------------------------------------------------------------ */

/* Top-k routing of one layer: per token the k experts with the largest
 * logits (ties: lower expert index first), in that order, and their gating
 * weights (softmax over the k selected logits when renormalize != 0, else
 * the full softmax over E evaluated at the selected experts).  fp64, then
 * rounded to f32.  Follows the top-6-of-256 / top-16-of-896 routing that
 * the DeepSeek-V4-Flash (issue 2172, Environment) and Kimi-K3 (Kimi-K3 SM120
 * README, Phase 0 audit table) models use. */
int mxo_route(const float* logits, int T, int E, int k, int renormalize, int32_t* ids, float* w)
{
    int t;
    if (T < 0 || E <= 0 || k <= 0 || k > E) return MXO_ERR_ARG;
    for (t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        char* taken = (char*)calloc((size_t)E, 1);
        double lmax, denom = 0.0;
        int j, e;
        if (!taken) return MXO_ERR_NOMEM;
        for (j = 0; j < k; ++j) {
            int best = -1;
            for (e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: lower index wins ties */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        lmax = (double)l[ids[(size_t)t * k]];
        if (renormalize) {
            for (j = 0; j < k; ++j) denom += exp((double)l[ids[(size_t)t * k + j]] - lmax);
        } else {
            for (e = 0; e < E; ++e) denom += exp((double)l[e] - lmax);
        }
        for (j = 0; j < k; ++j)
            w[(size_t)t * k + j] = (float)(exp((double)l[ids[(size_t)t * k + j]] - lmax) / denom);
        free(taken);
    }
    return MXO_OK;
}

/* Token-to-expert permutation of S = T*k slots (s = t*k + j):
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + count[e]
 *   rank(s)    = #{ s' < s : ids[s'] == ids[s] }        (stable)
 *   p          = offsets[ids[s]] + rank(s); perm[p] = s; inv_perm[s] = p.
 * Slots whose id is outside [0, E) are left out: inv_perm[s] = -1, and the
 * unused tail perm[offsets[E] .. S) is -1.  Returns the number of such
 * slots (>= 0) or a negative error. */
int mxo_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv_perm)
{
    long S = (long)T * k, s;
    int e, bad = 0;
    int32_t* fill;
    if (T < 0 || k <= 0 || E <= 0) return MXO_ERR_ARG;
    fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!fill) return MXO_ERR_NOMEM;
    for (e = 0; e <= E; ++e) offsets[e] = 0;
    for (s = 0; s < S; ++s) {
        int32_t id = ids[s];
        if (id >= 0 && id < E) offsets[id + 1] += 1;
    }
    for (e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    for (s = 0; s < S; ++s) perm[s] = -1;
    for (s = 0; s < S; ++s) {
        int32_t id = ids[s];
        if (id < 0 || id >= E) { inv_perm[s] = -1; ++bad; continue; }
        inv_perm[s] = offsets[id] + fill[id];
        perm[offsets[id] + fill[id]] = (int32_t)s;
        fill[id] += 1;
    }
    free(fill);
    return bad;
}

/* ------------------------------------------------------------------ */
/* Block-scaled dot products.                                         */
/* ------------------------------------------------------------------ */

/* One output of an MXFP8 x MXFP4 contraction over K (K % 32 == 0):
 *   sum_b 2^(sa_b-127) * 2^(sw_b-127) * sum_{i<32} a[32b+i] * w[32b+i]
 * a_val: the e4m3 elements already decoded to doubles, sa: their e8m0
 * bytes; w: packed e2m1 (element 2i low nibble of byte i), sw: e8m0 bytes.
 * fp64; every product and block sum is exact. */
static double dot_mxfp8_mxfp4(const double* a_val, const uint8_t* sa, const uint8_t* w, const uint8_t* sw, int K)
{
    double e2m1[16], acc = 0.0;
    int b, i;
    for (i = 0; i < 16; ++i) e2m1[i] = mxo_e2m1_value((unsigned)i);
    for (b = 0; b < K / 32; ++b) {
        double blk = 0.0;
        for (i = 0; i < 32; ++i) {
            int kk = 32 * b + i;
            unsigned byte = w[kk / 2];
            unsigned nib = (kk & 1) ? (byte >> 4) : (byte & 15u);
            blk += a_val[kk] * e2m1[nib];
        }
        acc += mxo_e8m0_value(sa[b]) * mxo_e8m0_value(sw[b]) * blk;
    }
    return acc;
}

static void decode_e4m3_row(const uint8_t* codes, int n, double* out)
{
    int i;
    for (i = 0; i < n; ++i) out[i] = mxo_e4m3_value(codes[i]);
}

static int scales_finite(const uint8_t* s, size_t n)
{
    size_t i;
    for (i = 0; i < n; ++i)
        if (s[i] == 255u) return 0;
    return 1;
}

/* Plain block-scaled GEMM: out[m, n] = dot(a row m, w row n) over K.
 * a: e4m3 [M, K] + e8m0 [M, K/32]; w: packed e2m1 [N, K/2] + e8m0 [N, K/32]. */
int mxo_gemm_mxfp8_mxfp4(const uint8_t* a, const uint8_t* a_sf, int M, int K,
                         const uint8_t* w, const uint8_t* w_sf, int N, double* out)
{
    int m;
    if (M < 0 || N < 0 || K <= 0 || K % 32) return MXO_ERR_SHAPE;
    if (!scales_finite(a_sf, (size_t)M * (K / 32)) || !scales_finite(w_sf, (size_t)N * (K / 32)))
        return MXO_ERR_NAN_SCALE;
#pragma omp parallel for schedule(dynamic)
    for (m = 0; m < M; ++m) {
        int n;
        double* av = (double*)malloc(sizeof(double) * (size_t)K);
        if (!av) continue;
        decode_e4m3_row(a + (size_t)m * K, K, av);
        for (n = 0; n < N; ++n)
            out[(size_t)m * N + n] = dot_mxfp8_mxfp4(av, a_sf + (size_t)m * (K / 32),
                                                     w + (size_t)n * (K / 2), w_sf + (size_t)n * (K / 32), K);
        free(av);
    }
    return MXO_OK;
}

/* ------------------------------------------------------------------ */
/* The MoE layer.                                                     */
/* ------------------------------------------------------------------ */

/* The gated activation of one FC1 output pair (gate g, up u):
 *   act 0, SwiGLU:          h = silu(g) * u = g / (1 + e^-g) * u
 *   act 1, clamped SwiGLU:  g' = min(g, limit), u' = min(max(u, -limit), limit),
 *                           h = g' / (1 + e^(-alpha g')) * (u' + 1)
 * (for GPT-OSS-format checkpoints alpha = 1.702 and limit = 7).  fp64. */
static double gated_activation(double g, double u, int act, double alpha, double limit)
{
    if (act == 0) return g / (1.0 + exp(-g)) * u;
    if (g > limit) g = limit;
    if (u > limit) u = limit;
    if (u < -limit) u = -limit;
    return g / (1.0 + exp(-alpha * g)) * (u + 1.0);
}

/* Forward of the MoE layer for a list of tokens (each token's output depends
 * only on its own hidden row and routing, so a subset is exact):
 *   a      = MXFP8(hidden[t])                                  (per 32 along H)
 *   acc    = a . w13[e]^T   (2I outputs, block-scaled, fp64)
 *   h      = silu(acc[0:I]) * acc[I:2I]      (or, with gate_up_interleaved,
 *            gate i = acc[2i], up i = acc[2i+1]; act selects the activation,
 *            see gated_activation)
 *   a2     = MXFP8(h)                                          (per 32 along I)
 *   y      = a2 . w2[e]^T   (H outputs)
 *   out[t] = bf16( sum_j topk_w[t, j] * y(t, ids[t, j]) )
 * Shapes: hidden bf16 [T, H]; ids/w [T, k]; w13 [E, 2I, H/2] + [E, 2I, H/32];
 * w2 [E, H, I/2] + [E, H, I/32].  Slots with an id outside [0, E) add
 * nothing.  Optional outputs (NULL to skip), indexed by position in
 * `tokens`: out_f64 [n, H] (before bf16 rounding), a2 [n, k, I] and
 * a2_sf [n, k, I/32] (zero for skipped slots), y [n, k, H]. */
int mxo_moe_forward_tokens_ex(const uint16_t* hidden, int T, int H,
                              const int32_t* ids, const float* topk_w, int k,
                              const uint8_t* w13, const uint8_t* w13_sf,
                              const uint8_t* w2, const uint8_t* w2_sf, int E, int I,
                              const int32_t* tokens, int n_tokens,
                              uint16_t* out, double* out_f64,
                              uint8_t* a2_out, uint8_t* a2_sf_out, double* y_out, int nthreads,
                              int gate_up_interleaved, int act, double alpha, double limit)
{
    int ti, err = MXO_OK;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || n_tokens < 0) return MXO_ERR_ARG;
    if (act != 0 && act != 1) return MXO_ERR_ARG;
    if (H % 32 || I % 32) return MXO_ERR_SHAPE;
    if (!scales_finite(w13_sf, (size_t)E * 2 * I * (H / 32)) || !scales_finite(w2_sf, (size_t)E * H * (I / 32)))
        return MXO_ERR_NAN_SCALE;
    for (ti = 0; ti < n_tokens; ++ti)
        if (tokens[ti] < 0 || tokens[ti] >= T) return MXO_ERR_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic)
    for (ti = 0; ti < n_tokens; ++ti) {
        int t = tokens[ti], j, n, i;
        double* x = (double*)malloc(sizeof(double) * (size_t)H);
        double* acc = (double*)malloc(sizeof(double) * (size_t)2 * I);
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        double* sum = (double*)calloc((size_t)H, sizeof(double));
        double* av = (double*)malloc(sizeof(double) * (size_t)H);
        double* a2v = (double*)malloc(sizeof(double) * (size_t)I);
        uint8_t* a = (uint8_t*)malloc((size_t)H);
        uint8_t* sa = (uint8_t*)malloc((size_t)H / 32);
        uint8_t* a2 = (uint8_t*)malloc((size_t)I);
        uint8_t* sa2 = (uint8_t*)malloc((size_t)I / 32);
        if (!x || !acc || !h || !sum || !av || !a2v || !a || !sa || !a2 || !sa2) {
#pragma omp atomic write
            err = MXO_ERR_NOMEM;
        } else {
            for (i = 0; i < H; ++i) x[i] = mxo_bf16_value(hidden[(size_t)t * H + i]);
            mxo_quant_mxfp8(x, H, a, sa);
            decode_e4m3_row(a, H, av);
            for (j = 0; j < k; ++j) {
                int e = ids[(size_t)t * k + j];
                double wj = (double)topk_w[(size_t)t * k + j];
                if (e < 0 || e >= E) {
                    if (a2_out) memset(a2_out + ((size_t)ti * k + j) * I, 0, (size_t)I);
                    if (a2_sf_out) memset(a2_sf_out + ((size_t)ti * k + j) * (I / 32), 0, (size_t)I / 32);
                    if (y_out)
                        for (n = 0; n < H; ++n) y_out[((size_t)ti * k + j) * H + n] = 0.0;
                    continue;
                }
                for (n = 0; n < 2 * I; ++n) {
                    size_t row = (size_t)e * 2 * I + n;
                    acc[n] = dot_mxfp8_mxfp4(av, sa, w13 + row * (H / 2), w13_sf + row * (H / 32), H);
                }
                for (i = 0; i < I; ++i) {
                    double g, u;
                    if (gate_up_interleaved) { g = acc[2 * i]; u = acc[2 * i + 1]; }
                    else { g = acc[i]; u = acc[I + i]; }
                    h[i] = gated_activation(g, u, act, alpha, limit);
                }
                mxo_quant_mxfp8(h, I, a2, sa2);
                decode_e4m3_row(a2, I, a2v);
                if (a2_out) memcpy(a2_out + ((size_t)ti * k + j) * I, a2, (size_t)I);
                if (a2_sf_out) memcpy(a2_sf_out + ((size_t)ti * k + j) * (I / 32), sa2, (size_t)I / 32);
                for (n = 0; n < H; ++n) {
                    size_t row = (size_t)e * H + n;
                    double y = dot_mxfp8_mxfp4(a2v, sa2, w2 + row * (I / 2), w2_sf + row * (I / 32), I);
                    if (y_out) y_out[((size_t)ti * k + j) * H + n] = y;
                    sum[n] += wj * y;
                }
            }
            for (n = 0; n < H; ++n) {
                if (out_f64) out_f64[(size_t)ti * H + n] = sum[n];
                if (out) out[(size_t)ti * H + n] = mxo_bf16_round(sum[n]);
            }
        }
        free(x); free(acc); free(h); free(sum); free(av); free(a2v); free(a); free(sa); free(a2); free(sa2);
    }
    return err;
}

/* The layer with the default gate | up halves and SwiGLU. */
int mxo_moe_forward_tokens(const uint16_t* hidden, int T, int H,
                           const int32_t* ids, const float* topk_w, int k,
                           const uint8_t* w13, const uint8_t* w13_sf,
                           const uint8_t* w2, const uint8_t* w2_sf, int E, int I,
                           const int32_t* tokens, int n_tokens,
                           uint16_t* out, double* out_f64,
                           uint8_t* a2_out, uint8_t* a2_sf_out, double* y_out, int nthreads)
{
    return mxo_moe_forward_tokens_ex(hidden, T, H, ids, topk_w, k, w13, w13_sf, w2, w2_sf, E, I, tokens, n_tokens,
                                     out, out_f64, a2_out, a2_sf_out, y_out, nthreads, 0, 0, 0.0, 0.0);
}

int mxo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
