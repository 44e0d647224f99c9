/*
 * CPU oracle for the block-quantized-weight matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Arithmetic: dequantized weights in f32 (exact by construction), products
 * and sums in f64 in k order, one final rounding to the output type.
 *
 * Sources (pages of the reference material, by title and section):
 *  - Q4 split-plane format: "oxinfer 0.0.5 src/metal.rs", shader section
 *    "Dequantizers" (struct Q4W, nib_lo / nib_hi and load(Q4W ...)): block b
 *    of row n is 16 bytes at n*K/2 + 16*b; byte i holds element i in its low
 *    nibble and element 16+i in its high nibble; value = (nibble - 8) * d,
 *    d the fp16 block scale at n*(K/32) + b.  The same order is restated by
 *    the GGUF Q4_0 decoder on the same page (load(Q4_0W ...)).
 *  - Q8-row format: "cortiq-engine 0.8.3 src/gpu_metal/qi21.rs", module
 *    header (q8_row: int8 weights, row scale on the f32 result).
 *  - GEMM reference shape (dequantize, then an f64 dot product per output):
 *    "oxinfer 0.0.5 src/metal.rs", tests module, functions dense / matvec.
 *  - MoE chain (per token and routed expert: gate/up, SiLU(g)*u, down, the
 *    weighted sum): same tests module, mma_moe_matches_cpu; SiLU as
 *    g/(1+exp(-g)) from the silu_half shader.  Expert-major grouping of the
 *    routed rows, token order inside an expert: same page, Backend::moe.
 *  - Format variants: Q8 per 32-k block and affine Q4 from the same
 *    "Dequantizers" section (load(Q8W ...), load(Q4A ...)); q8_2f from
 *    "cortiq-engine 0.8.3 src/gpu_metal/qi21.rs" (module header, fn build_block).
 *  - Routing from router logits (top-k, lower index first on ties, weights
 *    renormalised over the picked experts; the shared expert's sigmoid gate):
 *    "cortiq-engine 0.8.44 src/clover.rs" (moe_route, the route closure) and
 *    "cortiq-engine 0.8.41 src/gpu_metal/clover.rs", fn run_on.
 *  - Dense FFN chain (gate/up, SwiGLU, down for every token): "cortiq-engine
 *    0.8.3 src/gpu_metal/qi21.rs", fn blocks (gemm(TG, TU) -> swiglu ->
 *    gemm(TD)) and its module header.
 *
 * Every function is single-purpose; the only parallelism is OpenMP over
 * independent outputs, which leaves each output's arithmetic unchanged.
 *
 * Pins (tests marked "not gpu"): hand-built blocks for the dequantizers,
 * exact rational brute force and a library f64 matmul for the GEMM, closed
 * forms and invariants for the MoE chain and the layout, a one-hot closed
 * form, library matmuls and the one-expert MoE chain for the dense FFN,
 * a stable library argsort and closed-form weights for the routing,
 * reductions to the pinned formats, library f32 arithmetic and exact
 * rationals for the format variants.  No function here
 * is left without a pin.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- number formats, from the IEEE 754 binary16 and bfloat16 definitions ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Subnormals are fraction * 2^-24; exponent 31 is inf/NaN. */
double or_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of a binary32. */
double or_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round an f64 to bfloat16 once, to nearest with ties to even.
 * bfloat16 keeps 8 significant bits, the smallest normal is 2^-126 and the
 * subnormal quantum 2^-133. */
uint16_t or_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);                      /* a = m * 2^e, m in [0.5, 1) */
    int qexp = e - 8;                  /* weight of the last kept bit */
    if (qexp < -133) qexp = -133;
    double r = nearbyint(ldexp(a, -qexp));   /* default mode: ties to even */
    double v = ldexp(r, qexp);
    if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)v;                /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)(u >> 16);
}

void or_f64_to_bf16_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_f64_to_bf16(x[i]);
}

void or_f64_to_f32_array(const double* x, int64_t n, float* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (float)x[i];   /* RNE in the default mode */
}

/* X as stored (fp16 or bf16 bits) -> f64, exact. */
void or_x_to_f64(const uint16_t* x, int is_bf16, int64_t n, double* out) {
    for (int64_t i = 0; i < n; i++) out[i] = is_bf16 ? or_bf16_to_f64(x[i]) : or_f16_to_f64(x[i]);
}

/* ---- Q4 packing and dequantization ---- */

/* codes[N][K] (0..15) -> Wq[N][K/2]: byte 16b+i of row n holds
 * codes[n][32b+i] in its low nibble and codes[n][32b+16+i] in its high one. */
void or_pack_q4(const uint8_t* codes, int64_t N, int64_t K, uint8_t* wq) {
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < K / 32; b++)
            for (int i = 0; i < 16; i++) {
                uint8_t lo = codes[n * K + 32 * b + i] & 15;
                uint8_t hi = codes[n * K + 32 * b + 16 + i] & 15;
                wq[n * (K / 2) + 16 * b + i] = (uint8_t)(lo | (hi << 4));
            }
}

/* W[n][32b+i] = (lo(byte) - 8) * d, W[n][32b+16+i] = (hi(byte) - 8) * d,
 * d = f32(fp16 scale).  The f32 product of a 4-bit integer and an 11-bit
 * significand is exact, so W is exact (the sign of zero follows IEEE). */
void or_dequant_q4(const uint8_t* wq, const uint16_t* ws, int64_t N, int64_t K, float* w) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < K / 32; b++) {
            float d = (float)or_f16_to_f64(ws[n * (K / 32) + b]);
            for (int i = 0; i < 16; i++) {
                uint8_t byte = wq[n * (K / 2) + 16 * b + i];
                w[n * K + 32 * b + i] = (float)((int)(byte & 15) - 8) * d;
                w[n * K + 32 * b + 16 + i] = (float)((int)(byte >> 4) - 8) * d;
            }
        }
}

/* Q8-row as a dense f32 matrix: W[n][k] = (float)q[n][k] * rs[n] (one f32
 * rounding).  The GEMM below uses the unscaled integers and applies rs to
 * the f64 sum instead, which is the format's own statement (row scale on
 * the result). */
void or_dequant_q8row(const int8_t* wq, const float* rs, int64_t N, int64_t K, float* w) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) w[n * K + k] = (float)wq[n * K + k] * rs[n];
}

/* ---- GEMM ---- */

/* Y[t][n] = sum_k W[n][k] * X[t][k] in f64, k ascending.  S[t][n] is the
 * error-bound denominator sum_k |W[n][k] * X[t][k]|.  W[N][K] f32, X[T][K]
 * f64 (the exact stored activations).  rowscale (nullable) multiplies each
 * output row n's sums (Q8-row). */
void or_gemm(const float* W, const double* X, int64_t T, int64_t N, int64_t K,
             const float* rowscale, double* Y, double* S) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < T; t++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0, abs_acc = 0.0;
            const float* wr = W + n * K;
            const double* xr = X + t * K;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)wr[k] * xr[k];
                acc += p;
                abs_acc += fabs(p);
            }
            double r = rowscale ? (double)rowscale[n] : 1.0;
            Y[t * N + n] = acc * r;
            if (S) S[t * N + n] = abs_acc * fabs(r);
        }
}

/* The same sums for a list of (t, n) output positions only. */
void or_gemm_sampled(const float* W, const double* X, int64_t N, int64_t K,
                     const float* rowscale, const int64_t* tn, int64_t count, double* Y, double* S) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; i++) {
        int64_t t = tn[2 * i], n = tn[2 * i + 1];
        double acc = 0.0, abs_acc = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double p = (double)W[n * K + k] * X[t * K + k];
            acc += p;
            abs_acc += fabs(p);
        }
        double r = rowscale ? (double)rowscale[n] : 1.0;
        (void)N;
        Y[i] = acc * r;
        S[i] = abs_acc * fabs(r);
    }
}

/* Q4 GEMM on packed rows, for sampled outputs at full size: dequantizes
 * only the rows it needs, one at a time (same arithmetic as or_dequant_q4
 * followed by or_gemm_sampled). */
void or_gemm_q4_sampled(const uint8_t* wq, const uint16_t* ws, const double* X, int64_t N, int64_t K,
                        const int64_t* tn, int64_t count, double* Y, double* S) {
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < count; i++) {
            int64_t t = tn[2 * i], n = tn[2 * i + 1];
            or_dequant_q4(wq + n * (K / 2), ws + n * (K / 32), 1, K, row);
            double acc = 0.0, abs_acc = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)row[k] * X[t * K + k];
                acc += p;
                abs_acc += fabs(p);
            }
            Y[i] = acc;
            S[i] = abs_acc;
        }
        free(row);
    }
    (void)N;
}

void or_gemm_q8_sampled(const int8_t* wq, const float* rs, const double* X, int64_t N, int64_t K,
                        const int64_t* tn, int64_t count, double* Y, double* S) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; i++) {
        int64_t t = tn[2 * i], n = tn[2 * i + 1];
        double acc = 0.0, abs_acc = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double p = (double)wq[n * K + k] * X[t * K + k];
            acc += p;
            abs_acc += fabs(p);
        }
        Y[i] = acc * (double)rs[n];
        S[i] = abs_acc * fabs((double)rs[n]);
    }
    (void)N;
}

/* ---- MoE expert panels ---- */

/* Routed (t, j) pairs grouped by expert: seg[e] = number of pairs routed to
 * experts below e (seg[E] = T*topk), and perm lists pair ids p = t*topk + j
 * sorted by (expert, t, j).  Returns -1 if an index is out of range. */
int or_moe_layout(const int32_t* idx, int64_t T, int64_t topk, int64_t E, int32_t* perm, int32_t* seg) {
    int64_t P = T * topk;
    int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t p = 0; p < P; p++) {
        if (idx[p] < 0 || idx[p] >= E) { free(count); return -1; }
        count[idx[p]]++;
    }
    seg[0] = 0;
    for (int64_t e = 0; e < E; e++) seg[e + 1] = seg[e] + (int32_t)count[e];
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t p = 0; p < P; p++) {          /* pairs in (t, j) order: stable */
        int32_t e = idx[p];
        perm[seg[e] + fill[e]] = (int32_t)p;
        fill[e]++;
    }
    free(count);
    free(fill);
    return 0;
}

/* One routed pair: o = Wd[e] . (silu(Wgate[e] . x) * (Wup[e] . x)), all f64.
 * wgu[2I][H] f32 (rows 0..I-1 gate, I..2I-1 up), wd[H][I] f32, x[H] f64.
 * a_out[I] (nullable) receives the SwiGLU activation; o[H], sabs[H] the
 * expert output and sum_k |Wd[n][k] * a[k]|. */
void or_moe_pair(const float* wgu, const float* wd, const double* x, int64_t H, int64_t I,
                 double* a_out, double* o, double* sabs) {
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    for (int64_t i = 0; i < I; i++) {
        double g = 0.0, u = 0.0;
        for (int64_t k = 0; k < H; k++) g += (double)wgu[i * H + k] * x[k];
        for (int64_t k = 0; k < H; k++) u += (double)wgu[(I + i) * H + k] * x[k];
        a[i] = g / (1.0 + exp(-g)) * u;
        if (a_out) a_out[i] = a[i];
    }
    for (int64_t n = 0; n < H; n++) {
        double acc = 0.0, abs_acc = 0.0;
        for (int64_t k = 0; k < I; k++) {
            double p = (double)wd[n * I + k] * a[k];
            acc += p;
            abs_acc += fabs(p);
        }
        o[n] = acc;
        sabs[n] = abs_acc;
    }
    free(a);
}

/* Full MoE output: Y[t] = sum_j w[t][j] * o(t, j), j ascending, and the
 * bound S[t] = sum_j |w[t][j]| * sabs(t, j).  Experts' dequantized weights
 * are looked up per pair from the packed planes (only touched experts are
 * decoded).  X[T][H] f64.  Returns -1 on an out-of-range index. */
int or_moe(const double* X, int64_t T, int64_t H, int64_t E, int64_t I, int64_t topk,
           const int32_t* idx, const float* w,
           const uint8_t* gu_q, const uint16_t* gu_s, const uint8_t* d_q, const uint16_t* d_s,
           double* Y, double* S) {
    for (int64_t p = 0; p < T * topk; p++)
        if (idx[p] < 0 || idx[p] >= E) return -1;
    /* decode each touched expert once */
    float** gu = (float**)calloc((size_t)E, sizeof(float*));
    float** dn = (float**)calloc((size_t)E, sizeof(float*));
    for (int64_t p = 0; p < T * topk; p++) {
        int64_t e = idx[p];
        if (gu[e]) continue;
        gu[e] = (float*)malloc(sizeof(float) * (size_t)(2 * I * H));
        dn[e] = (float*)malloc(sizeof(float) * (size_t)(H * I));
        or_dequant_q4(gu_q + e * (2 * I) * (H / 2), gu_s + e * (2 * I) * (H / 32), 2 * I, H, gu[e]);
        or_dequant_q4(d_q + e * H * (I / 2), d_s + e * H * (I / 32), H, I, dn[e]);
    }
    double* o = (double*)malloc(sizeof(double) * (size_t)(T * topk * H));
    double* sa = (double*)malloc(sizeof(double) * (size_t)(T * topk * H));
#pragma omp parallel for schedule(dynamic)
    for (int64_t p = 0; p < T * topk; p++) {
        int64_t t = p / topk, e = idx[p];
        or_moe_pair(gu[e], dn[e], X + t * H, H, I, NULL, o + p * H, sa + p * H);
    }
    for (int64_t t = 0; t < T; t++)
        for (int64_t n = 0; n < H; n++) {
            double y = 0.0, s = 0.0;
            for (int64_t j = 0; j < topk; j++) {
                int64_t p = t * topk + j;
                y += (double)w[p] * o[p * H + n];
                s += fabs((double)w[p]) * sa[p * H + n];
            }
            Y[t * H + n] = y;
            S[t * H + n] = s;
        }
    for (int64_t e = 0; e < E; e++) { free(gu[e]); free(dn[e]); }
    free(gu); free(dn); free(o); free(sa);
    return 0;
}

/* ---- dense FFN chain (gate/up -> SwiGLU -> down) ---- */

/* For every token t of X[T][H] (f64):
 *   g_i = sum_k Wg[i][k] x_k,  u_i = sum_k Wu[i][k] x_k       (i < I; f64, k ascending)
 *   a_i = g_i / (1 + exp(-g_i)) * u_i                          (f64)
 *   Y[t][n] = sum_i Wd[n][i] a_i,  S[t][n] = sum_i |Wd[n][i] a_i|
 * with Wgu[2I][H] the dequantized gate|up rows (gate 0..I-1, up I..2I-1) and
 * Wd[H][I], both Q4.  This is one routed pair of the MoE chain with weight 1
 * applied to every token: the denoiser block's GEMM chain gemm(TG, TU) ->
 * swiglu -> gemm(TD) ("cortiq-engine 0.8.3 src/gpu_metal/qi21.rs", fn blocks
 * and its module header).  A_out (nullable, [T][I]) receives a. */
void or_ffn(const double* X, int64_t T, int64_t H, int64_t I,
            const uint8_t* gu_q, const uint16_t* gu_s, const uint8_t* d_q, const uint16_t* d_s,
            double* Y, double* S, double* A_out) {
    float* wgu = (float*)malloc(sizeof(float) * (size_t)(2 * I * H));
    float* wd = (float*)malloc(sizeof(float) * (size_t)(H * I));
    or_dequant_q4(gu_q, gu_s, 2 * I, H, wgu);
    or_dequant_q4(d_q, d_s, H, I, wd);
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic)
        for (int64_t t = 0; t < T; t++) {
            const double* x = X + t * H;
            for (int64_t i = 0; i < I; i++) {
                double g = 0.0, u = 0.0;
                for (int64_t k = 0; k < H; k++) g += (double)wgu[i * H + k] * x[k];
                for (int64_t k = 0; k < H; k++) u += (double)wgu[(I + i) * H + k] * x[k];
                a[i] = g / (1.0 + exp(-g)) * u;
                if (A_out) A_out[t * I + i] = a[i];
            }
            for (int64_t n = 0; n < H; n++) {
                double acc = 0.0, abs_acc = 0.0;
                for (int64_t i = 0; i < I; i++) {
                    double p = (double)wd[n * I + i] * a[i];
                    acc += p;
                    abs_acc += fabs(p);
                }
                Y[t * H + n] = acc;
                S[t * H + n] = abs_acc;
            }
        }
        free(a);
    }
    free(wgu);
    free(wd);
}

/* ---- MoE routing from router logits ---- */

/* Per token t with logits l[0..E) (f32; one more, l[E], the shared expert's
 * gate logit when `shared`):
 *   - the top-k experts by logit, descending, the lower index first on ties
 *     (picked one at a time: the largest logit not yet picked, lowest index
 *     among equals), which is the top-k by softmax probability since exp is
 *     strictly increasing;
 *   - p_e = exp(l_e - max l) / sum_e' exp(l_e' - max l) in f64, and
 *     w_j = p_{e_j} / sum_{j'} p_{e_j'} over the picked experts, rounded to f32;
 *   - with `shared`, slot topk is the shared expert (index E) with weight
 *     1 / (1 + exp(-l[E])) (f64, rounded to f32).
 * ("cortiq-engine 0.8.44 src/clover.rs": the coreset's top-k comment
 * (descending, lower index first on ties), moe_route and the route closure
 * (p[e] / wsum); "cortiq-engine 0.8.41 src/gpu_metal/clover.rs", fn run_on:
 * the shared expert's slot appended after the routed ones with weight
 * 1 / (1 + exp(-sg)).)  idx[T][topk + shared], w[T][topk + shared]. */
void or_route(const float* logits, int64_t T, int64_t E, int64_t topk, int shared, int32_t* idx, float* w) {
    const int64_t ld = E + (shared ? 1 : 0), slots = topk + (shared ? 1 : 0);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    for (int64_t t = 0; t < T; t++) {
        const float* l = logits + t * ld;
        double mx = -INFINITY;
        for (int64_t e = 0; e < E; e++) if ((double)l[e] > mx) mx = (double)l[e];
        double sum = 0.0;
        for (int64_t e = 0; e < E; e++) sum += exp((double)l[e] - mx);
        memset(taken, 0, (size_t)E);
        double wsum = 0.0;
        double p[64];
        for (int64_t j = 0; j < topk; j++) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;   /* strict: the lower index wins ties */
            taken[best] = 1;
            idx[t * slots + j] = (int32_t)best;
            p[j] = exp((double)l[best] - mx) / sum;
            wsum += p[j];
        }
        for (int64_t j = 0; j < topk; j++) w[t * slots + j] = (float)(p[j] / wsum);
        if (shared) {
            idx[t * slots + topk] = (int32_t)E;
            w[t * slots + topk] = (float)(1.0 / (1.0 + exp(-(double)l[E])));
        }
    }
    free(taken);
}

/* ---- format variants ---- */

/* Q8 per 32-k block ("oxinfer 0.0.5 src/metal.rs", Dequantizers, struct Q8W
 * and load(Q8W ...)): int8 q[N][K], f32 scale s[N][K/32];
 * W[n][k] = f32(q[n][k]) * s[n][k/32] (one f32 rounding). */
void or_dequant_q8b(const int8_t* q, const float* s, int64_t N, int64_t K, float* w) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) w[n * K + k] = (float)q[n * K + k] * s[n * (K / 32) + k / 32];
}

/* Affine Q4 ("oxinfer 0.0.5 src/metal.rs", Dequantizers, struct Q4A and
 * load(Q4A ...)): the Q4 split-plane element (nibble - 8) * d (exact in f32)
 * plus the bf16 offset of its group of gk blocks, off[n][b / gk] (gpr = K/32/gk
 * offsets per row), added in f32 (one rounding). */
static float or_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
void or_dequant_q4a(const uint8_t* wq, const uint16_t* ws, const uint16_t* off, int64_t gk, int64_t N, int64_t K,
                    float* w) {
    const int64_t gpr = K / 32 / gk;
    or_dequant_q4(wq, ws, N, K, w);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) w[n * K + k] = w[n * K + k] + or_bf16_to_f32(off[n * gpr + (k / 32) / gk]);
}

/* q8_2f ("cortiq-engine 0.8.3 src/gpu_metal/qi21.rs", module header: int8
 * weights staged times the column field, the row scale in the epilogue; the
 * blob layout q[rows][cols], rs[rows], col[cols] from fn build_block):
 *   Y[t][n] = rs[n] * sum_k q[n][k] * col[k] * X[t][k]   (f64, k ascending),
 *   S[t][n] = |rs[n]| * sum_k |q[n][k] * col[k] * X[t][k]|.
 * rs and col as f32 (the stored f16 values widened exactly). */
void or_gemm_q8_2f(const int8_t* q, const float* rs, const float* col, const double* X, int64_t T, int64_t N,
                   int64_t K, double* Y, double* S) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < T; t++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0, abs_acc = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)q[n * K + k] * (double)col[k] * X[t * K + k];
                acc += p;
                abs_acc += fabs(p);
            }
            Y[t * N + n] = acc * (double)rs[n];
            S[t * N + n] = abs_acc * fabs((double)rs[n]);
        }
}
