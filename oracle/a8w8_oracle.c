/*
 * a8w8_oracle.c -- plain CPU oracle for the Qwen3-14B-shaped A8W8 decode layer
 * and decode step.
 *
 * TEST INFRASTRUCTURE. This file is the slow, obviously correct restatement of
 * what the decode path computes. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may build, load or call it. The CUDA path
 * shares no code, header, table or helper with it; the two meet only through
 * the seeded inputs both are given.
 *
 * Sources, cited by page title and section:
 *   [LIB-810]   "perf(qwen3-a8w8): optimize decode scheduling and data paths"
 *               (pypto-lib PR #810): sections "Decode scheduling",
 *               "Gate/Up INT8 path", "BF16 KV cache", "Validation", and the
 *               review's "Changes" table.
 *   [SRV-48]    "Add native Qwen3 14B A8W8 serving path" (pypto-serving PR #48):
 *               loader review (scale broadcast over output channels), "Summary"
 *               (physical decode batch 16), "Performance" test settings.
 *   [SRV-52]    "[Feature] Add native Qwen3-14B A8W8 serving path"
 *               (pypto-serving issue #52): "Current behavior" (fused QK norm +
 *               Q RoPE), "Measurement basis" (gate/up/silu/down MLP).
 *   [SRV-61]    "Add Qwen3 A8W8 L2 runner foundation" (pypto-serving PR #61):
 *               "Summary" (block-table / slot-mapping packing, padded decode
 *               rows, host-side KV bounds validation).
 * Where the pages are silent the plain reading is taken and marked "reading:".
 *
 * Precision: the pages fix FP32 for the dequantisation (activation scale times
 * weight scale, FP32 partials of the split down projection) and RNE for every
 * FP32->BF16 narrowing; those steps run here in float with IEEE semantics
 * (compile with -ffp-contract=off, never -ffast-math). Every other floating
 * point step (norms, RoPE, softmax attention, SiLU, LM head) runs in double
 * and is narrowed to BF16 once. Integer dot products are exact.
 *
 * Parity status of each function is stated in its comment; "pinned" names the
 * independent checks in the test suite that hold it in place.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* BF16 representation                                                       */
/* ------------------------------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32; widening is exact. */
double or_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double straight to BF16 with round-to-nearest-even ([LIB-810]
 * "Validation": every FP32->BF16 narrowing uses RNE). The value is scaled by
 * the BF16 unit in the last place at its binade, rounded to an integer with
 * ties to even (nearbyint in the default rounding mode), and scaled back; the
 * result is exactly representable, so the final float conversion is exact.
 * Rounding straight from double avoids a double rounding through float.
 * Pinned: hand-checked ties, overflow to infinity, signed zero, and agreement
 * with the bit-level float32 RNE rule on random floats (tests). */
uint16_t or_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    if (x == 0.0)
        return signbit(x) ? 0x8000 : 0x0000;
    if (isinf(x))
        return signbit(x) ? 0xFF80 : 0x7F80;
    int e;
    frexp(fabs(x), &e);           /* |x| = m * 2^e, m in [0.5, 1) */
    int lead = e - 1;             /* weight of the leading bit */
    if (lead < -126)
        lead = -126;              /* BF16 subnormals share float's exponent floor */
    double ulp = ldexp(1.0, lead - 7);   /* 8 significant bits */
    double r = nearbyint(x / ulp) * ulp;
    const double bf16_max = 3.3895313892515355e38; /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max)
        return signbit(x) ? 0xFF80 : 0x7F80;
    float f = (float)r;           /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void or_bf16_from_double_array(const double* x, long n, uint16_t* y)
{
    for (long i = 0; i < n; ++i)
        y[i] = or_bf16_from_double(x[i]);
}

/* ------------------------------------------------------------------------- */
/* a2 / a11 / a5: RMSNorm                                                     */
/* ------------------------------------------------------------------------- */

/* y = bf16( x * 1/sqrt(mean(x^2) + eps) * w ), one row at a time.
 * The pages name an input RMSNorm and a post-attention RMSNorm feeding the
 * quantiser ([LIB-810] "Gate/Up INT8 path": "post-attention RMSNorm
 * activations"; review sequence diagram). Reading: the mean of squares and the
 * products run in double, and the result is narrowed to BF16 once.
 * Pinned: constant rows (closed form), scale invariance, brute force. */
void or_rmsnorm(const uint16_t* x, const uint16_t* w, int rows, int cols,
                double eps, uint16_t* y)
{
    for (int r = 0; r < rows; ++r) {
        const uint16_t* xr = x + (long)r * cols;
        double ss = 0.0;
        for (int c = 0; c < cols; ++c) {
            double v = or_bf16_to_double(xr[c]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / cols + eps);
        for (int c = 0; c < cols; ++c)
            y[(long)r * cols + c] =
                or_bf16_from_double(or_bf16_to_double(xr[c]) * inv * or_bf16_to_double(w[c]));
    }
}

/* ------------------------------------------------------------------------- */
/* a3 / a9 / a11 / a13: per-row dynamic symmetric INT8 quantisation          */
/* ------------------------------------------------------------------------- */

/* [LIB-810] "Decode scheduling" (activation quantisation batched across
 * decode rows) and "Gate/Up INT8 path" (activations quantised dynamically
 * "once per row"). Reading of the formula: scale s = absmax / 127 as an IEEE
 * float32 division; q = clamp(rne(x / s), -127, 127) with x / s an IEEE
 * float32 division and ties to even; an all-zero row gives s = 0 and q = 0.
 * -128 is never produced. The input is the BF16 row.
 * Pinned: hand cases in tests/golden/quant_cases.txt, a numpy float32
 * restatement bit for bit, and invariants (|q| <= 127, the absmax element maps
 * to +-127). */
void or_quant_rows(const uint16_t* x, int rows, int cols, int8_t* q, float* scale)
{
    for (int r = 0; r < rows; ++r) {
        const uint16_t* xr = x + (long)r * cols;
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            float a = fabsf(bf16_to_float(xr[c]));
            if (a > amax)
                amax = a;
        }
        float s = amax / 127.0f;
        scale[r] = s;
        for (int c = 0; c < cols; ++c) {
            int8_t v = 0;
            if (s != 0.0f) {
                float t = bf16_to_float(xr[c]) / s;
                float rr = rintf(t);      /* ties to even */
                if (rr > 127.0f)
                    rr = 127.0f;
                if (rr < -127.0f)
                    rr = -127.0f;
                v = (int8_t)rr;
            }
            q[(long)r * cols + c] = v;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* a4 / a10 / a12 / a14: INT8 x INT8 -> INT32 accumulation                    */
/* ------------------------------------------------------------------------- */

/* acc[m][n] = sum over k in [k_begin, k_end) of x[m][k] * W[n][k], exactly.
 * [LIB-810] "Gate/Up INT8 path": INT8 x INT8 -> INT32 matmuls. W is [N, K]
 * row-major (one row per output channel). Accumulates in int64 and reports an
 * overflow of the int32 range through the return value (1 = overflow).
 * Pinned: numpy int64 brute force, split additivity. */
int or_matmul_i8(const int8_t* x, int M, int K, const int8_t* W, int N,
                 int k_begin, int k_end, int32_t* acc)
{
    int overflow = 0;
    for (int m = 0; m < M; ++m) {
        const int8_t* xr = x + (long)m * K;
#pragma omp parallel for schedule(static) reduction(| : overflow)
        for (int n = 0; n < N; ++n) {
            const int8_t* wr = W + (long)n * K;
            int64_t s = 0;
            for (int k = k_begin; k < k_end; ++k)
                s += (int64_t)xr[k] * (int64_t)wr[k];
            if (s > INT32_MAX || s < INT32_MIN)
                overflow = 1;
            acc[(long)m * N + n] = (int32_t)s;
        }
    }
    return overflow;
}

/* Dequantisation in FP32: (float(acc) * s_act) * s_w[n]. [LIB-810] "Gate/Up
 * INT8 path" (activation and weight scales applied during dequantisation) and
 * the review's "Changes" table (FP32 dequantisation scales). Weight scales are
 * per output channel ([SRV-48] loader review: the scale broadcasts over output
 * channels). Reading: the activation scale is applied first. */
float or_dequant(int32_t acc, float s_act, float s_w)
{
    float a = (float)acc;
    float p = a * s_act;
    return p * s_w;
}

/* y[m][n] = bf16( ((p_0 + p_1) + ... + p_{S-1}) + f32(residual[m][n]) ), where
 * p_j is the FP32 dequantisation of the INT32 accumulator over the j-th of S
 * equal contiguous K ranges. S = 1 is a plain projection; S = 2 with a
 * residual is the split down projection of [LIB-810] "Decode scheduling"
 * (two-way K parallelism with independent partial accumulators) and the
 * review's "Changes" table (FP32 partials accumulated, then cast with the
 * residual). Reading: the O projection adds its residual the same way.
 * acc_out (nullable) receives the full-K INT32 sum of the split accumulators.
 * Returns 0, or -1 if K is not a multiple of S, or 1 on int32 overflow. */
int or_linear(const int8_t* xq, const float* xs, int M, int K, const int8_t* W,
              const float* ws, int N, int k_splits, const uint16_t* residual,
              uint16_t* y, int32_t* acc_out)
{
    if (k_splits < 1 || K % k_splits != 0)
        return -1;
    int kc = K / k_splits;
    int32_t* part = (int32_t*)malloc(sizeof(int32_t) * (size_t)M * N * k_splits);
    int overflow = 0;
    for (int j = 0; j < k_splits; ++j)
        overflow |= or_matmul_i8(xq, M, K, W, N, j * kc, (j + 1) * kc,
                                 part + (size_t)j * M * N);
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            float sum = 0.0f;
            int64_t full = 0;
            for (int j = 0; j < k_splits; ++j) {
                int32_t a = part[(size_t)j * M * N + (size_t)m * N + n];
                float p = or_dequant(a, xs[m], ws[n]);
                sum = (j == 0) ? p : sum + p;
                full += a;
            }
            if (residual)
                sum = sum + bf16_to_float(residual[(size_t)m * N + n]);
            y[(size_t)m * N + n] = or_bf16_from_double((double)sum);
            if (acc_out)
                acc_out[(size_t)m * N + n] = (int32_t)full;
        }
    }
    free(part);
    return overflow;
}

/* a12: fused Gate/Up with SwiGLU. W_gu is [2I, K]: rows [0, I) are the gate
 * channels and rows [I, 2I) the up channels. g and u are FP32 dequantised
 * values that are not narrowed; act = bf16( silu(g) * u ) with
 * silu(g) = g / (1 + exp(-g)) in double. [LIB-810] "Gate/Up INT8 path"
 * (native INT8 gate/up, scales applied during dequantisation) and [SRV-52]
 * "Measurement basis" (the gate/up/silu/down MLP). acc_out (nullable) gets the
 * [M, 2I] INT32 accumulators. Pinned: silu(0) = 0 and silu(x) -> x for large x
 * through the closed-form tests, INT32 by brute force. */
int or_gate_up_swiglu(const int8_t* xq, const float* xs, int M, int K,
                      const int8_t* W_gu, const float* s_gu, int I,
                      uint16_t* act, int32_t* acc_out)
{
    int32_t* acc = (int32_t*)malloc(sizeof(int32_t) * (size_t)M * 2 * I);
    int overflow = or_matmul_i8(xq, M, K, W_gu, 2 * I, 0, K, acc);
    for (int m = 0; m < M; ++m) {
        for (int j = 0; j < I; ++j) {
            float g = or_dequant(acc[(size_t)m * 2 * I + j], xs[m], s_gu[j]);
            float u = or_dequant(acc[(size_t)m * 2 * I + I + j], xs[m], s_gu[I + j]);
            double gd = g, ud = u;
            double silu = gd / (1.0 + exp(-gd));
            act[(size_t)m * I + j] = or_bf16_from_double(silu * ud);
        }
    }
    if (acc_out)
        memcpy(acc_out, acc, sizeof(int32_t) * (size_t)M * 2 * I);
    free(acc);
    return overflow;
}

/* ------------------------------------------------------------------------- */
/* a6: rotary position embedding                                              */
/* ------------------------------------------------------------------------- */

/* Rotate-half RoPE over each [D] head vector of x (in place), in double:
 * for i < D/2, angle = pos * theta^(-2i/D),
 *   y[i]       = x[i] cos - x[i + D/2] sin
 *   y[i + D/2] = x[i + D/2] cos + x[i] sin,
 * narrowed to BF16 once. [SRV-52] "Current behavior" names the Q RoPE of the
 * fused QK-norm path; reading: the Qwen3 rotate-half form. pos[r] is the
 * position of row r (rows = tokens x heads, heads_per_token rows per token).
 * Pinned: position 0 is the identity, norms are preserved, and
 * <R_m q, R_n k> depends on m - n only (tests). */
void or_rope(uint16_t* x, int tokens, int heads, int D, const int32_t* pos,
             double theta)
{
    int half = D / 2;
    for (int t = 0; t < tokens; ++t) {
        double p = (double)pos[t];
        for (int h = 0; h < heads; ++h) {
            uint16_t* v = x + ((long)t * heads + h) * D;
            for (int i = 0; i < half; ++i) {
                double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
                double ang = p * inv_freq;
                double c = cos(ang), s = sin(ang);
                double x1 = or_bf16_to_double(v[i]);
                double x2 = or_bf16_to_double(v[i + half]);
                v[i] = or_bf16_from_double(x1 * c - x2 * s);
                v[i + half] = or_bf16_from_double(x2 * c + x1 * s);
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* a7: paged KV write                                                         */
/* ------------------------------------------------------------------------- */

/* Copy token t's K and V ([Hkv, D] each) into cache slot slot_mapping[t]; a
 * negative slot skips the token (padded decode rows, [SRV-61] "Summary").
 * Caches are [num_slots, Hkv, D] BF16 with num_slots = num_blocks * page
 * ([LIB-810] "BF16 KV cache": BF16 storage, no scale tensors). Returns -3 if a
 * slot is out of range (nothing written for that token), else 0.
 * Pinned: read-back and untouched-slot checks (tests). */
int or_kv_write(const uint16_t* k, const uint16_t* v, int T, int Hkv, int D,
                const int32_t* slot_mapping, uint16_t* k_cache, uint16_t* v_cache,
                long num_slots)
{
    int rc = 0;
    long row = (long)Hkv * D;
    for (int t = 0; t < T; ++t) {
        long s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_slots) {
            rc = -3;
            continue;
        }
        memcpy(k_cache + s * row, k + (long)t * row, sizeof(uint16_t) * row);
        memcpy(v_cache + s * row, v + (long)t * row, sizeof(uint16_t) * row);
    }
    return rc;
}

/* ------------------------------------------------------------------------- */
/* a8: GQA decode attention over the paged BF16 cache                        */
/* ------------------------------------------------------------------------- */

/* One cached element as a real number: the BF16 value, or for the INT8 cache
 * (scales != NULL) the code times its row's FP32 scale, exact in double. */
static double cache_elem(const void* cache, const float* scales, long slot, int Hkv,
                         int kvh, int D, int d)
{
    long r = slot * Hkv + kvh;
    if (!scales)
        return or_bf16_to_double(((const uint16_t*)cache)[r * D + d]);
    return (double)((const int8_t*)cache)[r * D + d] * (double)scales[r];
}

/* For request b and query head h (KV head kvh = h / (Hq / Hkv)), over the
 * ctx_lens[b] cached tokens t, whose slot is
 *   block_table[b][t / page] * page + t % page:
 *   s_t = scale * <q, K_t>,  p = softmax(s),  out = sum_t p_t V_t,
 * in double with the maximum subtracted, narrowed to BF16 once. [LIB-810]
 * "BF16 KV cache" (attention loads BF16 K/V directly, no dequantisation) and
 * [SRV-61] "Summary" (block table / slot mapping). A request with
 * ctx_lens[b] == 0 (a padded row) yields zeros. Returns -3 on an out-of-range
 * block id or context length (that head's output is zeroed), else 0.
 * Pinned: single-token context returns V, q = 0 returns the mean of V, paged
 * equals contiguous, shuffled pages give identical output, Hkv = Hq reduces to
 * per-head attention (tests). */
static int attention(const uint16_t* q, const void* k_cache, const void* v_cache,
                     const float* k_scale, const float* v_scale,
                     const int32_t* block_table, const int32_t* ctx_lens, int B, int Hq,
                     int Hkv, int D, int page, int max_blocks, int num_blocks,
                     double scale, uint16_t* out)
{
    int rc = 0;
    int G = Hq / Hkv;
    int max_ctx = max_blocks * page;
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        int n = ctx_lens[b];
        for (int h = 0; h < Hq; ++h) {
            uint16_t* ob = out + ((long)b * Hq + h) * D;
            int kvh = h / G;
            const uint16_t* qv = q + ((long)b * Hq + h) * D;
            int bad = (n < 0 || n > max_ctx);
            for (int t = 0; t < n && !bad; ++t) {
                int blk = block_table[(long)b * max_blocks + t / page];
                if (blk < 0 || blk >= num_blocks)
                    bad = 1;
            }
            if (bad)
                rc = -3;
            if (bad || n == 0) {
                for (int d = 0; d < D; ++d)
                    ob[d] = 0;
                continue;
            }
            double mx = -INFINITY;
            for (int t = 0; t < n; ++t) {
                long slot = (long)block_table[(long)b * max_blocks + t / page] * page + t % page;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += or_bf16_to_double(qv[d]) *
                           cache_elem(k_cache, k_scale, slot, Hkv, kvh, D, d);
                s[t] = dot * scale;
                if (s[t] > mx)
                    mx = s[t];
            }
            double l = 0.0;
            for (int t = 0; t < n; ++t) {
                s[t] = exp(s[t] - mx);
                l += s[t];
            }
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int t = 0; t < n; ++t) {
                long slot = (long)block_table[(long)b * max_blocks + t / page] * page + t % page;
                double p = s[t] / l;
                for (int d = 0; d < D; ++d)
                    o[d] += p * cache_elem(v_cache, v_scale, slot, Hkv, kvh, D, d);
            }
            for (int d = 0; d < D; ++d)
                ob[d] = or_bf16_from_double(o[d]);
        }
    }
    free(s);
    free(o);
    return rc;
}

int or_paged_attention(const uint16_t* q, const uint16_t* k_cache,
                       const uint16_t* v_cache, const int32_t* block_table,
                       const int32_t* ctx_lens, int B, int Hq, int Hkv, int D,
                       int page, int max_blocks, int num_blocks, double scale,
                       uint16_t* out)
{
    return attention(q, k_cache, v_cache, NULL, NULL, block_table, ctx_lens, B, Hq, Hkv,
                     D, page, max_blocks, num_blocks, scale, out);
}

/* ------------------------------------------------------------------------- */
/* Variant: INT8 KV cache with FP32 row scales                               */
/* ------------------------------------------------------------------------- */

/* [LIB-810] "BF16 KV cache" names the storage that BF16 replaced: INT8 K/V
 * cache rows with FP32 row scales, each token's K and V quantised when it is
 * written (decode and prefill) and every row dequantised where attention reads
 * it, the scales travelling in their own tensors.
 * Reading: a row is one KV head's D values of one token, quantised by the
 * activation formula (or_quant_rows: scale = absmax / 127, RNE, clamp +-127)
 * from the BF16 values the BF16 cache would hold (after QK RMSNorm and RoPE).
 * Codes [num_slots, Hkv, D] int8; scales [num_slots, Hkv] float. A negative
 * slot skips the token; an out-of-range slot returns -3 and writes nothing
 * for that token.
 * Pinned: every written row equals the quantisation of its head row, the
 * round trip stays within half a scale step, untouched slots stay untouched
 * (tests). */
int or_kv_write_i8(const uint16_t* k, const uint16_t* v, int T, int Hkv, int D,
                   const int32_t* slot_mapping, int8_t* k_codes, int8_t* v_codes,
                   float* k_scale, float* v_scale, long num_slots)
{
    int rc = 0;
    long row = (long)Hkv * D;
    for (int t = 0; t < T; ++t) {
        long s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_slots) {
            rc = -3;
            continue;
        }
        or_quant_rows(k + (long)t * row, Hkv, D, k_codes + s * row, k_scale + s * Hkv);
        or_quant_rows(v + (long)t * row, Hkv, D, v_codes + s * row, v_scale + s * Hkv);
    }
    return rc;
}

/* GQA decode attention over the INT8 cache: the BF16 form above with every
 * K_t and V_t element read as code x row scale ([LIB-810] "BF16 KV cache":
 * per-row K/V dequantisation inside attention). Same layout, bounds and
 * return codes as or_paged_attention.
 * Pinned: rows whose scale is a power of two (codes times 2^e exactly
 * representable in BF16) give the BF16-cache result bit for bit, with
 * different K and V scales per token and head; a single-token context
 * returns the dequantised V row (tests). */
int or_paged_attention_i8(const uint16_t* q, const int8_t* k_codes,
                          const int8_t* v_codes, const float* k_scale,
                          const float* v_scale, const int32_t* block_table,
                          const int32_t* ctx_lens, int B, int Hq, int Hkv, int D,
                          int page, int max_blocks, int num_blocks, double scale,
                          uint16_t* out)
{
    return attention(q, k_codes, v_codes, k_scale, v_scale, block_table, ctx_lens, B, Hq,
                     Hkv, D, page, max_blocks, num_blocks, scale, out);
}

/* ------------------------------------------------------------------------- */
/* Layer and step                                                            */
/* ------------------------------------------------------------------------- */

typedef struct {
    int hidden, num_q_heads, num_kv_heads, head_dim, intermediate;
    int num_layers, vocab, page_size, down_k_splits;
    double rms_eps, rope_theta;
} or_config;

typedef struct {
    const uint16_t* input_norm_w;   /* [H] */
    const int8_t* w_qkv;            /* [Hq*D + 2*Hkv*D, H]: Q heads, K heads, V heads */
    const float* s_qkv;
    const uint16_t* q_norm_w;       /* [D] */
    const uint16_t* k_norm_w;       /* [D] */
    const int8_t* w_o;              /* [H, Hq*D] */
    const float* s_o;
    const uint16_t* post_norm_w;    /* [H] */
    const int8_t* w_gate_up;        /* [2I, H]: gate rows then up rows */
    const float* s_gate_up;
    const int8_t* w_down;           /* [H, I] */
    const float* s_down;
} or_layer_weights;

/* Optional taps of every intermediate of one layer (any pointer may be NULL).
 * They mirror the pages' debug-stage switches for numerical diagnosis
 * ("Add Qwen3-14B A8W8 kernel implementation" summary quoted on [SRV-48]). */
typedef struct {
    uint16_t* xn;      int8_t* xq;   float* xs;   int32_t* acc_qkv; uint16_t* qkv;
    uint16_t* q_rot;   uint16_t* k_rot;  uint16_t* attn;  int8_t* aq;  float* as;
    int32_t* acc_o;    uint16_t* h1;  uint16_t* hn;  int8_t* hq;  float* hs;
    int32_t* acc_gu;   uint16_t* act; int8_t* actq;  float* acts; int32_t* acc_down;
} or_layer_taps;

#define TAP(ptr, src, bytes) do { if (taps && taps->ptr) memcpy(taps->ptr, src, bytes); } while (0)

/* One A8W8 decode layer on B rows, in the order of the method:
 *   a2 input RMSNorm, a3 quant, a4 QKV, a5 per-head QK RMSNorm, a6 RoPE at
 *   position ctx_len - 1, a7 KV write, a8 paged GQA attention, a9 quant,
 *   a10 O + residual, a11 post-attention RMSNorm + quant, a12 gate/up +
 *   SwiGLU, a13 quant, a14 split-K down + residual.
 * hidden [B, H] is updated in place. Caches are [num_blocks * page, Hkv, D].
 * Padded rows (slot -1, ctx_len 0) write no KV and attend to nothing.
 * Returns 0, or a negative code (-1 shapes, -3 bounds), or 1 on int32
 * overflow. */
static int layer(const or_layer_weights* w, const or_config* cfg, int B,
                 uint16_t* hidden, const int32_t* slot_mapping,
                 const int32_t* block_table, int max_blocks, int num_blocks,
                 const int32_t* ctx_lens, void* k_cache, void* v_cache, float* k_scale,
                 float* v_scale, const or_layer_taps* taps)
{
    const int H = cfg->hidden, Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
    const int D = cfg->head_dim, I = cfg->intermediate;
    const int NQ = Hq * D, NK = Hkv * D, NQKV = NQ + 2 * NK;
    if (Hq % Hkv != 0 || D % 2 != 0)
        return -1;
    int rc = 0, ov = 0;
    size_t bh = (size_t)B * H;

    uint16_t* xn = malloc(sizeof(uint16_t) * bh);
    int8_t* xq = malloc(bh);
    float* xs = malloc(sizeof(float) * B);
    int32_t* acc = malloc(sizeof(int32_t) * (size_t)B * (NQKV > 2 * I ? NQKV : 2 * I));
    uint16_t* qkv = malloc(sizeof(uint16_t) * (size_t)B * NQKV);
    uint16_t* q = malloc(sizeof(uint16_t) * (size_t)B * NQ);
    uint16_t* k = malloc(sizeof(uint16_t) * (size_t)B * NK);
    uint16_t* v = malloc(sizeof(uint16_t) * (size_t)B * NK);
    uint16_t* attn = malloc(sizeof(uint16_t) * (size_t)B * NQ);
    int8_t* aq = malloc((size_t)B * (NQ > I ? NQ : I));
    float* as = malloc(sizeof(float) * B);
    uint16_t* act = malloc(sizeof(uint16_t) * (size_t)B * I);
    int32_t* pos = malloc(sizeof(int32_t) * B);

    /* a2, a3 */
    or_rmsnorm(hidden, w->input_norm_w, B, H, cfg->rms_eps, xn);
    or_quant_rows(xn, B, H, xq, xs);
    TAP(xn, xn, sizeof(uint16_t) * bh);
    TAP(xq, xq, bh);
    TAP(xs, xs, sizeof(float) * B);
    /* a4 */
    ov |= or_linear(xq, xs, B, H, w->w_qkv, w->s_qkv, NQKV, 1, NULL, qkv, acc);
    TAP(acc_qkv, acc, sizeof(int32_t) * (size_t)B * NQKV);
    TAP(qkv, qkv, sizeof(uint16_t) * (size_t)B * NQKV);
    for (int b = 0; b < B; ++b) {
        memcpy(q + (size_t)b * NQ, qkv + (size_t)b * NQKV, sizeof(uint16_t) * NQ);
        memcpy(k + (size_t)b * NK, qkv + (size_t)b * NQKV + NQ, sizeof(uint16_t) * NK);
        memcpy(v + (size_t)b * NK, qkv + (size_t)b * NQKV + NQ + NK, sizeof(uint16_t) * NK);
        pos[b] = ctx_lens[b] - 1;
    }
    /* a5: per-head RMSNorm over D, in place (rows = tokens x heads) */
    or_rmsnorm(q, w->q_norm_w, B * Hq, D, cfg->rms_eps, q);
    or_rmsnorm(k, w->k_norm_w, B * Hkv, D, cfg->rms_eps, k);
    /* a6 */
    or_rope(q, B, Hq, D, pos, cfg->rope_theta);
    or_rope(k, B, Hkv, D, pos, cfg->rope_theta);
    TAP(q_rot, q, sizeof(uint16_t) * (size_t)B * NQ);
    TAP(k_rot, k, sizeof(uint16_t) * (size_t)B * NK);
    /* a7 */
    long num_slots = (long)num_blocks * cfg->page_size;
    int wr = k_scale ? or_kv_write_i8(k, v, B, Hkv, D, slot_mapping, (int8_t*)k_cache,
                                      (int8_t*)v_cache, k_scale, v_scale, num_slots)
                     : or_kv_write(k, v, B, Hkv, D, slot_mapping, (uint16_t*)k_cache,
                                   (uint16_t*)v_cache, num_slots);
    if (wr != 0)
        rc = -3;
    /* a8 */
    if (attention(q, k_cache, v_cache, k_scale, v_scale, block_table, ctx_lens, B, Hq, Hkv,
                  D, cfg->page_size, max_blocks, num_blocks, 1.0 / sqrt((double)D),
                  attn) != 0)
        rc = -3;
    TAP(attn, attn, sizeof(uint16_t) * (size_t)B * NQ);
    /* a9, a10: the residual is the layer input */
    or_quant_rows(attn, B, NQ, aq, as);
    TAP(aq, aq, (size_t)B * NQ);
    TAP(as, as, sizeof(float) * B);
    ov |= or_linear(aq, as, B, NQ, w->w_o, w->s_o, H, 1, hidden, hidden, acc);
    TAP(acc_o, acc, sizeof(int32_t) * bh);
    TAP(h1, hidden, sizeof(uint16_t) * bh);
    /* a11 */
    or_rmsnorm(hidden, w->post_norm_w, B, H, cfg->rms_eps, xn);
    or_quant_rows(xn, B, H, xq, xs);
    TAP(hn, xn, sizeof(uint16_t) * bh);
    TAP(hq, xq, bh);
    TAP(hs, xs, sizeof(float) * B);
    /* a12 */
    ov |= or_gate_up_swiglu(xq, xs, B, H, w->w_gate_up, w->s_gate_up, I, act, acc);
    TAP(acc_gu, acc, sizeof(int32_t) * (size_t)B * 2 * I);
    TAP(act, act, sizeof(uint16_t) * (size_t)B * I);
    /* a13, a14 */
    or_quant_rows(act, B, I, aq, as);
    TAP(actq, aq, (size_t)B * I);
    TAP(acts, as, sizeof(float) * B);
    int lr = or_linear(aq, as, B, I, w->w_down, w->s_down, H, cfg->down_k_splits,
                       hidden, hidden, acc);
    if (lr < 0)
        rc = -1;
    else
        ov |= lr;
    TAP(acc_down, acc, sizeof(int32_t) * bh);

    free(xn); free(xq); free(xs); free(acc); free(qkv); free(q); free(k); free(v);
    free(attn); free(aq); free(as); free(act); free(pos);
    return rc != 0 ? rc : ov;
}

int or_decode_layer(const or_layer_weights* w, const or_config* cfg, int B,
                    uint16_t* hidden, const int32_t* slot_mapping,
                    const int32_t* block_table, int max_blocks, int num_blocks,
                    const int32_t* ctx_lens, uint16_t* k_cache, uint16_t* v_cache,
                    const or_layer_taps* taps)
{
    return layer(w, cfg, B, hidden, slot_mapping, block_table, max_blocks, num_blocks,
                 ctx_lens, k_cache, v_cache, NULL, NULL, taps);
}

/* The same layer over the INT8 KV cache with FP32 row scales: a7 quantises
 * each written K/V head row (or_kv_write_i8) and a8 dequantises every row it
 * reads (or_paged_attention_i8); every other step is unchanged ([LIB-810]
 * "BF16 KV cache", the storage it replaced). Codes [num_blocks * page, Hkv, D],
 * scales [num_blocks * page, Hkv].
 * Pinned: the steps before a7 equal the BF16-cache layer's bit for bit, the
 * cache holds the quantised K/V rows of that layer at their slots (tests). */
int or_decode_layer_i8kv(const or_layer_weights* w, const or_config* cfg, int B,
                         uint16_t* hidden, const int32_t* slot_mapping,
                         const int32_t* block_table, int max_blocks, int num_blocks,
                         const int32_t* ctx_lens, int8_t* k_codes, int8_t* v_codes,
                         float* k_scale, float* v_scale, const or_layer_taps* taps)
{
    if (!k_scale || !v_scale)
        return -1;
    return layer(w, cfg, B, hidden, slot_mapping, block_table, max_blocks, num_blocks,
                 ctx_lens, k_codes, v_codes, k_scale, v_scale, taps);
}

/* ------------------------------------------------------------------------- */
/* Variant: BF16 (unquantised) decode layer                                  */
/* ------------------------------------------------------------------------- */

/* [LIB-810] (the kernel PR's summary quoted there) and [SRV-48] "Summary"
 * keep the ordinary BF16 Qwen3-14B path beside the A8W8 one without spelling
 * out its arithmetic. Reading: the same layer with BF16 weights and no
 * quantisation, each projection the real-valued sum narrowed to BF16 once:
 *   y[m][n] = bf16( sum_k x[m][k] W[n][k] (+ residual[m][n]) ),
 * evaluated in double (each BF16 x BF16 product is exact there; the sum's
 * rounding is far below the BF16 step). W is [N, K] row-major.
 * Pinned: brute force in rational arithmetic; operands that are powers of two
 * times INT8 codes reproduce the pinned A8W8 projection (tests). */
void or_linear_bf16(const uint16_t* x, int M, int K, const uint16_t* W, int N,
                    const uint16_t* residual, uint16_t* y)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t* xr = x + (long)m * K;
#pragma omp parallel for schedule(static)
        for (int n = 0; n < N; ++n) {
            const uint16_t* wr = W + (long)n * K;
            double s = 0.0;
            for (int k = 0; k < K; ++k)
                s += or_bf16_to_double(xr[k]) * or_bf16_to_double(wr[k]);
            if (residual)
                s += or_bf16_to_double(residual[(long)m * N + n]);
            y[(long)m * N + n] = or_bf16_from_double(s);
        }
    }
}

/* Fused Gate/Up with SwiGLU on BF16 weights W_gu [2I, K] (gate rows, then up
 * rows): g and u are the real-valued sums, not narrowed, and
 * act = bf16( g / (1 + exp(-g)) * u ) in double, as in the A8W8 form.
 * Pinned through the layer taps and the closed forms of the A8W8 form's SiLU
 * (tests). */
void or_gate_up_swiglu_bf16(const uint16_t* x, int M, int K, const uint16_t* W_gu, int I,
                            uint16_t* act)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t* xr = x + (long)m * K;
#pragma omp parallel for schedule(static)
        for (int j = 0; j < I; ++j) {
            const uint16_t* wg = W_gu + (long)j * K;
            const uint16_t* wu = W_gu + (long)(I + j) * K;
            double g = 0.0, u = 0.0;
            for (int k = 0; k < K; ++k) {
                double xv = or_bf16_to_double(xr[k]);
                g += xv * or_bf16_to_double(wg[k]);
                u += xv * or_bf16_to_double(wu[k]);
            }
            act[(long)m * I + j] = or_bf16_from_double(g / (1.0 + exp(-g)) * u);
        }
    }
}

typedef struct {
    const uint16_t* input_norm_w;   /* [H] */
    const uint16_t* w_qkv;          /* [Hq*D + 2*Hkv*D, H]: Q heads, K heads, V heads */
    const uint16_t* q_norm_w;       /* [D] */
    const uint16_t* k_norm_w;       /* [D] */
    const uint16_t* w_o;            /* [H, Hq*D] */
    const uint16_t* post_norm_w;    /* [H] */
    const uint16_t* w_gate_up;      /* [2I, H]: gate rows then up rows */
    const uint16_t* w_down;         /* [H, I] */
} or_layer_weights_bf16;

/* One BF16 decode layer on B rows: input RMSNorm, QKV projection, per-head QK
 * RMSNorm, RoPE at position ctx_len - 1, KV write, paged GQA attention, O
 * projection + residual, post-attention RMSNorm, Gate/Up + SwiGLU, down
 * projection + residual; the A8W8 layer's order with every quantisation step
 * removed and the projections by or_linear_bf16. Taps used: xn, qkv, q_rot,
 * k_rot, attn, h1, hn, act (the others are left untouched). hidden [B, H] is
 * updated in place; caches are BF16 [num_blocks * page, Hkv, D]. Returns 0,
 * -1 on shapes, -3 on bounds.
 * Pinned: every tap equals the pinned steps composed in order; zero O and
 * down weights keep the residual; the first token attends to its own V. */
int or_decode_layer_bf16(const or_layer_weights_bf16* w, const or_config* cfg, int B,
                         uint16_t* hidden, const int32_t* slot_mapping,
                         const int32_t* block_table, int max_blocks, int num_blocks,
                         const int32_t* ctx_lens, uint16_t* k_cache, uint16_t* v_cache,
                         const or_layer_taps* taps)
{
    const int H = cfg->hidden, Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
    const int D = cfg->head_dim, I = cfg->intermediate;
    const int NQ = Hq * D, NK = Hkv * D, NQKV = NQ + 2 * NK;
    if (Hq % Hkv != 0 || D % 2 != 0)
        return -1;
    int rc = 0;
    size_t bh = (size_t)B * H;
    uint16_t* xn = malloc(sizeof(uint16_t) * bh);
    uint16_t* qkv = malloc(sizeof(uint16_t) * (size_t)B * NQKV);
    uint16_t* q = malloc(sizeof(uint16_t) * (size_t)B * NQ);
    uint16_t* k = malloc(sizeof(uint16_t) * (size_t)B * NK);
    uint16_t* v = malloc(sizeof(uint16_t) * (size_t)B * NK);
    uint16_t* attn = malloc(sizeof(uint16_t) * (size_t)B * NQ);
    uint16_t* act = malloc(sizeof(uint16_t) * (size_t)B * I);
    int32_t* pos = malloc(sizeof(int32_t) * B);

    or_rmsnorm(hidden, w->input_norm_w, B, H, cfg->rms_eps, xn);
    TAP(xn, xn, sizeof(uint16_t) * bh);
    or_linear_bf16(xn, B, H, w->w_qkv, NQKV, NULL, qkv);
    TAP(qkv, qkv, sizeof(uint16_t) * (size_t)B * NQKV);
    for (int b = 0; b < B; ++b) {
        memcpy(q + (size_t)b * NQ, qkv + (size_t)b * NQKV, sizeof(uint16_t) * NQ);
        memcpy(k + (size_t)b * NK, qkv + (size_t)b * NQKV + NQ, sizeof(uint16_t) * NK);
        memcpy(v + (size_t)b * NK, qkv + (size_t)b * NQKV + NQ + NK, sizeof(uint16_t) * NK);
        pos[b] = ctx_lens[b] - 1;
    }
    or_rmsnorm(q, w->q_norm_w, B * Hq, D, cfg->rms_eps, q);
    or_rmsnorm(k, w->k_norm_w, B * Hkv, D, cfg->rms_eps, k);
    or_rope(q, B, Hq, D, pos, cfg->rope_theta);
    or_rope(k, B, Hkv, D, pos, cfg->rope_theta);
    TAP(q_rot, q, sizeof(uint16_t) * (size_t)B * NQ);
    TAP(k_rot, k, sizeof(uint16_t) * (size_t)B * NK);
    long num_slots = (long)num_blocks * cfg->page_size;
    if (or_kv_write(k, v, B, Hkv, D, slot_mapping, k_cache, v_cache, num_slots) != 0)
        rc = -3;
    if (or_paged_attention(q, k_cache, v_cache, block_table, ctx_lens, B, Hq, Hkv, D,
                           cfg->page_size, max_blocks, num_blocks, 1.0 / sqrt((double)D),
                           attn) != 0)
        rc = -3;
    TAP(attn, attn, sizeof(uint16_t) * (size_t)B * NQ);
    or_linear_bf16(attn, B, NQ, w->w_o, H, hidden, hidden);
    TAP(h1, hidden, sizeof(uint16_t) * bh);
    or_rmsnorm(hidden, w->post_norm_w, B, H, cfg->rms_eps, xn);
    TAP(hn, xn, sizeof(uint16_t) * bh);
    or_gate_up_swiglu_bf16(xn, B, H, w->w_gate_up, I, act);
    TAP(act, act, sizeof(uint16_t) * (size_t)B * I);
    or_linear_bf16(act, B, I, w->w_down, H, hidden, hidden);

    free(xn); free(qkv); free(q); free(k); free(v); free(attn); free(act); free(pos);
    return rc;
}

/* Final RMSNorm, BF16 LM head and greedy argmax.
 * logits[b][v] = sum_k hn[b][k] * W_lm[v][k] in double (BF16 operands);
 * next[b] = the lowest index of the maximum logit. [SRV-48] "Performance"
 * settings (temperature 0, top_p 1: greedy decoding) and [SRV-61] "Related"
 * (device-side embedding and sampling). Reading: LM head in BF16, argmax ties
 * go to the lowest index. Pinned: brute-force argmax and ties (tests). */
void or_argmax_f64(const double* logits, int B, int V, int32_t* next)
{
    for (int b = 0; b < B; ++b) {
        const double* l = logits + (long)b * V;
        int best = 0;
        for (int v = 1; v < V; ++v)
            if (l[v] > l[best])
                best = v;
        next[b] = best;
    }
}

/* The same argmax over FP32 logits, so that a decision taken on a GPU's FP32
 * logits can be checked in the GPU's own precision. */
void or_argmax_f32(const float* logits, int B, int V, int32_t* next)
{
    for (int b = 0; b < B; ++b) {
        const float* l = logits + (long)b * V;
        int best = 0;
        for (int v = 1; v < V; ++v)
            if (l[v] > l[best])
                best = v;
        next[b] = best;
    }
}

void or_lm_head(const uint16_t* hn, int B, int H, const uint16_t* W_lm, int V,
                double* logits)
{
    for (int b = 0; b < B; ++b) {
        const uint16_t* h = hn + (long)b * H;
#pragma omp parallel for schedule(static)
        for (int v = 0; v < V; ++v) {
            const uint16_t* wr = W_lm + (long)v * H;
            double s = 0.0;
            for (int k = 0; k < H; ++k)
                s += or_bf16_to_double(h[k]) * or_bf16_to_double(wr[k]);
            logits[(long)b * V + v] = s;
        }
    }
}

typedef struct {
    const uint16_t* embed;              /* [vocab, H] */
    const or_layer_weights* layers;     /* [num_layers] */
    const uint16_t* final_norm_w;       /* [H] */
    const uint16_t* lm_head;            /* [vocab, H] */
} or_model;

/* One decode step: a1 embedding gather, the layers, a15 final RMSNorm, LM
 * head, greedy argmax. k_caches / v_caches hold one cache per layer.
 * final_hidden [B, H] (nullable) receives the normalised last hidden state;
 * logits [B, vocab] (nullable) the double logits. Returns as or_decode_layer,
 * or -3 for an out-of-range token id. */
int or_decode_step(const or_model* m, const or_config* cfg, int B,
                   const int32_t* token_ids, const int32_t* slot_mapping,
                   const int32_t* block_table, int max_blocks, int num_blocks,
                   const int32_t* ctx_lens, uint16_t* const* k_caches,
                   uint16_t* const* v_caches, int32_t* next_tokens,
                   double* logits, uint16_t* final_hidden)
{
    const int H = cfg->hidden, V = cfg->vocab;
    int rc = 0;
    uint16_t* hidden = malloc(sizeof(uint16_t) * (size_t)B * H);
    uint16_t* hn = malloc(sizeof(uint16_t) * (size_t)B * H);
    double* lg = logits ? logits : malloc(sizeof(double) * (size_t)B * V);
    for (int b = 0; b < B; ++b) {
        int id = token_ids[b];
        if (id < 0 || id >= V) {
            rc = -3;
            memset(hidden + (size_t)b * H, 0, sizeof(uint16_t) * H);
            continue;
        }
        memcpy(hidden + (size_t)b * H, m->embed + (size_t)id * H, sizeof(uint16_t) * H);
    }
    for (int l = 0; l < cfg->num_layers; ++l) {
        int r = or_decode_layer(&m->layers[l], cfg, B, hidden, slot_mapping, block_table,
                                max_blocks, num_blocks, ctx_lens, k_caches[l], v_caches[l],
                                NULL);
        if (r != 0 && rc == 0)
            rc = r;
    }
    or_rmsnorm(hidden, m->final_norm_w, B, H, cfg->rms_eps, hn);
    if (final_hidden)
        memcpy(final_hidden, hn, sizeof(uint16_t) * (size_t)B * H);
    or_lm_head(hn, B, H, m->lm_head, V, lg);
    or_argmax_f64(lg, B, V, next_tokens);
    if (!logits)
        free(lg);
    free(hidden);
    free(hn);
    return rc;
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
