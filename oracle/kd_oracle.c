/*
 * kd_oracle.c -- plain, slow CPU reference of one batched decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  The product
 * path (the CUDA library) shares no code, header, table or helper with it.
 *
 * What it computes follows the batched decode step of memra-engine's
 * `decode_batch.rs` (module header "EXACTNESS CONTRACT"; `decode_batch_layers`,
 * the per-layer body; `decode_step_batch_lean_masked`, embedding and head;
 * `decode_batch_epilogue`, the device argmax), restricted to a dense
 * Llama-shaped model: no QK-norm, no output gate, no linear-attention or MoE
 * layers.  Batching changes no arithmetic ("row-parallel ops batch trivially";
 * every projection row is bit-identical to its m=1 result), so the oracle is
 * the plain single-session step, run once per session.
 *
 * All arithmetic is fp64.  Only the method's storage roundings are mirrored:
 *   - matmul inputs (normed activations, attention output, SwiGLU output) are
 *     rounded to fp16, the KV cache is fp16, the residual stream and the
 *     logits are fp32.
 * Conventions the pages leave open (each is listed with its reason in the
 * design notes): Q8_0 blocks run along the input dimension; RoPE is the NeoX
 * rotate-half form over the whole head; q head h reads KV head
 * h / (n_heads / n_kv_heads); the attention scale is 1/sqrt(head_dim); the new
 * token is written at its position p and attends keys 0..p; argmax ties go
 * to the lowest index and NaN never wins.
 *
 * No blocking, fusion or reordering: every dot product runs over its blocks in
 * order; OpenMP only spreads independent output rows or heads over threads,
 * so the results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDO_EXPORT __attribute__((visibility("default")))

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary64, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 holds
 * the subnormals (fraction * 2^-24), exponent 31 holds Inf and NaN.
 * ------------------------------------------------------------------------- */
KDO_EXPORT double kdo_half_to_double(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(f + 1024), e - 25);
    return sign ? -v : v;
}

/* Round to nearest, ties to even (nearbyint in the default rounding mode). */
KDO_EXPORT uint16_t kdo_double_to_half(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return 0x7e00;
    if (isinf(x)) return sign | 0x7c00;
    double a = fabs(x);
    if (a < ldexp(1.0, -14)) {                 /* subnormal range: units of 2^-24 */
        double r = nearbyint(a * 16777216.0);  /* exact scaling, one rounding */
        return sign | (uint16_t)r;             /* r == 1024 is the smallest normal */
    }
    int e;
    double f = frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
    double r = nearbyint(ldexp(f, 11));        /* 11 significant bits: [1024, 2048] */
    if (r == 2048.0) { r = 1024.0; e += 1; }
    int be = e - 1 + 15;
    if (be >= 31) return sign | 0x7c00;        /* overflow rounds to infinity */
    return sign | (uint16_t)(be << 10) | (uint16_t)((int)r - 1024);
}

static double round_half(double x) { return kdo_half_to_double(kdo_double_to_half(x)); }

/* The same decoding as a table over all 65536 bit patterns, filled from
 * kdo_half_to_double when the library loads: identical values, one load per
 * cached K/V element instead of a call (the attention reads tens of millions
 * of them per long-context step). */
static double g_half_table[65536];
__attribute__((constructor)) static void fill_half_table(void) {
    for (uint32_t h = 0; h < 65536; ++h) g_half_table[h] = kdo_half_to_double((uint16_t)h);
}
static inline double half_value(uint16_t h) { return g_half_table[h]; }
static double round_float(double x) { return (double)(float)x; }

/* ---------------------------------------------------------------------------
 * Q8_0: one block = fp16 scale d then 32 int8 quants q_j; value_j = q_j * d.
 * (Named as the weight format on memra's and hf2q's pages; the closed form is
 * value = int8 x fp16 scale per 32-element block.)
 * ------------------------------------------------------------------------- */
#define QK 32
#define QB 34

static double q8_scale(const uint8_t* blk) {
    uint16_t h = (uint16_t)blk[0] | ((uint16_t)blk[1] << 8);
    return kdo_half_to_double(h);
}

/* Dequantise one row of `cols` values (cols a multiple of 32). */
KDO_EXPORT void kdo_q8_0_dequant_row(const uint8_t* row, int32_t cols, double* out) {
    for (int b = 0; b < cols / QK; ++b) {
        const uint8_t* blk = row + (size_t)b * QB;
        double d = q8_scale(blk);
        for (int j = 0; j < QK; ++j) out[b * QK + j] = (double)(int8_t)blk[2 + j] * d;
    }
}

/* y[r] = sum over blocks b of d_rb * sum_j q_rbj * x[32b + j]  (W is [rows][cols/32] blocks).
 * This is the projection `matmul(W, x)` of the layer body, one input vector. */
KDO_EXPORT void kdo_matvec_q8_0(const uint8_t* W, int32_t rows, int32_t cols,
                                const double* x, double* y) {
    const size_t row_bytes = (size_t)(cols / QK) * QB;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint8_t* row = W + (size_t)r * row_bytes;
        double acc = 0.0;
        for (int b = 0; b < cols / QK; ++b) {
            const uint8_t* blk = row + (size_t)b * QB;
            double s = 0.0;
            for (int j = 0; j < QK; ++j) s += (double)(int8_t)blk[2 + j] * x[b * QK + j];
            acc += q8_scale(blk) * s;
        }
        y[r] = acc;
    }
}

/* RMSNorm then fp16 rounding: out_i = fp16(x_i / sqrt(mean(x^2) + eps) * w_i).
 * (`rms_norm(x, w, out, n_embd, rows, eps)` of the layer body.) */
KDO_EXPORT void kdo_rmsnorm_f16(const double* x, const float* w, int32_t n, double eps,
                                double* out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) out[i] = round_half(x[i] * r * (double)w[i]);
}

/* NeoX rotate-half RoPE of one head vector u[hd] at position pos:
 * for i < hd/2, with w_i = theta^(-2i/hd) and a = pos * w_i,
 * (u_i, u_{i+hd/2}) <- (u_i cos a - u_{i+hd/2} sin a, u_i sin a + u_{i+hd/2} cos a).
 * (`rope_neox(x, pos_d, head_dim, rope_dims, n_heads, B, base, 1.0)`, each row at its own position.) */
KDO_EXPORT void kdo_rope_neox(double* u, int32_t hd, int32_t pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double a = (double)pos * pow(theta, -2.0 * i / hd);
        double c = cos(a), s = sin(a);
        double x0 = u[i], x1 = u[i + half];
        u[i] = x0 * c - x1 * s;
        u[i + half] = x0 * s + x1 * c;
    }
}

/* Single-head attention over t_kv cached rows, two-pass softmax:
 * s_t = scale * q . K_t ; m = max_t s_t ; a = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m).
 * K, V are fp16 bits with row stride `stride` elements. */
KDO_EXPORT void kdo_attention_head(const double* q, const uint16_t* K, const uint16_t* V,
                                   int32_t t_kv, int32_t hd, int64_t stride, double scale,
                                   double* out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(t_kv > 0 ? t_kv : 1));
    double m = -INFINITY;
    for (int t = 0; t < t_kv; ++t) {
        double dot = 0.0;
        for (int i = 0; i < hd; ++i) dot += q[i] * half_value(K[(size_t)t * stride + i]);
        s[t] = dot * scale;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int t = 0; t < t_kv; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
    /* a_i = sum over t in order of s_t V_t,i (row by row through V; each
     * dimension's sum still runs over t = 0, 1, ... in order) */
    double* acc = (double*)calloc((size_t)hd, sizeof(double));
    for (int t = 0; t < t_kv; ++t)
        for (int i = 0; i < hd; ++i) acc[i] += s[t] * half_value(V[(size_t)t * stride + i]);
    for (int i = 0; i < hd; ++i) out[i] = acc[i] / l;
    free(acc);
    free(s);
}

/* ---------------------------------------------------------------------------
 * Q8_0 KV cache (the long-context option: memra appends quantized K/V,
 * `decode_batch_layers` phase A; hf2q ADR-040 measures against llama.cpp with
 * q8_0 K/V).  A cached head row of hd values is hd/32 canonical blocks.
 * Quantisation, in fp32 (the precision the kernel takes the integer decision
 * in): per block d = max|x| / 127, stored as fp16(d); q_j = x_j / d rounded to
 * the nearest integer, halves away from zero, within [-127, 127]; an all-zero
 * block gives d = 0, q = 0.  Inputs are finite.  Dequantised value = q * fp16(d).
 * ------------------------------------------------------------------------- */
KDO_EXPORT void kdo_q8_0_quantize_f32(const float* x, int32_t n, uint8_t* out) {
    for (int b = 0; b < n / QK; ++b) {
        const float* xb = x + (size_t)b * QK;
        uint8_t* ob = out + (size_t)b * QB;
        float amax = 0.0f;
        for (int j = 0; j < QK; ++j) {
            const float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        const float d = amax / 127.0f;
        const uint16_t dh = kdo_double_to_half((double)d);
        ob[0] = (uint8_t)(dh & 0xff);
        ob[1] = (uint8_t)(dh >> 8);
        for (int j = 0; j < QK; ++j) {
            int q = 0;
            if (d > 0.0f) {
                q = (int)roundf(xb[j] / d);
                if (q > 127) q = 127;
                if (q < -127) q = -127;
            }
            ob[2 + j] = (uint8_t)(int8_t)q;
        }
    }
}

/* Element i of a cached Q8_0 row. */
static double q8_row_value(const uint8_t* row, int i) {
    const uint8_t* blk = row + (size_t)(i / QK) * QB;
    return (double)(int8_t)blk[2 + i % QK] * q8_scale(blk);
}

/* kdo_attention_head over a Q8_0 cache: rows of row_bytes, values dequantised. */
KDO_EXPORT void kdo_attention_head_q8(const double* q, const uint8_t* K, const uint8_t* V, int32_t t_kv,
                                      int32_t hd, int64_t row_bytes, double scale, double* out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(t_kv > 0 ? t_kv : 1));
    double m = -INFINITY;
    for (int t = 0; t < t_kv; ++t) {
        double dot = 0.0;
        for (int i = 0; i < hd; ++i) dot += q[i] * q8_row_value(K + (size_t)t * row_bytes, i);
        s[t] = dot * scale;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int t = 0; t < t_kv; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
    double* acc = (double*)calloc((size_t)hd, sizeof(double));
    for (int t = 0; t < t_kv; ++t)
        for (int i = 0; i < hd; ++i) acc[i] += s[t] * q8_row_value(V + (size_t)t * row_bytes, i);
    for (int i = 0; i < hd; ++i) out[i] = acc[i] / l;
    free(acc);
    free(s);
}

/* silu(y) = y / (1 + e^-y). (`silu_mul(g, u, act, n)` computes silu(g) * u.) */
KDO_EXPORT double kdo_silu(double y) { return y / (1.0 + exp(-y)); }

/* Greedy pick: the largest value, ties to the lowest index, NaN never wins;
 * a row with no non-NaN value gives -1.  (`argmax_token_device_col`.) */
KDO_EXPORT int32_t kdo_argmax_f32(const float* v, int32_t n) {
    int32_t best = -1;
    for (int32_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best;
}

/* ---------------------------------------------------------------------------
 * Device temperature sampling (memra-engine decode_batch.rs,
 * `decode_step_batch_sampled`: a Gumbel perturbation keyed by (seed, counter,
 * temperature) followed by the same argmax is one categorical draw from
 * softmax(logits / temperature); temperature <= 0 is the greedy argmax; the
 * draw depends on (seed, counter) only, never on the rest of the batch).
 *
 * The pages name Philox as the counter-based generator and fix nothing else;
 * the reading taken: Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11), vocabulary entry v drawing word
 * v mod 4 of the block at counter (v / 4, counter, 0, 0) under key (seed, 0);
 * u = (top 24 bits + 1/2) / 2^24, g = -log(-log u), z = logit / T + g, all in
 * fp32 (the decision is taken in the kernel's precision); the pick is the
 * argmax of z with the greedy rule's ties and NaN handling.
 * ------------------------------------------------------------------------- */
static void mul64_hilo(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
    /* 64 x 64 -> 128 from 32-bit halves */
    const uint64_t a0 = a & 0xffffffffu, a1 = a >> 32, b0 = b & 0xffffffffu, b1 = b >> 32;
    const uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    const uint64_t mid = (p00 >> 32) + (p01 & 0xffffffffu) + (p10 & 0xffffffffu);
    *lo = (mid << 32) | (p00 & 0xffffffffu);
    *hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

/* Philox4x64 with 10 rounds: each round multiplies words 0 and 2 by the two
 * round multipliers, mixes the high halves with words 1 and 3 and the key,
 * and permutes; the key is bumped by the two Weyl constants between rounds. */
KDO_EXPORT void kdo_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += W0; k1 += W1; }
        uint64_t hi0, lo0, hi1, lo1;
        mul64_hilo(M0, c0, &hi0, &lo0);
        mul64_hilo(M1, c2, &hi1, &lo1);
        const uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The perturbed value of vocabulary entry v (fp32). */
KDO_EXPORT float kdo_gumbel_perturbed(float logit, int32_t v, float temperature, uint64_t seed, uint64_t counter) {
    const uint64_t ctr[4] = {(uint64_t)(v / 4), counter, 0, 0}, key[2] = {seed, 0};
    uint64_t w[4];
    kdo_philox4x64_10(ctr, key, w);
    const float u = ((float)(w[v % 4] >> 40) + 0.5f) * 0x1p-24f;  /* in (0, 1), exact */
    const float g = -logf(-logf(u));
    return logit / temperature + g;
}

/* One draw per the reading above: the index, or -1 if every logit is NaN. */
KDO_EXPORT int32_t kdo_sample_f32(const float* logits, int32_t n, float temperature, uint64_t seed,
                                  uint64_t counter) {
    if (!(temperature > 0.0f)) return kdo_argmax_f32(logits, n);
    int32_t best = -1;
    float bv = 0.0f;
    for (int32_t i = 0; i < n; ++i) {
        if (isnan(logits[i])) continue;
        const float z = kdo_gumbel_perturbed(logits[i], i, temperature, seed, counter);
        if (isnan(z)) continue;
        if (best < 0 || z > bv) { best = i; bv = z; }
    }
    return best;
}

/* ---------------------------------------------------------------------------
 * The model and one decode step.
 * ------------------------------------------------------------------------- */
typedef struct {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
    double rope_theta, rms_eps;
    int32_t kv_q8_0;  /* 0: fp16 KV caches; 1: Q8_0 KV caches */
} kdo_config;

/* Bytes of one cached head row. */
static size_t kv_row_bytes(const kdo_config* c) {
    return c->kv_q8_0 ? (size_t)(c->head_dim / QK) * QB : (size_t)c->head_dim * 2;
}

typedef struct {
    const uint8_t* tok_embd;          /* Q8_0 [vocab][hidden/32] */
    const uint8_t* output;            /* Q8_0 [vocab][hidden/32] (lm_head) */
    const float* output_norm;         /* [hidden] */
    const uint8_t* const* wq;         /* per layer, Q8_0 [n_heads*hd][hidden/32] */
    const uint8_t* const* wk;         /* [n_kv*hd][hidden/32] */
    const uint8_t* const* wv;         /* [n_kv*hd][hidden/32] */
    const uint8_t* const* wo;         /* [hidden][n_heads*hd/32] */
    const uint8_t* const* w_gate;     /* [ffn][hidden/32] */
    const uint8_t* const* w_up;       /* [ffn][hidden/32] */
    const uint8_t* const* w_down;     /* [hidden][ffn/32] */
    const float* const* attn_norm;    /* [hidden] */
    const float* const* ffn_norm;     /* [hidden] */
} kdo_weights;

/* One layer of one session (the body of `decode_batch_layers` for one row):
 * x is the fp32-valued residual stream [hidden], updated in place.  The layer's
 * caches are [n_kv][cap] rows (fp16 [hd], or Q8_0 blocks with kv_q8_0); row
 * `pos` is written, rows 0..pos are read. */
KDO_EXPORT int32_t kdo_layer_step(const kdo_config* c, const kdo_weights* w, int32_t l,
                                  int32_t pos, void* Kv, void* Vv, int32_t cap,
                                  double* x) {
    uint16_t* Kl = (uint16_t*)Kv;
    uint16_t* Vl = (uint16_t*)Vv;
    uint8_t* Kq = (uint8_t*)Kv;
    uint8_t* Vq = (uint8_t*)Vv;
    const size_t rb = kv_row_bytes(c);
    const int H = c->hidden, nh = c->n_heads, nkv = c->n_kv_heads, hd = c->head_dim;
    const int F = c->ffn;
    if (l < 0 || l >= c->n_layers || pos < 0 || pos >= cap || nh % nkv || hd % 2) return -1;
    const int group = nh / nkv;
    const double scale = 1.0 / sqrt((double)hd);
    double* xn = malloc(sizeof(double) * H);
    double* q = malloc(sizeof(double) * nh * hd);
    double* k = malloc(sizeof(double) * nkv * hd);
    double* v = malloc(sizeof(double) * nkv * hd);
    double* att = malloc(sizeof(double) * nh * hd);
    double* o = malloc(sizeof(double) * H);
    double* g = malloc(sizeof(double) * F);
    double* u = malloc(sizeof(double) * F);
    double* act = malloc(sizeof(double) * F);

    /* attn_norm, then the q/k/v projections of the fp16 normed row. */
    kdo_rmsnorm_f16(x, w->attn_norm[l], H, c->rms_eps, xn);
    kdo_matvec_q8_0(w->wq[l], nh * hd, H, xn, q);
    kdo_matvec_q8_0(w->wk[l], nkv * hd, H, xn, k);
    kdo_matvec_q8_0(w->wv[l], nkv * hd, H, xn, v);
    /* RoPE of q and k at this session's own position. */
    for (int h = 0; h < nh; ++h) kdo_rope_neox(q + h * hd, hd, pos, c->rope_theta);
    for (int h = 0; h < nkv; ++h) kdo_rope_neox(k + h * hd, hd, pos, c->rope_theta);
    /* KV append: row `pos` of this session's cache, stored as fp16, or (Q8_0
     * cache) the row as fp32, quantised. */
    if (!c->kv_q8_0) {
        for (int h = 0; h < nkv; ++h)
            for (int i = 0; i < hd; ++i) {
                Kl[((size_t)h * cap + pos) * hd + i] = kdo_double_to_half(k[h * hd + i]);
                Vl[((size_t)h * cap + pos) * hd + i] = kdo_double_to_half(v[h * hd + i]);
            }
    } else {
        float* rowf = malloc(sizeof(float) * hd);
        for (int h = 0; h < nkv; ++h) {
            for (int i = 0; i < hd; ++i) rowf[i] = (float)k[h * hd + i];
            kdo_q8_0_quantize_f32(rowf, hd, Kq + ((size_t)h * cap + pos) * rb);
            for (int i = 0; i < hd; ++i) rowf[i] = (float)v[h * hd + i];
            kdo_q8_0_quantize_f32(rowf, hd, Vq + ((size_t)h * cap + pos) * rb);
        }
        free(rowf);
    }
    /* Attention over keys 0..pos (t_kv = pos + 1), GQA head mapping h -> h / group. */
#pragma omp parallel for schedule(static)
    for (int h = 0; h < nh; ++h) {
        int kh = h / group;
        if (!c->kv_q8_0)
            kdo_attention_head(q + h * hd, Kl + (size_t)kh * cap * hd, Vl + (size_t)kh * cap * hd,
                               pos + 1, hd, hd, scale, att + h * hd);
        else
            kdo_attention_head_q8(q + h * hd, Kq + (size_t)kh * cap * rb, Vq + (size_t)kh * cap * rb,
                                  pos + 1, hd, (int64_t)rb, scale, att + h * hd);
    }
    for (int i = 0; i < nh * hd; ++i) att[i] = round_half(att[i]);
    /* o-projection and residual add (fp32 residual). */
    kdo_matvec_q8_0(w->wo[l], H, nh * hd, att, o);
    for (int i = 0; i < H; ++i) x[i] = round_float(x[i] + o[i]);
    /* ffn_norm, SwiGLU, down-projection, residual add. */
    kdo_rmsnorm_f16(x, w->ffn_norm[l], H, c->rms_eps, xn);
    kdo_matvec_q8_0(w->w_gate[l], F, H, xn, g);
    kdo_matvec_q8_0(w->w_up[l], F, H, xn, u);
    for (int i = 0; i < F; ++i) act[i] = round_half(kdo_silu(g[i]) * u[i]);
    kdo_matvec_q8_0(w->w_down[l], H, F, act, o);
    for (int i = 0; i < H; ++i) x[i] = round_float(x[i] + o[i]);

    free(xn); free(q); free(k); free(v); free(att); free(o); free(g); free(u); free(act);
    return 0;
}

/* One session, one step.  k_cache / v_cache are the session's caches,
 * [n_layers][n_kv][cap] rows (fp16 [hd], or Q8_0 blocks); rows 0..pos-1 hold its
 * history, row `pos` is overwritten with this step's key/value, rows beyond pos
 * are never read.
 * logits: [vocab] fp32.  hidden: NULL or [n_layers+1][hidden] fp32, the residual
 * after the embedding and after every layer. */
KDO_EXPORT int32_t kdo_session_step(const kdo_config* c, const kdo_weights* w,
                                    int32_t token, int32_t pos,
                                    void* k_cache, void* v_cache, int32_t cap,
                                    float* logits, float* hidden) {
    const int H = c->hidden, nkv = c->n_kv_heads;
    const size_t layer_bytes = (size_t)nkv * cap * kv_row_bytes(c);
    const int V = c->vocab, L = c->n_layers;
    if (token < 0 || token >= V || pos < 0 || pos >= cap) return -1;
    double* x = malloc(sizeof(double) * H);
    double* xn = malloc(sizeof(double) * H);
    double* lg = malloc(sizeof(double) * V);

    /* Embedding: the token's Q8_0 row, dequantised (exact in fp32). */
    kdo_q8_0_dequant_row(w->tok_embd + (size_t)token * (H / QK) * QB, H, x);
    for (int i = 0; i < H; ++i) x[i] = round_float(x[i]);
    if (hidden) for (int i = 0; i < H; ++i) hidden[i] = (float)x[i];

    int32_t rc = 0;
    for (int l = 0; l < L && rc == 0; ++l) {
        rc = kdo_layer_step(c, w, l, pos, (uint8_t*)k_cache + (size_t)l * layer_bytes,
                            (uint8_t*)v_cache + (size_t)l * layer_bytes, cap, x);
        if (hidden) for (int i = 0; i < H; ++i) hidden[(size_t)(l + 1) * H + i] = (float)x[i];
    }
    if (rc == 0) {
        /* Head: output_norm, lm_head, fp32 logits. */
        kdo_rmsnorm_f16(x, w->output_norm, H, c->rms_eps, xn);
        kdo_matvec_q8_0(w->output, V, H, xn, lg);
        for (int i = 0; i < V; ++i) logits[i] = (float)lg[i];
    }
    free(x); free(xn); free(lg);
    return rc;
}

/* B sessions, one step each: the batched step is B independent single-session
 * steps (the exactness contract).  Per-session arrays: k_caches[b], v_caches[b].
 * logits [B][vocab]; hidden NULL or [B][n_layers+1][hidden]; argmax [B]. */
KDO_EXPORT int32_t kdo_decode_step(const kdo_config* c, const kdo_weights* w, int32_t B,
                                   const int32_t* tokens, const int32_t* positions,
                                   void* const* k_caches, void* const* v_caches,
                                   int32_t cap, float* logits, float* hidden, int32_t* argmax) {
    for (int b = 0; b < B; ++b) {
        float* lg = logits + (size_t)b * c->vocab;
        float* hb = hidden ? hidden + (size_t)b * (c->n_layers + 1) * c->hidden : NULL;
        int32_t rc = kdo_session_step(c, w, tokens[b], positions[b], k_caches[b], v_caches[b],
                                      cap, lg, hb);
        if (rc) return rc;
        if (argmax) argmax[b] = kdo_argmax_f32(lg, c->vocab);
    }
    return 0;
}
