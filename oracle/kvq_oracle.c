/*
 * kvq_oracle.c -- the oracle: a plain, slow, single-threaded CPU statement of
 * what the INT4 group-quantized paged KV cache computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path
 * (the CUDA library and its Python binding) never includes, links or calls
 * anything here, and nothing here includes the product's headers: the layout
 * below is restated from the specification in prose, not shared code.
 *
 * Sources (web pages, cited by title and section):
 *  [Q] "4-bit KV cache compression" (lpnh.cn/news/2042373), section 2.1
 *      "symmetric uniform quantization, one scale per group":
 *      amax = max |x| over a group, scale = amax / 7, an all-zero group takes
 *      scale 1, q = round(x / scale) clamped to [-7, 7], dequant = q * scale.
 *      Section 2.2: storage bits per element 4 + 16/G; K grouped at 64 and V
 *      at 128 along the last (head) dimension.
 *  [M] "AI inference tuning: KV Cache optimisation and memory management"
 *      (bxzpzcl.cn/news/2871434), section 3.1 (KVCacheManager: fixed pages of
 *      page_size tokens, ceil(n / page_size) pages per request) and section
 *      3.2 (scaled dot-product attention with scale = head_dim^-0.5, softmax,
 *      then weights @ V; GQA repeats each KV head over n_rep = Hq / Hkv
 *      consecutive query heads).
 *  [S] "LLM long-context inference: managing the KV cache with an INT4 state
 *      machine" (pwwt.cn/news/4219524), section 2 (KV bytes per token
 *      2 * layers * heads * head_dim * dtype_size) and section 5 step 5
 *      (the inference layer reads INT4 directly and dequantizes inside the
 *      operator).
 *
 * Conventions the pages leave open, fixed by the workload statement:
 *  - the scale is computed as fp32 amax / 7.0f and then rounded to fp16
 *    (round-to-nearest-even); the zero test is made on that fp16 value;
 *  - codes are clamp(rne(fp32(x) / fp32(scale16)), -7, 7), the division an
 *    IEEE fp32 division, the rounding half-to-even;
 *  - a code c is stored as the nibble c + 8; byte j of a row holds the code of
 *    element 2j in its low nibble and element 2j+1 in its high nibble.
 *
 * Paged layout (one block per (page, kv-head); block index page*Hkv + h):
 *    K codes   P rows x d/2 bytes        (row = token slot in the page)
 *    V codes   P rows x d/2 bytes
 *    K scales  P rows x d/Gk fp16, little-endian
 *    V scales  P rows x d/Gv fp16
 *    zero padding up to a multiple of 16 bytes.
 * Token position t of sequence b lives in page block_table[b*max_blocks + t/P],
 * slot t % P.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -shared -fPIC.
 * Contraction is off so every fp32 operation rounds exactly once.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ERANGE 2

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 <-> binary32 / binary64, written from the format's      */
/* definition: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.     */
/* ------------------------------------------------------------------------ */

/* Round v / 2^s to an integer, ties to even (s >= 1). */
static uint64_t shift_right_rne(uint64_t v, int s) {
    if (s >= 64) return 0;
    uint64_t q = v >> s;
    uint64_t rem = v & ((((uint64_t)1) << s) - 1);
    uint64_t half = ((uint64_t)1) << (s - 1);
    if (rem > half || (rem == half && (q & 1))) q += 1;
    return q;
}

uint16_t kvq_oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u) /* infinity or NaN */
        return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x0200u : 0u));
    if (ax < 0x00800000u) /* fp32 zero or subnormal: below 2^-126, far under half the smallest fp16 subnormal */
        return sign;
    int e = (int)(ax >> 23) - 127;              /* value = M * 2^(e-23) */
    uint64_t M = (uint64_t)((ax & 0x7fffffu) | 0x800000u);
    if (e >= -14) {
        /* normal fp16 candidate: keep 11 significant bits */
        uint64_t m16 = shift_right_rne(M, 13);
        if (m16 == 2048) { m16 = 1024; e += 1; }
        if (e > 15) return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(m16 - 1024));
    }
    /* subnormal fp16: value / 2^-24 = M * 2^(e+1), rounded to an integer k in [0, 1024] */
    int s = -(e + 1);
    uint64_t k = shift_right_rne(M, s);
    return (uint16_t)(sign | (uint16_t)k); /* k == 1024 is exactly the smallest normal */
}

double kvq_oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)fr, -24);
    else if (ex == 31)
        v = fr ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fr), ex - 25);
    return sign ? -v : v;
}

float kvq_oracle_f16_to_f32(uint16_t h) { return (float)kvq_oracle_f16_to_f64(h); }

/* Array forms of the two conversions (used to check them against other implementations in bulk). */
void kvq_oracle_f32_to_f16_array(const float *x, uint16_t *out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = kvq_oracle_f32_to_f16(x[i]);
}
void kvq_oracle_f16_to_f64_array(const uint16_t *h, double *out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = kvq_oracle_f16_to_f64(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Sizes                                                                      */
/* ------------------------------------------------------------------------ */

/* Bytes of one (page, kv-head) block, per the layout in the file header. */
size_t kvq_oracle_block_bytes(int head_dim, int page_size, int group_k, int group_v) {
    size_t codes = (size_t)page_size * (size_t)head_dim;                 /* K and V: P*d/2 each */
    size_t scales = 2u * (size_t)page_size * (size_t)(head_dim / group_k + head_dim / group_v);
    size_t raw = codes + scales;
    return (raw + 15u) / 16u * 16u;
}

/* FP16 KV bytes: 2 (K and V) * layers * kv_heads * head_dim * tokens * 2 bytes
 * ([S] section 2; [Q] section 1.2 with S*B tokens). */
double kvq_oracle_fp16_kv_bytes(int layers, int kv_heads, int head_dim, double tokens) {
    return 2.0 * layers * kv_heads * head_dim * tokens * 2.0;
}

/* ------------------------------------------------------------------------ */
/* Quantization of one group ([Q] section 2.1)                                */
/* ------------------------------------------------------------------------ */

/* x: G fp16 values.  codes: G signed codes in [-7, 7].  *scale16: fp16 bits. */
void kvq_oracle_quantize_group(const uint16_t *x, int G, int8_t *codes, uint16_t *scale16) {
    float amax = 0.0f;
    for (int i = 0; i < G; ++i) {
        float a = fabsf(kvq_oracle_f16_to_f32(x[i]));
        if (a > amax) amax = a;
    }
    float s32 = amax / 7.0f;
    uint16_t s16 = kvq_oracle_f32_to_f16(s32);
    if ((s16 & 0x7fffu) == 0) s16 = 0x3c00u; /* an all-zero group (or a scale that rounds to zero) gets 1 */
    float s = kvq_oracle_f16_to_f32(s16);
    for (int i = 0; i < G; ++i) {
        float q = kvq_oracle_f16_to_f32(x[i]) / s;
        float r = nearbyintf(q); /* default rounding mode: to nearest, ties to even */
        if (r > 7.0f) r = 7.0f;
        if (r < -7.0f) r = -7.0f;
        codes[i] = (int8_t)r;
    }
    *scale16 = s16;
}

/* ------------------------------------------------------------------------ */
/* Paged pool access                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int Hkv, d, P, Gk, Gv, num_pages;
    size_t block;
} layout_t;

static int make_layout(layout_t *L, int Hkv, int d, int P, int Gk, int Gv, int num_pages) {
    if (Hkv <= 0 || d <= 0 || P <= 0 || Gk <= 0 || Gv <= 0 || num_pages <= 0) return ORACLE_EINVAL;
    if (d % 2 || d % Gk || d % Gv) return ORACLE_EINVAL;
    L->Hkv = Hkv; L->d = d; L->P = P; L->Gk = Gk; L->Gv = Gv; L->num_pages = num_pages;
    L->block = kvq_oracle_block_bytes(d, P, Gk, Gv);
    return ORACLE_OK;
}

static uint8_t *block_ptr(const layout_t *L, uint8_t *pool, int page, int h) {
    return pool + ((size_t)page * (size_t)L->Hkv + (size_t)h) * L->block;
}
static uint8_t *k_codes_row(const layout_t *L, uint8_t *blk, int slot) { return blk + (size_t)slot * (size_t)(L->d / 2); }
static uint8_t *v_codes_row(const layout_t *L, uint8_t *blk, int slot) {
    return blk + (size_t)L->P * (size_t)(L->d / 2) + (size_t)slot * (size_t)(L->d / 2);
}
static uint8_t *k_scales_row(const layout_t *L, uint8_t *blk, int slot) {
    return blk + (size_t)L->P * (size_t)L->d + (size_t)slot * (size_t)(L->d / L->Gk) * 2u;
}
static uint8_t *v_scales_row(const layout_t *L, uint8_t *blk, int slot) {
    return blk + (size_t)L->P * (size_t)L->d + (size_t)L->P * (size_t)(L->d / L->Gk) * 2u +
           (size_t)slot * (size_t)(L->d / L->Gv) * 2u;
}

static void put_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Quantize one row of d fp16 values in groups of G; write codes (d/2 bytes) and scales (d/G fp16). */
static void quantize_row(const uint16_t *x, int d, int G, uint8_t *codes_row, uint8_t *scales_row) {
    int8_t c[256];
    for (int g0 = 0; g0 < d; g0 += G) {
        uint16_t s16;
        kvq_oracle_quantize_group(x + g0, G, c + g0, &s16);
        put_u16(scales_row + (size_t)(g0 / G) * 2u, s16);
    }
    for (int j = 0; j < d / 2; ++j) {
        unsigned lo = (unsigned)(c[2 * j] + 8);
        unsigned hi = (unsigned)(c[2 * j + 1] + 8);
        codes_row[j] = (uint8_t)(lo | (hi << 4));
    }
}

/* Dequantize one row: element i = (nibble_i - 8) * scale[i / G], exact in fp32. */
static void dequant_row(const uint8_t *codes_row, const uint8_t *scales_row, int d, int G, float *out) {
    for (int i = 0; i < d; ++i) {
        uint8_t byte = codes_row[i / 2];
        int nib = (i & 1) ? (byte >> 4) : (byte & 0x0f);
        float s = kvq_oracle_f16_to_f32(get_u16(scales_row + (size_t)(i / G) * 2u));
        out[i] = (float)(nib - 8) * s;
    }
}

/*
 * Quantize-on-append.  k, v: fp16 [B, n_new, Hkv, d] contiguous.  For every b
 * and every t < n_new the token is written at position start_pos[b] + t.
 * Returns ORACLE_ERANGE (and writes nothing further) if a position falls
 * outside the block table or a page id is outside [0, num_pages).
 */
int kvq_oracle_quantize_append(uint8_t *pool, const uint16_t *k, const uint16_t *v,
                               const int32_t *block_table, int max_blocks, const int32_t *start_pos,
                               int B, int n_new, int Hkv, int d, int P, int Gk, int Gv, int num_pages) {
    layout_t L;
    if (make_layout(&L, Hkv, d, P, Gk, Gv, num_pages) || d > 256 || B < 0 || n_new < 0) return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < n_new; ++t) {
            long pos = (long)start_pos[b] + t;
            if (pos < 0 || pos / P >= max_blocks) return ORACLE_ERANGE;
            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
            int slot = (int)(pos % P);
            for (int h = 0; h < Hkv; ++h) {
                size_t off = (((size_t)b * (size_t)n_new + (size_t)t) * (size_t)Hkv + (size_t)h) * (size_t)d;
                uint8_t *blk = block_ptr(&L, pool, page, h);
                quantize_row(k + off, d, Gk, k_codes_row(&L, blk, slot), k_scales_row(&L, blk, slot));
                quantize_row(v + off, d, Gv, v_codes_row(&L, blk, slot), v_scales_row(&L, blk, slot));
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Dequantize positions [start, start+n) of sequence b into out_k, out_v laid
 * out [n, Hkv, d].  out_fp16 != 0: fp16 bits (RNE of the exact fp32 product);
 * otherwise fp32.
 */
int kvq_oracle_dequantize(const uint8_t *pool, const int32_t *block_table, int max_blocks, int b, int start,
                          int n, void *out_k, void *out_v, int out_fp16,
                          int Hkv, int d, int P, int Gk, int Gv, int num_pages) {
    layout_t L;
    if (make_layout(&L, Hkv, d, P, Gk, Gv, num_pages) || d > 256 || start < 0 || n < 0) return ORACLE_EINVAL;
    float rk[256], rv[256];
    for (int t = 0; t < n; ++t) {
        long pos = (long)start + t;
        if (pos / P >= max_blocks) return ORACLE_ERANGE;
        int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
        if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
        int slot = (int)(pos % P);
        for (int h = 0; h < Hkv; ++h) {
            uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, h);
            dequant_row(k_codes_row(&L, blk, slot), k_scales_row(&L, blk, slot), d, Gk, rk);
            dequant_row(v_codes_row(&L, blk, slot), v_scales_row(&L, blk, slot), d, Gv, rv);
            size_t off = ((size_t)t * (size_t)Hkv + (size_t)h) * (size_t)d;
            for (int i = 0; i < d; ++i) {
                if (out_fp16) {
                    ((uint16_t *)out_k)[off + i] = kvq_oracle_f32_to_f16(rk[i]);
                    ((uint16_t *)out_v)[off + i] = kvq_oracle_f32_to_f16(rv[i]);
                } else {
                    ((float *)out_k)[off + i] = rk[i];
                    ((float *)out_v)[off + i] = rv[i];
                }
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Decode attention over the quantized cache, in fp64 ([M] section 3.2 with the
 * dequantization of [Q] section 2.1 inside, as [S] section 5 step 5 puts it).
 * q: fp16 [B, Hq, d].  Query head hq reads KV head hq / (Hq / Hkv).  Sequence
 * b attends to positions 0 .. seq_lens[b]-1 (the appended token included).
 * out: fp64 [B, Hq, d].  A sequence of length 0 yields zeros.
 */
int kvq_oracle_decode_attention(const uint8_t *pool, const uint16_t *q, const int32_t *block_table,
                                int max_blocks, const int32_t *seq_lens, int B, int Hq, double softmax_scale,
                                double *out, int Hkv, int d, int P, int Gk, int Gv, int num_pages) {
    layout_t L;
    if (make_layout(&L, Hkv, d, P, Gk, Gv, num_pages) || d > 256 || Hq <= 0 || Hq % Hkv) return ORACLE_EINVAL;
    int n_rep = Hq / Hkv;
    float rk[256], rv[256];
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0 || (len + P - 1) / P > max_blocks) return ORACLE_ERANGE;
        for (int hq = 0; hq < Hq; ++hq) {
            int h = hq / n_rep;
            const uint16_t *qrow = q + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            double *o = out + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (len == 0) continue;
            /* pass 1: logits and their maximum */
            double zmax = -INFINITY;
            for (int t = 0; t < len; ++t) {
                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
                uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, h);
                dequant_row(k_codes_row(&L, blk, t % P), k_scales_row(&L, blk, t % P), d, Gk, rk);
                double z = 0.0;
                for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * (double)rk[i];
                z *= softmax_scale;
                if (z > zmax) zmax = z;
            }
            /* pass 2: softmax weights and the weighted sum of values */
            double l = 0.0;
            for (int t = 0; t < len; ++t) {
                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, h);
                dequant_row(k_codes_row(&L, blk, t % P), k_scales_row(&L, blk, t % P), d, Gk, rk);
                dequant_row(v_codes_row(&L, blk, t % P), v_scales_row(&L, blk, t % P), d, Gv, rv);
                double z = 0.0;
                for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * (double)rk[i];
                z *= softmax_scale;
                double p = exp(z - zmax);
                l += p;
                for (int i = 0; i < d; ++i) o[i] += p * (double)rv[i];
            }
            for (int i = 0; i < d; ++i) o[i] /= l;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Decode attention with a sliding window and sink tokens ([M] section 3.2, */
/* SlidingWindowAttention): query position i sees keys max(0, i - W + 1)     */
/* .. i and, when S > 0, the first S positions 0 .. S-1.  The decode query   */
/* is the last position i = len - 1, so the visible keys are                 */
/* [max(0, len - W), len) together with [0, min(S, len)).  window <= 0       */
/* means no window (every position is visible, as in plain decode            */
/* attention); sinks <= 0 means none.                                        */
/* ------------------------------------------------------------------------ */
static int visible_pos(int t, int len, int window, int sinks) {
    if (window <= 0) return 1;
    if (t >= len - window) return 1;
    return sinks > 0 && t < sinks;
}

int kvq_oracle_decode_attention_window(const uint8_t *pool, const uint16_t *q, const int32_t *block_table,
                                       int max_blocks, const int32_t *seq_lens, int B, int Hq, double softmax_scale,
                                       int window, int sinks, double *out, int Hkv, int d, int P, int Gk, int Gv,
                                       int num_pages) {
    layout_t L;
    if (make_layout(&L, Hkv, d, P, Gk, Gv, num_pages) || d > 256 || Hq <= 0 || Hq % Hkv) return ORACLE_EINVAL;
    int n_rep = Hq / Hkv;
    float rk[256], rv[256];
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0 || (len + P - 1) / P > max_blocks) return ORACLE_ERANGE;
        for (int hq = 0; hq < Hq; ++hq) {
            int kv = hq / n_rep;
            const uint16_t *qrow = q + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            double *o = out + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (len == 0) continue;
            /* pass 1: logits of the visible positions and their maximum */
            double zmax = -INFINITY;
            for (int t = 0; t < len; ++t) {
                if (!visible_pos(t, len, window, sinks)) continue;
                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
                uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, kv);
                dequant_row(k_codes_row(&L, blk, t % P), k_scales_row(&L, blk, t % P), d, Gk, rk);
                double z = 0.0;
                for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * (double)rk[i];
                z *= softmax_scale;
                if (z > zmax) zmax = z;
            }
            /* pass 2: softmax weights over the visible positions and the weighted sum of values */
            double l = 0.0;
            for (int t = 0; t < len; ++t) {
                if (!visible_pos(t, len, window, sinks)) continue;
                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, kv);
                dequant_row(k_codes_row(&L, blk, t % P), k_scales_row(&L, blk, t % P), d, Gk, rk);
                dequant_row(v_codes_row(&L, blk, t % P), v_scales_row(&L, blk, t % P), d, Gv, rv);
                double z = 0.0;
                for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * (double)rk[i];
                z *= softmax_scale;
                double w = exp(z - zmax);
                l += w;
                for (int i = 0; i < d; ++i) o[i] += w * (double)rv[i];
            }
            for (int i = 0; i < d; ++i) o[i] /= l;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The FP16 cache of the latency comparison ([S] section 7.4: FP16 baseline, */
/* INT4 dequantized first and then attended, INT4 dequantized inside the     */
/* operator).  Pages as in [M] section 3.1: one block per (page, kv-head),   */
/* block index page*Hkv + h, holding K rows P x d fp16 and then V rows        */
/* P x d fp16 (little-endian), 4*P*d bytes.                                  */
/* ------------------------------------------------------------------------ */
size_t kvq_oracle_fp16_block_bytes(int head_dim, int page_size) {
    if (head_dim <= 0 || page_size <= 0) return 0;
    return (size_t)4 * (size_t)page_size * (size_t)head_dim;
}

static uint8_t *fp16_row(uint8_t *pool16, int Hkv, int d, int P, int page, int h, int is_v, int slot) {
    size_t blk = ((size_t)page * (size_t)Hkv + (size_t)h) * ((size_t)4 * (size_t)P * (size_t)d);
    return pool16 + blk + ((size_t)is_v * (size_t)P + (size_t)slot) * (size_t)d * 2u;
}

/* Store fp16 K and V rows [B, n_new, Hkv, d] at positions start_pos[b] + t. */
int kvq_oracle_fp16_append(uint8_t *pool16, const uint16_t *k, const uint16_t *v, const int32_t *block_table,
                           int max_blocks, const int32_t *start_pos, int B, int n_new, int Hkv, int d, int P,
                           int num_pages) {
    if (Hkv <= 0 || d <= 0 || P <= 0 || B < 0 || n_new < 0) return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < n_new; ++t) {
            long pos = (long)start_pos[b] + t;
            if (pos < 0 || pos / P >= max_blocks) return ORACLE_ERANGE;
            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
            int slot = (int)(pos % P);
            for (int h = 0; h < Hkv; ++h) {
                size_t src = (((size_t)b * (size_t)n_new + (size_t)t) * (size_t)Hkv + (size_t)h) * (size_t)d;
                uint8_t *kr = fp16_row(pool16, Hkv, d, P, page, h, 0, slot);
                uint8_t *vr = fp16_row(pool16, Hkv, d, P, page, h, 1, slot);
                for (int i = 0; i < d; ++i) {
                    put_u16(kr + 2 * i, k[src + i]);
                    put_u16(vr + 2 * i, v[src + i]);
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Dequantize every position 0 .. seq_lens[b]-1 of the INT4 pool into the FP16
   pool, at the same page ids and slots: each value is the fp16 RNE of
   (nibble - 8) * scale ([Q] section 2.1). */
int kvq_oracle_dequantize_to_fp16_pool(const uint8_t *pool, uint8_t *pool16, const int32_t *block_table,
                                       int max_blocks, const int32_t *seq_lens, int B, int Hkv, int d, int P,
                                       int Gk, int Gv, int num_pages) {
    layout_t L;
    if (make_layout(&L, Hkv, d, P, Gk, Gv, num_pages) || d > 256) return ORACLE_EINVAL;
    float rk[256], rv[256];
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0 || (len + P - 1) / P > max_blocks) return ORACLE_ERANGE;
        for (int t = 0; t < len; ++t) {
            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
            for (int h = 0; h < Hkv; ++h) {
                uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, h);
                dequant_row(k_codes_row(&L, blk, t % P), k_scales_row(&L, blk, t % P), d, Gk, rk);
                dequant_row(v_codes_row(&L, blk, t % P), v_scales_row(&L, blk, t % P), d, Gv, rv);
                uint8_t *kr = fp16_row(pool16, Hkv, d, P, page, h, 0, t % P);
                uint8_t *vr = fp16_row(pool16, Hkv, d, P, page, h, 1, t % P);
                for (int i = 0; i < d; ++i) {
                    put_u16(kr + 2 * i, kvq_oracle_f32_to_f16(rk[i]));
                    put_u16(vr + 2 * i, kvq_oracle_f32_to_f16(rv[i]));
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Decode attention over the FP16 cache, in fp64 ([M] section 3.2): as
   kvq_oracle_decode_attention with the K and V rows read as fp16. */
int kvq_oracle_fp16_decode_attention(const uint8_t *pool16, const uint16_t *q, const int32_t *block_table,
                                     int max_blocks, const int32_t *seq_lens, int B, int Hq, double softmax_scale,
                                     double *out, int Hkv, int d, int P, int num_pages) {
    if (Hkv <= 0 || d <= 0 || P <= 0 || Hq <= 0 || Hq % Hkv) return ORACLE_EINVAL;
    int rep = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0 || (len + P - 1) / P > max_blocks) return ORACLE_ERANGE;
        for (int hq = 0; hq < Hq; ++hq) {
            int kvh = hq / rep;
            const uint16_t *qrow = q + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            double *o = out + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (len == 0) continue;
            double zmax = -INFINITY;
            for (int t = 0; t < len; ++t) {
                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
                const uint8_t *kr = fp16_row((uint8_t *)pool16, Hkv, d, P, page, kvh, 0, t % P);
                double z = 0.0;
                for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * kvq_oracle_f16_to_f64(get_u16(kr + 2 * i));
                z *= softmax_scale;
                if (z > zmax) zmax = z;
            }
            double lsum = 0.0;
            for (int t = 0; t < len; ++t) {
                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                const uint8_t *kr = fp16_row((uint8_t *)pool16, Hkv, d, P, page, kvh, 0, t % P);
                const uint8_t *vr = fp16_row((uint8_t *)pool16, Hkv, d, P, page, kvh, 1, t % P);
                double z = 0.0;
                for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * kvq_oracle_f16_to_f64(get_u16(kr + 2 * i));
                z *= softmax_scale;
                double wz = exp(z - zmax);
                lsum += wz;
                for (int i = 0; i < d; ++i) o[i] += wz * kvq_oracle_f16_to_f64(get_u16(vr + 2 * i));
            }
            for (int i = 0; i < d; ++i) o[i] /= lsum;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Mixed precision ([S] section 8.3, item 1: quantize the KV of old tokens   */
/* to INT4 first and keep recent tokens in FP16): for a sequence of len      */
/* positions, position t < len - residual is read from the INT4 pool, and    */
/* t >= len - residual from the FP16 pool (same page table layout each, own  */
/* block tables).  Plain decode attention over all len positions, in fp64.   */
/* ------------------------------------------------------------------------ */
int kvq_oracle_mixed_decode_attention(const uint8_t *pool, const int32_t *block_table, int max_blocks,
                                      const uint8_t *pool16, const int32_t *block_table16, int max_blocks16,
                                      const uint16_t *q, const int32_t *seq_lens, int B, int Hq, int residual,
                                      double softmax_scale, double *out, int Hkv, int d, int P, int Gk, int Gv,
                                      int num_pages, int num_pages16) {
    layout_t L;
    if (make_layout(&L, Hkv, d, P, Gk, Gv, num_pages) || d > 256 || Hq <= 0 || Hq % Hkv || residual < 0)
        return ORACLE_EINVAL;
    int grp = Hq / Hkv;
    float rk[256], rv[256];
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0) return ORACLE_ERANGE;
        int split = len - residual > 0 ? len - residual : 0;  /* first FP16 position */
        if ((split + P - 1) / P > max_blocks || (len + P - 1) / P > max_blocks16) return ORACLE_ERANGE;
        for (int hq = 0; hq < Hq; ++hq) {
            int hk = hq / grp;
            const uint16_t *qrow = q + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            double *o = out + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (len == 0) continue;
            double zmax = -INFINITY, lsum = 0.0;
            for (int pass = 0; pass < 2; ++pass) {
                for (int t = 0; t < len; ++t) {
                    double z = 0.0;
                    const uint8_t *vrow16 = 0;
                    if (t < split) {
                        int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                        if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
                        uint8_t *blk = block_ptr(&L, (uint8_t *)pool, page, hk);
                        dequant_row(k_codes_row(&L, blk, t % P), k_scales_row(&L, blk, t % P), d, Gk, rk);
                        dequant_row(v_codes_row(&L, blk, t % P), v_scales_row(&L, blk, t % P), d, Gv, rv);
                        for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * (double)rk[i];
                    } else {
                        int page = block_table16[(size_t)b * (size_t)max_blocks16 + (size_t)(t / P)];
                        if (page < 0 || page >= num_pages16) return ORACLE_ERANGE;
                        const uint8_t *kr = fp16_row((uint8_t *)pool16, Hkv, d, P, page, hk, 0, t % P);
                        vrow16 = fp16_row((uint8_t *)pool16, Hkv, d, P, page, hk, 1, t % P);
                        for (int i = 0; i < d; ++i)
                            z += kvq_oracle_f16_to_f64(qrow[i]) * kvq_oracle_f16_to_f64(get_u16(kr + 2 * i));
                    }
                    z *= softmax_scale;
                    if (pass == 0) {
                        if (z > zmax) zmax = z;
                        continue;
                    }
                    double e = exp(z - zmax);
                    lsum += e;
                    for (int i = 0; i < d; ++i)
                        o[i] += e * (vrow16 ? kvq_oracle_f16_to_f64(get_u16(vrow16 + 2 * i)) : (double)rv[i]);
                }
            }
            for (int i = 0; i < d; ++i) o[i] /= lsum;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* INT8 per-row codec ([M] section 3.1, KVCacheQuantizer.quantize_int8 /    */
/* dequantize_int8): one scale per row (token, kv head) over head_dim,       */
/* scale = amax / 127 clamped below at 1e-8, code = round(x / scale)         */
/* clamped to [-128, 127], value = code * scale.  The page computes in the   */
/* input's dtype; here every step is fp32 (amax is exact from fp16; the      */
/* division and the product round once to nearest), the rounding is         */
/* half-to-even, and the scale is stored as fp32.                           */
/* Block (page, kv head), index page*Hkv + h, 2*P*d + 8*P bytes: K codes     */
/* P x d int8, V codes P x d int8, K scales P fp32, V scales P fp32 (little- */
/* endian).                                                                  */
/* ------------------------------------------------------------------------ */
size_t kvq_oracle_int8_block_bytes(int head_dim, int page_size) {
    if (head_dim <= 0 || page_size <= 0) return 0;
    return (size_t)2 * (size_t)page_size * (size_t)head_dim + (size_t)8 * (size_t)page_size;
}

static uint8_t *int8_block(uint8_t *pool8, int Hkv, int d, int P, int page, int h) {
    return pool8 + ((size_t)page * (size_t)Hkv + (size_t)h) * kvq_oracle_int8_block_bytes(d, P);
}

static void put_f32(uint8_t *p, float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    p[0] = (uint8_t)u; p[1] = (uint8_t)(u >> 8); p[2] = (uint8_t)(u >> 16); p[3] = (uint8_t)(u >> 24);
}
static float get_f32(const uint8_t *p) {
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* one row of d fp16 values -> d int8 codes and the fp32 scale */
void kvq_oracle_int8_quantize_row(const uint16_t *x, int d, int8_t *codes, float *scale_out) {
    float amax = 0.0f;
    for (int i = 0; i < d; ++i) {
        float a = fabsf(kvq_oracle_f16_to_f32(x[i]));
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    if (s < 1e-8f) s = 1e-8f;
    for (int i = 0; i < d; ++i) {
        float r = nearbyintf(kvq_oracle_f16_to_f32(x[i]) / s);
        if (r > 127.0f) r = 127.0f;
        if (r < -128.0f) r = -128.0f;
        codes[i] = (int8_t)r;
    }
    *scale_out = s;
}

int kvq_oracle_int8_quantize_append(uint8_t *pool8, const uint16_t *k, const uint16_t *v, const int32_t *block_table,
                                    int max_blocks, const int32_t *start_pos, int B, int n_new, int Hkv, int d, int P,
                                    int num_pages) {
    if (Hkv <= 0 || d <= 0 || d > 256 || P <= 0 || B < 0 || n_new < 0) return ORACLE_EINVAL;
    int8_t codes[256];
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < n_new; ++t) {
            long pos = (long)start_pos[b] + t;
            if (pos < 0 || pos / P >= max_blocks) return ORACLE_ERANGE;
            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
            int slot = (int)(pos % P);
            for (int h = 0; h < Hkv; ++h) {
                size_t src = (((size_t)b * (size_t)n_new + (size_t)t) * (size_t)Hkv + (size_t)h) * (size_t)d;
                uint8_t *blk = int8_block(pool8, Hkv, d, P, page, h);
                float sk, sv;
                kvq_oracle_int8_quantize_row(k + src, d, codes, &sk);
                memcpy(blk + (size_t)slot * (size_t)d, codes, (size_t)d);
                kvq_oracle_int8_quantize_row(v + src, d, codes, &sv);
                memcpy(blk + (size_t)P * (size_t)d + (size_t)slot * (size_t)d, codes, (size_t)d);
                put_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * (size_t)slot, sk);
                put_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot), sv);
            }
        }
    }
    return ORACLE_OK;
}

/* Dequantize positions [start, start+n) of sequence b: value = fp32(code * scale). */
int kvq_oracle_int8_dequantize(const uint8_t *pool8, const int32_t *block_table, int max_blocks, int b, int start,
                               int n, float *out_k, float *out_v, int Hkv, int d, int P, int num_pages) {
    if (Hkv <= 0 || d <= 0 || P <= 0 || start < 0 || n < 0) return ORACLE_EINVAL;
    for (int t = 0; t < n; ++t) {
        long pos = (long)start + t;
        if (pos / P >= max_blocks) return ORACLE_ERANGE;
        int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
        if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
        int slot = (int)(pos % P);
        for (int h = 0; h < Hkv; ++h) {
            const uint8_t *blk = int8_block((uint8_t *)pool8, Hkv, d, P, page, h);
            float sk = get_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * (size_t)slot);
            float sv = get_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot));
            size_t off = ((size_t)t * (size_t)Hkv + (size_t)h) * (size_t)d;
            for (int i = 0; i < d; ++i) {
                out_k[off + i] = (float)(int8_t)blk[(size_t)slot * (size_t)d + (size_t)i] * sk;
                out_v[off + i] = (float)(int8_t)blk[((size_t)P + (size_t)slot) * (size_t)d + (size_t)i] * sv;
            }
        }
    }
    return ORACLE_OK;
}

/* Decode attention over the INT8 cache, in fp64 ([M] section 3.2) over the dequantized rows. */
int kvq_oracle_int8_decode_attention(const uint8_t *pool8, const uint16_t *q, const int32_t *block_table,
                                     int max_blocks, const int32_t *seq_lens, int B, int Hq, double softmax_scale,
                                     double *out, int Hkv, int d, int P, int num_pages) {
    if (Hkv <= 0 || d <= 0 || d > 256 || P <= 0 || Hq <= 0 || Hq % Hkv) return ORACLE_EINVAL;
    int per = Hq / Hkv;
    float rk[256], rv[256];
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0 || (len + P - 1) / P > max_blocks) return ORACLE_ERANGE;
        for (int hq = 0; hq < Hq; ++hq) {
            int kh = hq / per;
            const uint16_t *qrow = q + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            double *o = out + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (len == 0) continue;
            double top = -INFINITY, den = 0.0;
            for (int pass = 0; pass < 2; ++pass) {
                for (int t = 0; t < len; ++t) {
                    int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                    if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
                    const uint8_t *blk = int8_block((uint8_t *)pool8, Hkv, d, P, page, kh);
                    int slot = t % P;
                    float sk = get_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * (size_t)slot);
                    float sv = get_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot));
                    for (int i = 0; i < d; ++i) {
                        rk[i] = (float)(int8_t)blk[(size_t)slot * (size_t)d + (size_t)i] * sk;
                        rv[i] = (float)(int8_t)blk[((size_t)P + (size_t)slot) * (size_t)d + (size_t)i] * sv;
                    }
                    double z = 0.0;
                    for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * (double)rk[i];
                    z *= softmax_scale;
                    if (pass == 0) {
                        if (z > top) top = z;
                        continue;
                    }
                    double e = exp(z - top);
                    den += e;
                    for (int i = 0; i < d; ++i) o[i] += e * (double)rv[i];
                }
            }
            for (int i = 0; i < d; ++i) o[i] /= den;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The rotated 4-bit codec ([L] "LARQL KV cache engines", engine three,      */
/* codec/turbo-quant: each K or V row of a head is rotated by a Walsh-       */
/* Hadamard transform and quantized with a Lloyd-Max codebook to 3 or 4     */
/* bits; head_dim must be a power of two; approximate, per-row cosine       */
/* about 0.9954 at 4 bits).  The page names the two steps only; the reading */
/* written out here (and restated independently by the CUDA library):       */
/*  - x_i = fp32(fp16 input), d = 128;                                       */
/*  - y = H x, H the unnormalised Sylvester-order Walsh-Hadamard matrix,     */
/*    computed by the fast transform: stages h = 1, 2, 4, .., d/2, each pair */
/*    (i, i+h) with (i & h) == 0 becoming (y_i + y_{i+h}, y_i - y_{i+h}),    */
/*    one fp32 rounding per addition;                                        */
/*  - sigma = sqrt(sum x_i^2) = the RMS of y (H H = d I), the squares and    */
/*    sums rounded to fp32 in a fixed tree: 32 partial sums of 4 elements    */
/*    ((x0^2 + x1^2) + (x2^2 + x3^2)) for elements 4l .. 4l+3, then for      */
/*    off = 16, 8, 4, 2, 1 every partial l becomes s_l + s_{l xor off};     */
/*  - u_i = y_i / sigma (fp32 division); the code of u_i is the number of   */
/*    thresholds T_1 < .. < T_15 with u_i >= T_j, T_j = fp32 of the midpoint */
/*    of Lloyd-Max levels j-1 and j (fp64) for the standard normal, 16      */
/*    levels; an all-zero row (sigma = 0) takes codes 0;                    */
/*  - stored: the codes as nibbles (element 2j in the low nibble of byte j) */
/*    and sigma as fp32;                                                     */
/*  - dequantized: x^ = H (sigma * c) / d, c_j = fp32 of level j.            */
/* Block (page, kv head), index page*Hkv + h, P*(d + 8) bytes: K codes      */
/* P x d/2, V codes P x d/2, K sigma P fp32, V sigma P fp32.                 */
/* ------------------------------------------------------------------------ */

static double std_normal_pdf(double t) {
    if (isinf(t)) return 0.0;
    return exp(-0.5 * t * t) / sqrt(2.0 * 3.14159265358979323846);
}
static double std_normal_cdf(double t) {
    if (isinf(t)) return t > 0 ? 1.0 : 0.0;
    return 0.5 * erfc(-t / sqrt(2.0));
}

/* Lloyd-Max quantizer of the standard normal with 2^bits levels (bits 1..5),
 * by Lloyd's alternation: the thresholds are the midpoints of adjacent levels,
 * each level the mean of the normal restricted to its cell,
 *   L_j = (pdf(T_j) - pdf(T_{j+1})) / (cdf(T_{j+1}) - cdf(T_j)),
 * iterated from evenly spaced levels until no level moves by more than
 * 1e-15.  The normal law is symmetric, and so is its quantizer: the levels are
 * then made exactly antisymmetric (level n-1-j set to (L_{n-1-j} - L_j) / 2 and
 * level j to its negation), which puts the middle threshold at exactly 0.
 * levels[2^bits] ascending; thresholds[2^bits - 1], thresholds[j-1] between
 * levels j-1 and j.  Returns the iteration count, or -1. */
int kvq_oracle_lloyd_max_normal(int bits, double *levels, double *thresholds) {
    if (bits < 1 || bits > 5) return -1;
    int n = 1 << bits;
    double lv[32], tb[33];
    for (int j = 0; j < n; ++j) lv[j] = -3.0 + 6.0 * (j + 0.5) / n;
    int it;
    for (it = 1; it <= 200000; ++it) {
        tb[0] = -INFINITY;
        tb[n] = INFINITY;
        for (int j = 1; j < n; ++j) tb[j] = 0.5 * (lv[j - 1] + lv[j]);
        double moved = 0.0;
        for (int j = 0; j < n; ++j) {
            double mass = std_normal_cdf(tb[j + 1]) - std_normal_cdf(tb[j]);
            double nl = (std_normal_pdf(tb[j]) - std_normal_pdf(tb[j + 1])) / mass;
            double dj = fabs(nl - lv[j]);
            if (dj > moved) moved = dj;
            lv[j] = nl;
        }
        if (moved <= 1e-15) break;
    }
    for (int j = 0; j < n / 2; ++j) {
        double a = 0.5 * (lv[n - 1 - j] - lv[j]);
        lv[j] = -a;
        lv[n - 1 - j] = a;
    }
    for (int j = 0; j < n; ++j) levels[j] = lv[j];
    for (int j = 1; j < n; ++j) thresholds[j - 1] = 0.5 * (lv[j - 1] + lv[j]);
    return it;
}

/* The fast Walsh-Hadamard transform in place, fp32, stage order h = 1, 2, .. */
void kvq_oracle_wht_f32(float *y, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; ++i)
            if ((i & h) == 0) {
                float a = y[i], b = y[i + h];
                y[i] = a + b;
                y[i + h] = a - b;
            }
}

/* The same transform in fp64. */
static void wht_f64(double *y, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; ++i)
            if ((i & h) == 0) {
                double a = y[i], b = y[i + h];
                y[i] = a + b;
                y[i + h] = a - b;
            }
}

size_t kvq_oracle_wht4_block_bytes(int head_dim, int page_size) {
    if (head_dim <= 0 || page_size <= 0) return 0;
    return (size_t)page_size * ((size_t)head_dim + 8);
}

/* fp32 codebook of the 4-bit codec: levels c_j and thresholds T_j */
static void wht4_tables(float *c, float *T) {
    static int ready = 0;
    static float cs[16], ts[15];
    if (!ready) {
        double lv[16], tb[15];
        kvq_oracle_lloyd_max_normal(4, lv, tb);
        for (int j = 0; j < 16; ++j) cs[j] = (float)lv[j];
        for (int j = 0; j < 15; ++j) ts[j] = (float)tb[j];
        ready = 1;
    }
    memcpy(c, cs, sizeof cs);
    memcpy(T, ts, sizeof ts);
}

void kvq_oracle_wht4_tables(float *levels16, float *thresholds15) { wht4_tables(levels16, thresholds15); }

/* one row of d = 128 fp16 values -> d/2 code bytes and sigma */
int kvq_oracle_wht4_quantize_row(const uint16_t *x, int d, uint8_t *codes, float *sigma_out) {
    if (d != 128) return ORACLE_EINVAL;
    float c[16], T[15], y[128], s[32];
    wht4_tables(c, T);
    for (int i = 0; i < d; ++i) y[i] = kvq_oracle_f16_to_f32(x[i]);
    for (int l = 0; l < 32; ++l) {
        float a0 = y[4 * l] * y[4 * l], a1 = y[4 * l + 1] * y[4 * l + 1];
        float a2 = y[4 * l + 2] * y[4 * l + 2], a3 = y[4 * l + 3] * y[4 * l + 3];
        s[l] = (a0 + a1) + (a2 + a3);
    }
    for (int off = 16; off > 0; off >>= 1) {
        float t[32];
        for (int l = 0; l < 32; ++l) t[l] = s[l] + s[l ^ off];
        memcpy(s, t, sizeof t);
    }
    float sigma = sqrtf(s[0]);
    kvq_oracle_wht_f32(y, d);
    memset(codes, 0, (size_t)d / 2);
    for (int i = 0; i < d; ++i) {
        int code = 0;
        if (sigma > 0.0f) {
            float u = y[i] / sigma;
            for (int j = 0; j < 15; ++j) code += u >= T[j];
        }
        codes[i / 2] |= (uint8_t)(code << (4 * (i & 1)));
    }
    *sigma_out = sigma;
    return ORACLE_OK;
}

/* x^ = H (sigma * c[code]) / d in fp64 */
static void wht4_dequant_row_f64(const uint8_t *codes, float sigma, int d, double *out) {
    float c[16], T[15];
    wht4_tables(c, T);
    for (int i = 0; i < d; ++i) {
        int code = (codes[i / 2] >> (4 * (i & 1))) & 15;
        out[i] = (double)(sigma * c[code]);
    }
    wht_f64(out, d);
    for (int i = 0; i < d; ++i) out[i] /= d;
}

static uint8_t *wht4_block(uint8_t *pool, int Hkv, int d, int P, int page, int h) {
    return pool + ((size_t)page * (size_t)Hkv + (size_t)h) * kvq_oracle_wht4_block_bytes(d, P);
}

int kvq_oracle_wht4_quantize_append(uint8_t *pool, const uint16_t *k, const uint16_t *v, const int32_t *block_table,
                                    int max_blocks, const int32_t *start_pos, int B, int n_new, int Hkv, int d, int P,
                                    int num_pages) {
    if (Hkv <= 0 || d != 128 || P <= 0 || B < 0 || n_new < 0) return ORACLE_EINVAL;
    uint8_t codes[64];
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < n_new; ++t) {
            long pos = (long)start_pos[b] + t;
            if (pos < 0 || pos / P >= max_blocks) return ORACLE_ERANGE;
            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
            int slot = (int)(pos % P);
            for (int h = 0; h < Hkv; ++h) {
                size_t src = (((size_t)b * (size_t)n_new + (size_t)t) * (size_t)Hkv + (size_t)h) * (size_t)d;
                uint8_t *blk = wht4_block(pool, Hkv, d, P, page, h);
                float sk, sv;
                kvq_oracle_wht4_quantize_row(k + src, d, codes, &sk);
                memcpy(blk + (size_t)slot * (size_t)(d / 2), codes, (size_t)d / 2);
                kvq_oracle_wht4_quantize_row(v + src, d, codes, &sv);
                memcpy(blk + ((size_t)P + (size_t)slot) * (size_t)(d / 2), codes, (size_t)d / 2);
                put_f32(blk + (size_t)P * (size_t)d + (size_t)4 * (size_t)slot, sk);
                put_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot), sv);
            }
        }
    }
    return ORACLE_OK;
}

/* Dequantize positions [start, start+n) of sequence b (fp64 rounded to fp32). */
int kvq_oracle_wht4_dequantize(const uint8_t *pool, const int32_t *block_table, int max_blocks, int b, int start,
                               int n, float *out_k, float *out_v, int Hkv, int d, int P, int num_pages) {
    if (Hkv <= 0 || d != 128 || P <= 0 || start < 0 || n < 0) return ORACLE_EINVAL;
    double r[128];
    for (int t = 0; t < n; ++t) {
        long pos = (long)start + t;
        if (pos / P >= max_blocks) return ORACLE_ERANGE;
        int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];
        if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
        int slot = (int)(pos % P);
        for (int h = 0; h < Hkv; ++h) {
            const uint8_t *blk = wht4_block((uint8_t *)pool, Hkv, d, P, page, h);
            size_t off = ((size_t)t * (size_t)Hkv + (size_t)h) * (size_t)d;
            wht4_dequant_row_f64(blk + (size_t)slot * (size_t)(d / 2), get_f32(blk + (size_t)P * (size_t)d + (size_t)4 * (size_t)slot), d, r);
            for (int i = 0; i < d; ++i) out_k[off + i] = (float)r[i];
            wht4_dequant_row_f64(blk + ((size_t)P + (size_t)slot) * (size_t)(d / 2),
                                 get_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot)), d, r);
            for (int i = 0; i < d; ++i) out_v[off + i] = (float)r[i];
        }
    }
    return ORACLE_OK;
}

/* Decode attention over the rotated 4-bit cache, in fp64 ([M] section 3.2) over the
 * dequantized rows x^ = H (sigma * c) / d. */
int kvq_oracle_wht4_decode_attention(const uint8_t *pool, const uint16_t *q, const int32_t *block_table,
                                     int max_blocks, const int32_t *seq_lens, int B, int Hq, double softmax_scale,
                                     double *out, int Hkv, int d, int P, int num_pages) {
    if (Hkv <= 0 || d != 128 || P <= 0 || Hq <= 0 || Hq % Hkv) return ORACLE_EINVAL;
    int grp = Hq / Hkv;
    double rk[128], rv[128];
    for (int b = 0; b < B; ++b) {
        int len = seq_lens[b];
        if (len < 0 || (len + P - 1) / P > max_blocks) return ORACLE_ERANGE;
        for (int hq = 0; hq < Hq; ++hq) {
            int kvh = hq / grp;
            const uint16_t *qrow = q + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            double *o = out + ((size_t)b * (size_t)Hq + (size_t)hq) * (size_t)d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (len == 0) continue;
            double top = -INFINITY, den = 0.0;
            for (int pass = 0; pass < 2; ++pass) {
                for (int t = 0; t < len; ++t) {
                    int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];
                    if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
                    const uint8_t *blk = wht4_block((uint8_t *)pool, Hkv, d, P, page, kvh);
                    int slot = t % P;
                    wht4_dequant_row_f64(blk + (size_t)slot * (size_t)(d / 2),
                                         get_f32(blk + (size_t)P * (size_t)d + (size_t)4 * (size_t)slot), d, rk);
                    double z = 0.0;
                    for (int i = 0; i < d; ++i) z += kvq_oracle_f16_to_f64(qrow[i]) * rk[i];
                    z *= softmax_scale;
                    if (pass == 0) {
                        if (z > top) top = z;
                        continue;
                    }
                    wht4_dequant_row_f64(blk + ((size_t)P + (size_t)slot) * (size_t)(d / 2),
                                         get_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot)), d, rv);
                    double e = exp(z - top);
                    den += e;
                    for (int i = 0; i < d; ++i) o[i] += e * rv[i];
                }
            }
            for (int i = 0; i < d; ++i) o[i] /= den;
        }
    }
    return ORACLE_OK;
}
