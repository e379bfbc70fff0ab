/*
 * CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library. It shares no code, header or constant with the CUDA
 * library; it reads host copies of the caches that tests fill through their
 * own scatter (orc_append*) and computes everything the slow, plain way.
 *
 * Citations name the page and the section it falls in:
 *   [p1] "大模型推理优化全攻略" (zhengtianqi.github.io) §2.1-2.3
 *   [p3] "KV Cache ... PagedAttention" (devpress.csdn.net) §二 formula, §七 block table
 *   [p4] "cs336 lecture 10" notes: KV Cache workflow, GQA/MQA, Quantization
 *
 * Cache layout (this project's reading; the pages fix none): per K and per V,
 * cache[num_blocks][num_kv_heads][block_size][head_dim], and for INT8 a
 * per-(token, kv_head) fp32 scale and int8 zero point, [num_blocks][num_kv_heads][block_size];
 * for FP8 (E4M3) one fp32 scale per kv head, [num_kv_heads] (p2 "ybb.press" §5.2:
 * per-head scaling factors for an FP8 KV cache).
 * A slot is phys_block * block_size + offset; a negative slot is skipped.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math: the
 * quantiser depends on IEEE fp32 division and round-half-to-even).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORC_F16 0
#define ORC_BF16 1
#define ORC_F32 2
#define ORC_INT8 3
#define ORC_FP8 4

/* ---- element decoding from the IEEE 754 definitions ---------------------- */

/* binary16: sign, 5-bit exponent (bias 15), 10-bit fraction */
static double f16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                  /* subnormal: m * 2^-24 */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);             /* (1 + m/2^10) * 2^(e-15) */
    return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float src_to_f32(const uint16_t* p, int dtype) {
    /* a binary16 value is exactly representable in binary32 */
    return dtype == ORC_BF16 ? bf16_to_f32(*p) : (float)f16_to_f64(*p);
}

double orc_f16_to_f64(uint16_t h) { return f16_to_f64(h); }

/* ---- INT8 quantiser ([p4] Quantization: x_q = round(x/scale) + zero_point) --
 * Readings: one (scale, zero_point) per (token, kv_head) row; the range is
 * widened to include 0; scale = (max - min)/255 in fp32 (1 if that is 0);
 * zero_point = clamp(-128 - round(min/scale)); round = half-to-even (rintf) on
 * the correctly rounded fp32 quotient; codes clamped to [-128, 127].        */
void orc_quantize_row(const float* x, int d, int8_t* codes, float* scale_out,
                      int8_t* zp_out) {
    float mn = 0.0f, mx = 0.0f;
    for (int j = 0; j < d; ++j) {
        if (x[j] < mn) mn = x[j];
        if (x[j] > mx) mx = x[j];
    }
    float scale = (mx - mn) / 255.0f;
    if (scale == 0.0f) scale = 1.0f;
    float zf = -128.0f - rintf(mn / scale);
    int zp = (int)zf;
    if (zp < -128) zp = -128;
    if (zp > 127) zp = 127;
    for (int j = 0; j < d; ++j) {
        int c = (int)rintf(x[j] / scale) + zp;
        if (c < -128) c = -128;
        if (c > 127) c = 127;
        codes[j] = (int8_t)c;
    }
    *scale_out = scale;
    *zp_out = (int8_t)zp;
}

/* ---- FP8 E4M3 (the OCP 8-bit float "E4M3": 1 sign bit, 4 exponent bits with
 * bias 7, 3 fraction bits; no infinities; exponent 15 with fraction 7 is NaN,
 * so the largest finite value is 1.75 * 2^8 = 448; exponent 0 holds the
 * subnormals m * 2^-9). Decoded here from that definition.                   */
double orc_e4m3_to_f64(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);                /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Nearest E4M3 value, ties to even; magnitudes above 448 (including infinity)
 * saturate to 448; NaN gives 0x7F. The value is scaled by a power of two so
 * that rint() (round half to even) picks the fraction exactly.              */
uint8_t orc_e4m3_encode(float xf) {
    double x = (double)xf;
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    uint8_t code;
    if (a >= 448.0) {
        code = 0x7e;
    } else if (a < ldexp(1.0, -6)) {                        /* subnormal range */
        code = (uint8_t)rint(ldexp(a, 9));                  /* 0..8; 8 is the smallest normal */
    } else {
        int k;
        frexp(a, &k);                                       /* a = f * 2^k, f in [0.5, 1) */
        int e = k - 1;                                      /* 2^e <= a < 2^(e+1) */
        double n = rint(ldexp(a, 3 - e));                   /* 8..16 */
        if (n == 16.0) {
            n = 8.0;
            e += 1;
        }
        int c = ((e + 7) << 3) | ((int)n - 8);
        code = (uint8_t)(c > 0x7e ? 0x7e : c);
    }
    return sign | code;
}

/* FP8 quantiser: code = E4M3(x / scale), the quotient the correctly rounded
 * fp32 division; dequantised value = E4M3 value * scale in fp32.             */
void orc_append_fp8(uint8_t* codes, const float* head_scale, const uint16_t* src,
                    int src_dtype, const int64_t* slots, int64_t num_tokens,
                    int num_kv_heads, int head_dim, int block_size) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int g = 0; g < num_kv_heads; ++g) {
            const uint16_t* s = src + (t * num_kv_heads + g) * head_dim;
            uint8_t* dst = codes + ((blk * num_kv_heads + g) * block_size + off) * head_dim;
            for (int j = 0; j < head_dim; ++j) {
                float y = src_to_f32(s + j, src_dtype) / head_scale[g];
                dst[j] = orc_e4m3_encode(y);
            }
        }
    }
}

static double dequant_fp8(uint8_t c, float scale) {
    float x = (float)orc_e4m3_to_f64(c) * scale;            /* E4M3 values are exact in fp32 */
    return (double)x;
}

/* [p4] Quantization: x = (x_q - zero_point) * scale, one fp32 rounding */
static double dequant(int8_t c, int8_t zp, float scale) {
    float x = (float)((int)c - (int)zp) * scale;
    return (double)x;
}

/* ---- append: write new K/V rows through the slot mapping ([p4] workflow step
 * "append the new K, V to the cache"; [p3] §七 logical->physical blocks) ---- */
void orc_append(uint16_t* cache, const uint16_t* src, const int64_t* slots,
                int64_t num_tokens, int num_kv_heads, int head_dim,
                int block_size) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int g = 0; g < num_kv_heads; ++g) {
            uint16_t* dst = cache + ((blk * num_kv_heads + g) * block_size + off) * head_dim;
            const uint16_t* s = src + (t * num_kv_heads + g) * head_dim;
            memcpy(dst, s, (size_t)head_dim * sizeof(uint16_t));
        }
    }
}

void orc_append_int8(int8_t* codes, float* scales, int8_t* zps,
                     const uint16_t* src, int src_dtype, const int64_t* slots,
                     int64_t num_tokens, int num_kv_heads, int head_dim,
                     int block_size) {
    float* row = (float*)malloc((size_t)head_dim * sizeof(float));
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int g = 0; g < num_kv_heads; ++g) {
            const uint16_t* s = src + (t * num_kv_heads + g) * head_dim;
            for (int j = 0; j < head_dim; ++j) row[j] = src_to_f32(s + j, src_dtype);
            int64_t r = (blk * num_kv_heads + g) * block_size + off;
            orc_quantize_row(row, head_dim, codes + r * head_dim, scales + r, zps + r);
        }
    }
    free(row);
}

/* ---- copy-on-write: copy whole physical blocks (p2 "ybb.press" §2.1) ---- */
void orc_copy_blocks(uint8_t* base, int64_t bytes_per_block,
                     const int32_t* pairs, int n_pairs) {
    for (int i = 0; i < n_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        memcpy(base + dst * bytes_per_block, base + src * bytes_per_block,
               (size_t)bytes_per_block);
    }
}

/* ---- attention -----------------------------------------------------------
 * [p3] §二: Attention(Q,K,V) = softmax(Q K^T / sqrt(d)) V; [p4] decode step:
 * score the new token's q against every cached K, weight the cached V.
 * GQA ([p4] GQA/MQA): q head h reads kv head h / (H_q / H_kv).
 * A query run of r tokens (speculative verify) puts query i at absolute
 * position L - r + i; it sees keys 0 .. L - r + i (causal).
 *
 * This routine covers the keys t in [t_begin, t_end) that the query sees and
 * returns, per (query token, q head): m = max logit (-inf if no key), l = sum
 * of exp(logit - m), and o = sum exp(logit - m) V / l (0 if no key). With the
 * full range it is plain softmax attention; a sub-range gives a split-KV
 * partition's partial result.                                             */
typedef struct {
    const void* k_cache;
    const void* v_cache;
    int kv_dtype;
    const float* k_scale;
    const float* v_scale;
    const int8_t* k_zp;
    const int8_t* v_zp;
    const int32_t* block_tables;
    int max_blocks;
    int num_kv_heads;
    int head_dim;
    int block_size;
} orc_cache;

static double load_kv(const orc_cache* c, int is_v, int64_t blk, int g, int off, int j) {
    int64_t r = (blk * c->num_kv_heads + g) * c->block_size + off;
    int64_t e = r * c->head_dim + j;
    const void* base = is_v ? c->v_cache : c->k_cache;
    switch (c->kv_dtype) {
        case ORC_F16: return f16_to_f64(((const uint16_t*)base)[e]);
        case ORC_BF16: return (double)bf16_to_f32(((const uint16_t*)base)[e]);
        case ORC_F32: return (double)((const float*)base)[e];
        case ORC_FP8:
            return dequant_fp8(((const uint8_t*)base)[e], (is_v ? c->v_scale : c->k_scale)[g]);
        default:
            return dequant(((const int8_t*)base)[e],
                           (is_v ? c->v_zp : c->k_zp)[r],
                           (is_v ? c->v_scale : c->k_scale)[r]);
    }
}

int orc_attend_range(double* out_o, double* out_m, double* out_l,
                     const double* q, const orc_cache* c,
                     const int32_t* context_lens, const int32_t* query_start_loc,
                     int num_seqs, int num_heads, double scale,
                     int64_t t_begin, int64_t t_end, int threads) {
    const int H_kv = c->num_kv_heads, d = c->head_dim, bs = c->block_size;
    if (num_heads % H_kv != 0) return 1;
    const int G = num_heads / H_kv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic) num_threads(threads) reduction(|:bad)
    for (int64_t task = 0; task < (int64_t)num_seqs * H_kv; ++task) {
        int s = (int)(task / H_kv), g = (int)(task % H_kv);
        int64_t L = context_lens[s];
        int64_t q0 = query_start_loc ? query_start_loc[s] : s;
        int64_t r = query_start_loc ? query_start_loc[s + 1] - q0 : 1;
        if (L < 1 || r < 1 || r > L) { bad = 1; continue; }
        /* gather this sequence's keys and values for kv head g, contiguous, fp64 */
        double* K = (double*)malloc((size_t)(L * d) * sizeof(double));
        double* V = (double*)malloc((size_t)(L * d) * sizeof(double));
        double* z = (double*)malloc((size_t)L * sizeof(double));
        for (int64_t t = 0; t < L; ++t) {
            int64_t blk = c->block_tables[(int64_t)s * c->max_blocks + t / bs];
            int off = (int)(t % bs);
            for (int j = 0; j < d; ++j) {
                K[t * d + j] = load_kv(c, 0, blk, g, off, j);
                V[t * d + j] = load_kv(c, 1, blk, g, off, j);
            }
        }
        for (int64_t i = 0; i < r; ++i) {
            int64_t last = L - r + i;                     /* causal: keys 0..last */
            int64_t lo = t_begin, hi = t_end < last + 1 ? t_end : last + 1;
            if (lo < 0) lo = 0;
            for (int hh = 0; hh < G; ++hh) {
                int h = g * G + hh;
                int64_t row = (q0 + i) * num_heads + h;
                const double* qv = q + row * d;
                double m = -INFINITY;
                for (int64_t t = lo; t < hi; ++t) {
                    double acc = 0.0;
                    for (int j = 0; j < d; ++j) acc += qv[j] * K[t * d + j];
                    z[t] = scale * acc;
                    if (z[t] > m) m = z[t];
                }
                double l = 0.0;
                double* o = out_o + row * d;
                for (int j = 0; j < d; ++j) o[j] = 0.0;
                for (int64_t t = lo; t < hi; ++t) {
                    double w = exp(z[t] - m);
                    l += w;
                    for (int j = 0; j < d; ++j) o[j] += w * V[t * d + j];
                }
                if (l > 0.0)
                    for (int j = 0; j < d; ++j) o[j] /= l;
                if (out_m) out_m[row] = m;
                if (out_l) out_l[row] = l;
            }
        }
        free(K);
        free(V);
        free(z);
    }
    return bad ? 2 : 0;
}

/* caller-friendly wrapper with the cache description spelled out */
int orc_attend(double* out_o, double* out_m, double* out_l, const double* q,
               const void* k_cache, const void* v_cache, int kv_dtype,
               const float* k_scale, const float* v_scale, const int8_t* k_zp,
               const int8_t* v_zp, const int32_t* block_tables, int max_blocks,
               const int32_t* context_lens, const int32_t* query_start_loc,
               int num_seqs, int num_heads, int num_kv_heads, int head_dim,
               int block_size, double scale, int64_t t_begin, int64_t t_end,
               int threads) {
    orc_cache c = {k_cache, v_cache, kv_dtype, k_scale, v_scale, k_zp, v_zp,
                   block_tables, max_blocks, num_kv_heads, head_dim, block_size};
    return orc_attend_range(out_o, out_m, out_l, q, &c, context_lens,
                            query_start_loc, num_seqs, num_heads, scale,
                            t_begin, t_end, threads);
}
