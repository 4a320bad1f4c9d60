/*
 * pkv_oracle.c -- plain, slow, FP64 CPU oracle for the paged-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg are the only code allowed to load
 * this library.  The CUDA library never calls it; the two share no source,
 * header, table, constant or helper.  Every function below is a direct
 * restatement of a definition, written for a reader to check by eye, with no
 * blocking, fusion or reordering.
 *
 * Sources (web pages describing the engine this path belongs to):
 *  [S3] "从零用 C++ 和 CUDA 实现 Llama 3.2 1B 推理引擎:6 小时视频与 85 页手写笔记"
 *       (summary of the samir-vllm README), section "目前已完成的功能"
 *       (features done so far): a shared BF16 KV page pool with per-sequence,
 *       per-layer block tables; each physical page holds K and V of 16 tokens;
 *       decode appends one token at its absolute RoPE position; paged decode
 *       attention streams a sequence's cached pages with an FP32 online
 *       softmax and never gathers a contiguous prefix or stores the scores.
 *  [S2] "从零构建大模型推理引擎：KV缓存、算子融合与量化优化实战", section 3.2
 *       (efficient attention): scores = q K^T, divided by sqrt(head_dim),
 *       softmax with the maximum subtracted, then the weighted sum of V;
 *       section 2.1: the contiguous [batch, heads, seq, head_dim] cache;
 *       section 4.1: rotary position embedding injects absolute position.
 *  [S1] "使用 Tiny-vLLM 從零開始構建高性能 LLM 推理引擎", section "Bfloat16 的選擇":
 *       BF16 keeps the FP32 exponent (8 bits) and 7 fraction bits.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - in-page layout [K|V][kv_head][slot][dim], pages contiguous in one slab;
 *  - RoPE pairs dimension i with i + head_dim/2 ("rotate half"), frequency
 *    theta^(-2i/head_dim); no Llama-3 frequency rescaling;
 *  - query head h reads KV head h / (Hq / Hkv);
 *  - a sequence of length L holds tokens 0..L-1; the decode token sits at
 *    position L-1 and attends to itself.
 *
 * Built with -ffp-contract=off so that no multiply-add is fused and the same
 * source gives the same bits on x86-64 and AArch64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_PAGE (-2)
#define ORACLE_NO_MEMORY (-3)

/* ------------------------------------------------------------------------ */
/* BF16 <-> FP64 [S1]: a BF16 value is the upper 16 bits of an IEEE binary32. */

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round an FP64 value to the nearest BF16, ties to even, in ONE rounding
 * (no intermediate FP32).  Method: find the power-of-two quantum q of the
 * BF16 grid around |x| (8 significant bits; below 2^-126 the grid is the
 * fixed subnormal spacing 2^-133), scale by 1/q (exact), round to an integer
 * with rint() in the default round-to-nearest-even mode, and scale back. */
uint16_t oracle_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e with m in [0.5, 1) */
    int exponent = e - 1;        /* a in [2^exponent, 2^(exponent+1)) */
    if (exponent < -126)
        exponent = -126;         /* subnormal BF16 numbers share this spacing */
    double quantum = ldexp(1.0, exponent - 7);
    double n = rint(a / quantum);
    double r = n * quantum;
    /* largest finite BF16 is (2 - 2^-7) * 2^127 */
    if (r > ldexp(255.0, 120))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)r;          /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (bits >> 16));
}

/* ------------------------------------------------------------------------ */
/* Rotary position embedding [S2 4.1, S3 RoPE item].
 * Pair i (0 <= i < head_dim/2) is the plane (x[i], x[i + head_dim/2]); at
 * absolute position pos it is turned by the angle pos * theta^(-2i/head_dim):
 *   y[i]          = x[i] cos(a) - x[i+half] sin(a)
 *   y[i+half]     = x[i+half] cos(a) + x[i] sin(a)                         */

double oracle_rope_inv_freq(double theta, int head_dim, int i)
{
    return pow(theta, -2.0 * (double)i / (double)head_dim);
}

void oracle_rope_rotate(const double *x, int head_dim, long long pos, double theta, double *y)
{
    int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        double angle = (double)pos * oracle_rope_inv_freq(theta, head_dim, i);
        double c = cos(angle);
        double s = sin(angle);
        double x1 = x[i];
        double x2 = x[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
}

/* ------------------------------------------------------------------------ */
/* The page pool [S3 page-pool item].  One slab of num_pages pages; a page is
 * [2 (K then V)][num_kv_heads][page_size slots][head_dim] BF16 values.        */

typedef struct {
    int32_t num_pages;
    int32_t page_size;
    int32_t num_kv_heads;
    int32_t head_dim;
} oracle_pool_geom;

int64_t oracle_pool_index(const oracle_pool_geom *g, int page, int kv, int head, int slot, int dim)
{
    int64_t idx = page;
    idx = idx * 2 + kv;
    idx = idx * g->num_kv_heads + head;
    idx = idx * g->page_size + slot;
    idx = idx * g->head_dim + dim;
    return idx;
}

/* Logical token t of a sequence lives in logical page t / page_size, at slot
 * t % page_size; the block-table row maps the logical page to a physical one. */
static int token_page(const oracle_pool_geom *g, const int32_t *bt_row, int max_blocks, int t,
                      int *page, int *slot)
{
    int logical = t / g->page_size;
    if (t < 0 || logical >= max_blocks)
        return ORACLE_BAD_ARG;
    int p = bt_row[logical];
    if (p < 0 || p >= g->num_pages)
        return ORACLE_BAD_PAGE;
    *page = p;
    *slot = t % g->page_size;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Append [S3: "decode appends one new token at its absolute RoPE position"].
 * For each sequence b with position p = pos[b]:
 *   K slot  <- BF16(RoPE_p(k_new[b][g]))  for every KV head g,
 *   V slot  <- v_new[b][g]                (not rotated, bits copied),
 *   q[b][h] <- BF16(RoPE_p(q[b][h]))      in place, when q is given.
 * pool: uint16 BF16 bits, geometry g; bt: [B][max_blocks]; k_new, v_new:
 * [B][num_kv_heads][head_dim]; q: [B][num_q_heads][head_dim] or NULL.        */
int oracle_append(uint16_t *pool, const oracle_pool_geom *g, const int32_t *bt, int max_blocks,
                  const int32_t *pos, int B, const uint16_t *k_new, const uint16_t *v_new,
                  uint16_t *q, int num_q_heads, double theta)
{
    int D = g->head_dim;
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    double *y = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x || !y) {
        free(x);
        free(y);
        return ORACLE_NO_MEMORY;
    }
    int status = ORACLE_OK;
    for (int b = 0; b < B && status == ORACLE_OK; ++b) {
        int p = pos[b];
        int page, slot;
        status = token_page(g, bt + (size_t)b * max_blocks, max_blocks, p, &page, &slot);
        if (status != ORACLE_OK)
            break;
        for (int h = 0; h < g->num_kv_heads; ++h) {
            const uint16_t *k = k_new + ((size_t)b * g->num_kv_heads + h) * D;
            const uint16_t *v = v_new + ((size_t)b * g->num_kv_heads + h) * D;
            for (int d = 0; d < D; ++d)
                x[d] = oracle_bf16_to_double(k[d]);
            oracle_rope_rotate(x, D, p, theta, y);
            for (int d = 0; d < D; ++d) {
                pool[oracle_pool_index(g, page, 0, h, slot, d)] = oracle_bf16_from_double(y[d]);
                pool[oracle_pool_index(g, page, 1, h, slot, d)] = v[d];
            }
        }
        if (q) {
            for (int h = 0; h < num_q_heads; ++h) {
                uint16_t *qh = q + ((size_t)b * num_q_heads + h) * D;
                for (int d = 0; d < D; ++d)
                    x[d] = oracle_bf16_to_double(qh[d]);
                oracle_rope_rotate(x, D, p, theta, y);
                for (int d = 0; d < D; ++d)
                    qh[d] = oracle_bf16_from_double(y[d]);
            }
        }
    }
    free(x);
    free(y);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Paged decode attention for ONE (sequence, query head) [S3 paged-attention
 * item, S2 3.2].  Walks the block-table row token by token:
 *   s_t = scale * sum_d q[d] k_t[d]            t = 0 .. L-1
 *   m   = max_t s_t
 *   w_t = exp(s_t - m) / sum_u exp(s_u - m)
 *   out = sum_t w_t v_t
 * out: [head_dim] doubles.  weights: [L] doubles or NULL.                    */
int oracle_decode_one(const uint16_t *pool, const oracle_pool_geom *g, const int32_t *bt_row,
                      int max_blocks, int L, const uint16_t *q_row, int kv_head, double scale,
                      double *out, double *weights)
{
    int D = g->head_dim;
    if (L < 1 || L > max_blocks * g->page_size || kv_head < 0 || kv_head >= g->num_kv_heads)
        return ORACLE_BAD_ARG;
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        return ORACLE_NO_MEMORY;

    for (int t = 0; t < L; ++t) {
        int page, slot;
        int st = token_page(g, bt_row, max_blocks, t, &page, &slot);
        if (st != ORACLE_OK) {
            free(s);
            return st;
        }
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += oracle_bf16_to_double(q_row[d]) *
                   oracle_bf16_to_double(pool[oracle_pool_index(g, page, 0, kv_head, slot, d)]);
        s[t] = scale * dot;
    }

    double m = s[0];
    for (int t = 1; t < L; ++t)
        if (s[t] > m)
            m = s[t];
    double z = 0.0;
    for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - m);
        z += s[t];
    }
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    for (int t = 0; t < L; ++t) {
        int page = 0, slot = 0;
        (void)token_page(g, bt_row, max_blocks, t, &page, &slot);
        double w = s[t] / z;
        if (weights)
            weights[t] = w;
        for (int d = 0; d < D; ++d)
            out[d] += w * oracle_bf16_to_double(pool[oracle_pool_index(g, page, 1, kv_head, slot, d)]);
    }
    free(s);
    return ORACLE_OK;
}

/* The whole batch: every sequence b, every query head h (KV head h/group).
 * q: [B][num_q_heads][head_dim] BF16; out_bf16: same shape, each value
 * rounded once from FP64; out_f64 (optional): the unrounded FP64 result.     */
int oracle_decode(const uint16_t *pool, const oracle_pool_geom *g, const int32_t *bt, int max_blocks,
                  const int32_t *seq_lens, int B, const uint16_t *q, int num_q_heads, double scale,
                  uint16_t *out_bf16, double *out_f64)
{
    int D = g->head_dim;
    if (num_q_heads < g->num_kv_heads || num_q_heads % g->num_kv_heads != 0)
        return ORACLE_BAD_ARG;
    int group = num_q_heads / g->num_kv_heads;
    double *o = (double *)malloc(sizeof(double) * (size_t)D);
    if (!o)
        return ORACLE_NO_MEMORY;
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < num_q_heads; ++h) {
            size_t row = (size_t)b * num_q_heads + h;
            int st = oracle_decode_one(pool, g, bt + (size_t)b * max_blocks, max_blocks, seq_lens[b],
                                       q + row * D, h / group, scale, o, NULL);
            if (st != ORACLE_OK) {
                free(o);
                return st;
            }
            for (int d = 0; d < D; ++d) {
                if (out_bf16)
                    out_bf16[row * D + d] = oracle_bf16_from_double(o[d]);
                if (out_f64)
                    out_f64[row * D + d] = o[d];
            }
        }
    }
    free(o);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Brute-force attention over a CONTIGUOUS cache [S2 2.1]: K, V are
 * [B][Hkv][S][D] doubles, sequence b uses rows 0 .. seq_lens[b]-1.  Same
 * definition as above, a second, independent walk used to cross-check the
 * paged one.  q: [B][Hq][D] doubles; out: [B][Hq][D] doubles.               */
int oracle_decode_contiguous(const double *K, const double *V, int S, const int32_t *seq_lens, int B,
                             const double *q, int Hq, int Hkv, int D, double scale, double *out)
{
    if (Hq % Hkv != 0)
        return ORACLE_BAD_ARG;
    double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    if (!s)
        return ORACLE_NO_MEMORY;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > S) {
            free(s);
            return ORACLE_BAD_ARG;
        }
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / (Hq / Hkv);
            const double *qh = q + ((size_t)b * Hq + h) * D;
            const double *Kh = K + ((size_t)b * Hkv + kvh) * (size_t)S * D;
            const double *Vh = V + ((size_t)b * Hkv + kvh) * (size_t)S * D;
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += qh[d] * Kh[(size_t)t * D + d];
                s[t] = scale * dot;
                if (s[t] > m)
                    m = s[t];
            }
            double z = 0.0;
            for (int t = 0; t < L; ++t) {
                s[t] = exp(s[t] - m);
                z += s[t];
            }
            double *oh = out + ((size_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int t = 0; t < L; ++t)
                    acc += s[t] * Vh[(size_t)t * D + d];
                oh[d] = acc / z;
            }
        }
    }
    free(s);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* FP8 KV pages ("从零构建大模型推理引擎" section 5.1: store the KV cache in low
 * precision and dequantize before attention).  The page gives no scheme; the
 * reading taken here:
 *  - element format FP8 E4M3 without infinities (largest finite 448), round to
 *    nearest even, saturating at +-448;
 *  - one FP32 scale per (token, KV head) row of 64 values: scale = amax / 448
 *    (FP32 division; 1 for an all-zero row), code = E4M3(x / scale) with x / scale
 *    an FP32 division; the row's input is the BF16 value the BF16 path would store;
 *  - page = kv_heads units, one per KV head, each the K codes [page_size][head_dim]
 *    (1 byte each, row-major), the V codes (same bytes, stored token-pair
 *    interleaved, below), then the scales [2 (K,V)][page_size] FP32:
 *    8 x (2048 + 128) = 17408 bytes for 8 x 16 x 64;
 *  - V codes: slots 2p and 2p+1 share a 2 x head_dim byte line; in it, dims
 *    8c .. 8c+7 of both slots form 16-byte chunk c (byte 2 (dim % 8) + slot % 2),
 *    stored at chunk position c XOR (2p mod head_dim/8) (head_dim/8 a power of two).
 *    Where each byte goes is storage only: every value is the same code.            */

uint8_t oracle_e4m3_from_double(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);  /* saturate to the largest finite value */
    if (a < ldexp(1.0, -6)) {           /* subnormal spacing 2^-9; 8 quanta = 2^-6 (code 8) */
        double n = rint(a / ldexp(1.0, -9));
        return (uint8_t)(sign | (uint8_t)n);
    }
    int e;
    (void)frexp(a, &e);
    int exponent = e - 1;               /* a in [2^exponent, 2^(exponent+1)), exponent >= -6 */
    double n = rint(a / ldexp(1.0, exponent - 3));  /* 8 .. 16 */
    if (n >= 16.0) {
        n = 8.0;
        exponent += 1;
    }
    if (exponent > 8 || (exponent == 8 && n > 14.0))
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | ((exponent + 7) << 3) | ((int)n - 8));
}

double oracle_e4m3_to_double(uint8_t c)
{
    double s = (c & 0x80) ? -1.0 : 1.0;
    int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        return s * ldexp((double)m, -9);
    return s * ldexp((double)(8 + m), e - 10);
}

/* Quantize n BF16 values (FP32 arithmetic, as defined above). */
void oracle_quantize_row_fp8(const uint16_t *row, int n, uint8_t *codes, float *scale_out)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf((float)oracle_bf16_to_double(row[i]));
        if (a > amax)
            amax = a;
    }
    float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < n; ++i) {
        float v = (float)oracle_bf16_to_double(row[i]) / scale;
        codes[i] = oracle_e4m3_from_double((double)v);
    }
    *scale_out = scale;
}

int64_t oracle_fp8_page_bytes(const oracle_pool_geom *g)
{
    return (int64_t)2 * g->num_kv_heads * g->page_size * (g->head_dim + 4);
}

/* bytes of one KV head's unit inside an FP8 page */
static int64_t fp8_unit_bytes(const oracle_pool_geom *g)
{
    return (int64_t)2 * g->page_size * (g->head_dim + 4);
}

/* byte offset of a code / of a row's scale inside the FP8 pool */
int64_t oracle_fp8_code_offset(const oracle_pool_geom *g, int page, int kv, int head, int slot, int dim)
{
    int64_t unit = (int64_t)page * oracle_fp8_page_bytes(g) + head * fp8_unit_bytes(g);
    if (kv == 0)
        return unit + (int64_t)slot * g->head_dim + dim;
    int pair = slot / 2, chunks = g->head_dim / 8;
    int chunk = (dim / 8) ^ ((2 * pair) % chunks);
    return unit + (int64_t)g->page_size * g->head_dim + (int64_t)pair * 2 * g->head_dim + chunk * 16 +
           2 * (dim % 8) + slot % 2;
}

int64_t oracle_fp8_scale_offset(const oracle_pool_geom *g, int page, int kv, int head, int slot)
{
    int64_t row = (int64_t)kv * g->page_size + slot;
    return (int64_t)page * oracle_fp8_page_bytes(g) + head * fp8_unit_bytes(g) +
           (int64_t)2 * g->page_size * g->head_dim + row * 4;
}

static void fp8_store_row(uint8_t *pool, const oracle_pool_geom *g, int page, int kv, int head, int slot,
                          const uint16_t *row)
{
    uint8_t codes[1024];
    float scale;
    oracle_quantize_row_fp8(row, g->head_dim, codes, &scale);
    for (int d = 0; d < g->head_dim; ++d)
        pool[oracle_fp8_code_offset(g, page, kv, head, slot, d)] = codes[d];
    memcpy(pool + oracle_fp8_scale_offset(g, page, kv, head, slot), &scale, sizeof scale);
}

/* As oracle_append, storing each appended K (rotated, BF16) and V row quantized. */
int oracle_append_fp8(uint8_t *pool, const oracle_pool_geom *g, const int32_t *bt, int max_blocks,
                      const int32_t *pos, int B, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                      int num_q_heads, double theta)
{
    int D = g->head_dim;
    if (D > 1024)
        return ORACLE_BAD_ARG;
    double x[1024], y[1024];
    uint16_t rot[1024];
    for (int b = 0; b < B; ++b) {
        int p = pos[b], page, slot;
        int st = token_page(g, bt + (size_t)b * max_blocks, max_blocks, p, &page, &slot);
        if (st != ORACLE_OK)
            return st;
        for (int h = 0; h < g->num_kv_heads; ++h) {
            const uint16_t *k = k_new + ((size_t)b * g->num_kv_heads + h) * D;
            for (int d = 0; d < D; ++d)
                x[d] = oracle_bf16_to_double(k[d]);
            oracle_rope_rotate(x, D, p, theta, y);
            for (int d = 0; d < D; ++d)
                rot[d] = oracle_bf16_from_double(y[d]);
            fp8_store_row(pool, g, page, 0, h, slot, rot);
            fp8_store_row(pool, g, page, 1, h, slot, v_new + ((size_t)b * g->num_kv_heads + h) * D);
        }
        if (q) {
            for (int h = 0; h < num_q_heads; ++h) {
                uint16_t *qh = q + ((size_t)b * num_q_heads + h) * D;
                for (int d = 0; d < D; ++d)
                    x[d] = oracle_bf16_to_double(qh[d]);
                oracle_rope_rotate(x, D, p, theta, y);
                for (int d = 0; d < D; ++d)
                    qh[d] = oracle_bf16_from_double(y[d]);
            }
        }
    }
    return ORACLE_OK;
}

static double fp8_value(const uint8_t *pool, const oracle_pool_geom *g, int page, int kv, int head, int slot, int d)
{
    float scale;
    memcpy(&scale, pool + oracle_fp8_scale_offset(g, page, kv, head, slot), sizeof scale);
    return oracle_e4m3_to_double(pool[oracle_fp8_code_offset(g, page, kv, head, slot, d)]) * (double)scale;
}

/* Paged decode attention over FP8 pages: the same definition as oracle_decode_one,
 * each K and V element dequantized as code * row scale (exact in FP64). */
int oracle_decode_one_fp8(const uint8_t *pool, const oracle_pool_geom *g, const int32_t *bt_row, int max_blocks,
                          int L, const uint16_t *q_row, int kv_head, double scale, double *out, double *weights)
{
    int D = g->head_dim;
    if (L < 1 || L > max_blocks * g->page_size || kv_head < 0 || kv_head >= g->num_kv_heads)
        return ORACLE_BAD_ARG;
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        return ORACLE_NO_MEMORY;
    for (int t = 0; t < L; ++t) {
        int page, slot;
        int st = token_page(g, bt_row, max_blocks, t, &page, &slot);
        if (st != ORACLE_OK) {
            free(s);
            return st;
        }
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += oracle_bf16_to_double(q_row[d]) * fp8_value(pool, g, page, 0, kv_head, slot, d);
        s[t] = scale * dot;
    }
    double m = s[0];
    for (int t = 1; t < L; ++t)
        if (s[t] > m)
            m = s[t];
    double z = 0.0;
    for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - m);
        z += s[t];
    }
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    for (int t = 0; t < L; ++t) {
        int page = 0, slot = 0;
        (void)token_page(g, bt_row, max_blocks, t, &page, &slot);
        double w = s[t] / z;
        if (weights)
            weights[t] = w;
        for (int d = 0; d < D; ++d)
            out[d] += w * fp8_value(pool, g, page, 1, kv_head, slot, d);
    }
    free(s);
    return ORACLE_OK;
}

int oracle_decode_fp8(const uint8_t *pool, const oracle_pool_geom *g, const int32_t *bt, int max_blocks,
                      const int32_t *seq_lens, int B, const uint16_t *q, int num_q_heads, double scale,
                      uint16_t *out_bf16, double *out_f64)
{
    int D = g->head_dim;
    if (num_q_heads < g->num_kv_heads || num_q_heads % g->num_kv_heads != 0)
        return ORACLE_BAD_ARG;
    int group = num_q_heads / g->num_kv_heads;
    double *o = (double *)malloc(sizeof(double) * (size_t)D);
    if (!o)
        return ORACLE_NO_MEMORY;
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < num_q_heads; ++h) {
            size_t row = (size_t)b * num_q_heads + h;
            int st = oracle_decode_one_fp8(pool, g, bt + (size_t)b * max_blocks, max_blocks, seq_lens[b],
                                           q + row * D, h / group, scale, o, NULL);
            if (st != ORACLE_OK) {
                free(o);
                return st;
            }
            for (int d = 0; d < D; ++d) {
                if (out_bf16)
                    out_bf16[row * D + d] = oracle_bf16_from_double(o[d]);
                if (out_f64)
                    out_f64[row * D + d] = o[d];
            }
        }
    }
    free(o);
    return ORACLE_OK;
}
