/*
 * oracle.c -- plain, slow, fp64 CPU oracle for one paged-KV attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header or table with the CUDA library and must never be used as a
 * fallback for it.
 *
 * What it follows, all from the page "TensorRT-LLM框架解析与高性能推理优化实践":
 *   - §4.2 "KV缓存管理细节": K/V live in fixed-size pages of a shared pool;
 *     a sequence's pages are listed in its block table.
 *   - §6.2 "Paged Attention优化": attention for one head walks the
 *     sequence's block table, dot-products q with each key and accumulates a
 *     weighted sum of values; several sequences may point at the same prefix
 *     pages (the section's list of optimisations).
 *   - §6.1 "Flash Attention实现": softmax kept with a running max and sum;
 *     the oracle uses the plain two-pass max-subtracted softmax, which the
 *     running form equals.
 *   - §7.2 "KV Cache量化": quantised KV is dequantised inside the attention
 *     kernel (its third item): value = e4m3(code) * scale, with one scale
 *     per tensor or, as its first item has it, one per attention (kv) head.
 *   - §5.3 "分块上下文处理": a long prompt is processed in chunks; token i of
 *     a chunk of C tokens appended to a sequence of final length L sits at
 *     position L - C + i and attends to keys 0 .. L - C + i.
 * The E4M3 format is written from the OCP 8-bit floating point
 * specification (OFP8, E4M3: bias 7, no infinities, NaN = S.1111.111,
 * largest finite 448), not from any library.
 *
 * Pool layout: pool[num_blocks][num_kv_heads][block_size][head_dim], bf16
 * bits (uint16) or E4M3 codes (uint8).  q and new K/V are bf16 bits.
 * GQA: q head a reads kv head a / (Hq / Hkv).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { PKVO_BF16 = 0, PKVO_FP8_E4M3 = 1 };

/* ---- element formats --------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32. */
double pkvo_bf16_value(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP E4M3: s eeee mmm.  e = 0: subnormal m * 2^-9;  e = 15, m = 7: NaN;
 * otherwise (1 + m/8) * 2^(e-7). */
double pkvo_e4m3_value(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round to nearest, ties to even, saturating to the largest finite value
 * (+-448).  Written as the definition: among the finite non-negative codes
 * 0x00..0x7E, whose values increase with the code, pick the one nearest to
 * |x|; at an exact midpoint pick the code with an even last bit.  NaN input
 * gives 0x7F. */
uint8_t pkvo_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    int c;
    if (isnan(x))
        return 0x7F;
    if (a >= 448.0)
        return sign | 0x7E;
    c = 0;
    while (c < 0x7E && pkvo_e4m3_value((uint8_t)(c + 1)) <= a)
        c++;
    if (pkvo_e4m3_value((uint8_t)c) != a) {
        double lo = pkvo_e4m3_value((uint8_t)c);
        double hi = pkvo_e4m3_value((uint8_t)(c + 1));
        double mid = 0.5 * (lo + hi);           /* exact in binary64 */
        if (a > mid || (a == mid && (c & 1)))
            c = c + 1;
    }
    return sign | (uint8_t)c;
}

/* Quantise one bf16 value with a per-tensor scale: the quotient is taken in
 * binary32 (the precision the kernel decides the code in), then encoded. */
uint8_t pkvo_quantize_bf16(uint16_t bits, float scale)
{
    float x = (float)pkvo_bf16_value(bits);
    float y = x / scale;
    return pkvo_e4m3_encode(y);
}

/* Array forms, for exhaustive tests. */
void pkvo_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = pkvo_e4m3_encode(x[i]);
}

void pkvo_e4m3_value_array(const uint8_t *code, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = pkvo_e4m3_value(code[i]);
}

static double kv_value(const void *pool, int kv_dtype, int64_t idx, float scale)
{
    if (kv_dtype == PKVO_BF16)
        return pkvo_bf16_value(((const uint16_t *)pool)[idx]);
    return pkvo_e4m3_value(((const uint8_t *)pool)[idx]) * (double)scale;
}

/* ---- kv_append --------------------------------------------------------- */

/* Store token t's K and V rows (all kv heads) at slot_mapping[t]:
 * page = slot / P, offset = slot % P.  Negative slots are skipped.  Returns
 * the number of tokens whose slot lies beyond the pool (also skipped).
 * FP8: kv head h is quantised with k_scales[h] / v_scales[h] when those
 * arrays are given, else with k_scale / v_scale. */
int pkvo_kv_append(const uint16_t *k_new, const uint16_t *v_new,
                   const int64_t *slot_mapping, int T, int Hkv, int P, int D,
                   int64_t num_blocks, int kv_dtype, float k_scale, float v_scale,
                   const float *k_scales, const float *v_scales,
                   void *k_pool, void *v_pool)
{
    int bad = 0;
    for (int t = 0; t < T; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * (int64_t)P) {
            bad++;
            continue;
        }
        int64_t page = slot / P, off = slot % P;
        for (int h = 0; h < Hkv; h++) {
            float ks = k_scales ? k_scales[h] : k_scale;
            float vs = v_scales ? v_scales[h] : v_scale;
            for (int d = 0; d < D; d++) {
                int64_t src = ((int64_t)t * Hkv + h) * D + d;
                int64_t dst = ((page * Hkv + h) * P + off) * D + d;
                if (kv_dtype == PKVO_BF16) {
                    ((uint16_t *)k_pool)[dst] = k_new[src];
                    ((uint16_t *)v_pool)[dst] = v_new[src];
                } else {
                    ((uint8_t *)k_pool)[dst] = pkvo_quantize_bf16(k_new[src], ks);
                    ((uint8_t *)v_pool)[dst] = pkvo_quantize_bf16(v_new[src], vs);
                }
            }
        }
    }
    return bad;
}

/* ---- attention for one (sequence, q head) -------------------------------- */

/* Attention of one query row over the first L tokens of a paged sequence.
 * Token i lives in page bt_row[i / P] at offset i % P.  Returns 0, or -1 if
 * a page id lies outside [0, num_blocks) (out is then zero). */
int pkvo_attention_one(const uint16_t *q_row, const void *k_pool,
                       const void *v_pool, int kv_dtype, float k_scale,
                       float v_scale, int64_t num_blocks, int Hkv, int P, int D,
                       int h, const int32_t *bt_row, int L, double scale,
                       double *out)
{
    double *z, m, den;
    for (int d = 0; d < D; d++)
        out[d] = 0.0;
    if (L <= 0)
        return 0;
    for (int j = 0; j < (L + P - 1) / P; j++)
        if (bt_row[j] < 0 || bt_row[j] >= num_blocks)
            return -1;
    z = (double *)malloc(sizeof(double) * (size_t)L);
    if (!z)
        return -2;
    /* scores: z_i = scale * <q, K_i> */
    for (int i = 0; i < L; i++) {
        int64_t base = (((int64_t)bt_row[i / P] * Hkv + h) * P + i % P) * D;
        double acc = 0.0;
        for (int d = 0; d < D; d++)
            acc += pkvo_bf16_value(q_row[d]) * kv_value(k_pool, kv_dtype, base + d, k_scale);
        z[i] = scale * acc;
    }
    /* max-subtracted softmax, then the weighted sum of V */
    m = z[0];
    for (int i = 1; i < L; i++)
        if (z[i] > m)
            m = z[i];
    den = 0.0;
    for (int i = 0; i < L; i++) {
        z[i] = exp(z[i] - m);
        den += z[i];
    }
    for (int i = 0; i < L; i++) {
        int64_t base = (((int64_t)bt_row[i / P] * Hkv + h) * P + i % P) * D;
        for (int d = 0; d < D; d++)
            out[d] += z[i] * kv_value(v_pool, kv_dtype, base + d, v_scale);
    }
    for (int d = 0; d < D; d++)
        out[d] /= den;
    free(z);
    return 0;
}

/* ---- decode: every (sequence, q head) ------------------------------------ */

/* q [B][Hq][D] bf16, block_tables [B][max_blocks], context_lens [B],
 * out [B][Hq][D] fp64.  FP8 scales per kv head when k_scales / v_scales are
 * given.  Returns the number of rows with a bad page id. */
int pkvo_paged_attention(const uint16_t *q, const void *k_pool, const void *v_pool,
                         int kv_dtype, float k_scale, float v_scale,
                         const float *k_scales, const float *v_scales,
                         int64_t num_blocks, int Hkv, int P, int D,
                         const int32_t *block_tables, int max_blocks,
                         const int32_t *context_lens, int B, int Hq,
                         double scale, double *out)
{
    int G = Hq / Hkv, bad = 0;
    for (int s = 0; s < B; s++)
        for (int a = 0; a < Hq; a++)
            bad += pkvo_attention_one(q + ((int64_t)s * Hq + a) * D, k_pool, v_pool,
                                      kv_dtype, k_scales ? k_scales[a / G] : k_scale,
                                      v_scales ? v_scales[a / G] : v_scale, num_blocks, Hkv, P,
                                      D, a / G, block_tables + (int64_t)s * max_blocks,
                                      context_lens[s], scale,
                                      out + ((int64_t)s * Hq + a) * D) != 0;
    return bad;
}

/* Selected (sequence, q head) rows only: out [n][D]. */
int pkvo_paged_attention_rows(const uint16_t *q, const void *k_pool,
                              const void *v_pool, int kv_dtype, float k_scale,
                              float v_scale, const float *k_scales,
                              const float *v_scales, int64_t num_blocks, int Hkv, int P,
                              int D, const int32_t *block_tables, int max_blocks,
                              const int32_t *context_lens, int Hq,
                              const int32_t *seq_ids, const int32_t *head_ids,
                              int n, double scale, double *out)
{
    int G = Hq / Hkv, bad = 0;
    for (int r = 0; r < n; r++) {
        int s = seq_ids[r], a = head_ids[r];
        bad += pkvo_attention_one(q + ((int64_t)s * Hq + a) * D, k_pool, v_pool,
                                  kv_dtype, k_scales ? k_scales[a / G] : k_scale,
                                  v_scales ? v_scales[a / G] : v_scale, num_blocks, Hkv, P, D,
                                  a / G, block_tables + (int64_t)s * max_blocks,
                                  context_lens[s], scale, out + (int64_t)r * D) != 0;
    }
    return bad;
}

/* ---- chunked prefill ----------------------------------------------------- */

/* q [T_p][Hq][D] packed: sequence s owns rows cu_seqlens_q[s] ..
 * cu_seqlens_q[s+1]-1, C_s of them; context_lens[s] = L_s counts the chunk.
 * Row i of sequence s attends to keys 0 .. L_s - C_s + i (causal over pages).
 * FP8 pools: scales per kv head when k_scales / v_scales are given, as in
 * the decode.  out [T_p][Hq][D] fp64. */
int pkvo_paged_prefill(const uint16_t *q, const int32_t *cu_seqlens_q,
                       const void *k_pool, const void *v_pool, int kv_dtype,
                       float k_scale, float v_scale, const float *k_scales,
                       const float *v_scales, int64_t num_blocks, int Hkv,
                       int P, int D, const int32_t *block_tables, int max_blocks,
                       const int32_t *context_lens, int n, int Hq, double scale,
                       double *out)
{
    int G = Hq / Hkv, bad = 0;
    for (int s = 0; s < n; s++) {
        int C = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        int L = context_lens[s];
        for (int i = 0; i < C; i++) {
            int64_t row = cu_seqlens_q[s] + i;
            int visible = L - C + i + 1;
            for (int a = 0; a < Hq; a++)
                bad += pkvo_attention_one(q + (row * Hq + a) * D, k_pool, v_pool,
                                          kv_dtype, k_scales ? k_scales[a / G] : k_scale,
                                          v_scales ? v_scales[a / G] : v_scale, num_blocks,
                                          Hkv, P, D, a / G,
                                          block_tables + (int64_t)s * max_blocks,
                                          visible, scale,
                                          out + (row * Hq + a) * D) != 0;
        }
    }
    return bad;
}
