/*
 * attn_oracle.c -- plain fp64 CPU attention: the checker the CUDA path is held to.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg do.
 *
 * What it computes is the plain definition of the attention the pages lower:
 *
 *   "AttentionRegion Transformation - Deriving FlashAttention via Memory-Centric
 *    Compilation in AICF", section 3 (Attention Pattern Detection):
 *        Scores = MatMul(Q, K^T);  Scores = Mask(Scores) (optional);
 *        Scores = Softmax(Scores); Output = MatMul(Scores, V)
 *   with the softmax in the stable canonical form of "AI Compiler pipeline stages"
 *   (IR Normalization): exp(x - max x) / sum exp(x - max x), evaluated in two passes.
 *   The score scale sits before the mask ("ADR-0060: AHBM GQA Fused Attention Kernel
 *   (Llama3-70B)", section 3: the scale epilogue is applied to Q.K^T, then the additive
 *   mask is added).
 *
 * For every output row (b, h, i) the whole score row over the keys is materialised
 * (Skv doubles), softmaxed in two passes and contracted with V.  Rows are independent
 * by definition, so a caller may ask for a subset of rows only (full-size parity checks
 * on sampled rows).
 *
 * Readings of what the pages leave open (each is listed in the design notes):
 *  - GQA: query head h reads KV head h / G with G = Hq / Hkv (contiguous groups;
 *    ADR-0060 section 0 stacks "the group's G query heads" of one KV head).
 *  - Causal alignment is bottom-right: query i sits at key position i + (Skv - Sq);
 *    key j is visible iff j <= i + Skv - Sq (ADR-0060 section 5.4 classifies tiles by
 *    global positions; decode with Sq = 1 then sees every key, section 5.2).
 *  - LSE is the natural log of sum_j exp(scale * q.k_j) over the visible keys.
 *  - A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Inputs are Q [B,Hq,Sq,d], K and V [B,Hkv,Skv_max,d], row-major, given either as fp32
 * or as bf16 bit patterns; both are widened exactly to double.  kv_len (nullable) gives
 * the number of valid keys of each batch entry (decode caches); rows past it are never
 * read.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_IN_F32 = 0, ORACLE_IN_BF16 = 1 };

static double widen(const void* base, int dtype, long long idx) {
    if (dtype == ORACLE_IN_F32) return (double)((const float*)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* One output row: o_row[d], *lse_row.  Returns 0. */
static void attention_row(const void* q, const void* k, const void* v, int dtype,
                          int Hq, int Hkv, int Sq, int Skv_max, int skv, int d,
                          double scale, int causal, int b, int h, int i,
                          double* s_row, double* q_row, double* o_row, double* lse_row) {
    const int G = Hq / Hkv;
    const int kvh = h / G;
    const long long q_off = (((long long)b * Hq + h) * Sq + i) * d;
    const long long kv_off = ((long long)b * Hkv + kvh) * (long long)Skv_max * d;
    int n_visible = skv;
    if (causal) {
        long long lim = (long long)i + (long long)skv - (long long)Sq + 1; /* keys j < lim */
        if (lim < 0) lim = 0;
        if (lim < n_visible) n_visible = (int)lim;
    }
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    if (n_visible <= 0) {
        *lse_row = -INFINITY;
        return;
    }
    for (int c = 0; c < d; ++c) q_row[c] = widen(q, dtype, q_off + c);

    /* S = scale * q . k_j, then the additive mask (-inf beyond the visible keys). */
    for (int j = 0; j < skv; ++j) {
        if (j >= n_visible) {
            s_row[j] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        const long long kj = kv_off + (long long)j * d;
        for (int c = 0; c < d; ++c) acc += q_row[c] * widen(k, dtype, kj + c);
        s_row[j] = scale * acc;
    }
    /* pass 1: row max */
    double m = -INFINITY;
    for (int j = 0; j < skv; ++j)
        if (s_row[j] > m) m = s_row[j];
    /* pass 2: exponentials and their sum */
    double l = 0.0;
    for (int j = 0; j < skv; ++j) {
        s_row[j] = exp(s_row[j] - m); /* exp(-inf) = 0 for masked keys */
        l += s_row[j];
    }
    /* P = e / l, O = P V */
    for (int j = 0; j < skv; ++j) {
        const double p = s_row[j] / l;
        if (p == 0.0) continue;
        const long long vj = kv_off + (long long)j * d;
        for (int c = 0; c < d; ++c) o_row[c] += p * widen(v, dtype, vj + c);
    }
    *lse_row = m + log(l);
}

/*
 * oracle_attention: O and LSE for all rows (rows == NULL) or for the listed flat row
 * ids r = (b * Hq + h) * Sq + i (rows != NULL, nrows entries; output row n holds r[n]).
 * o: [nrows or B*Hq*Sq, d] doubles, lse: [nrows or B*Hq*Sq] doubles.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attention(const void* q, const void* k, const void* v, int dtype,
                     double* o, double* lse, int B, int Hq, int Hkv, int Sq, int Skv_max,
                     const int* kv_len, int d, double scale, int causal,
                     const long long* rows, long long nrows, int nthreads) {
    if (!q || !k || !v || !o || !lse) return -1;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv_max <= 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if (dtype != ORACLE_IN_F32 && dtype != ORACLE_IN_BF16) return -1;
    const long long total = rows ? nrows : (long long)B * Hq * Sq;
    if (kv_len)
        for (int b = 0; b < B; ++b)
            if (kv_len[b] < 0 || kv_len[b] > Skv_max) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double* s_row = (double*)malloc(sizeof(double) * (size_t)Skv_max);
        double* q_row = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s_row || !q_row) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long long n = 0; n < total; ++n) {
                const long long r = rows ? rows[n] : n;
                if (r < 0 || r >= (long long)B * Hq * Sq) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                const int i = (int)(r % Sq);
                const int h = (int)((r / Sq) % Hq);
                const int b = (int)(r / ((long long)Sq * Hq));
                const int skv = kv_len ? kv_len[b] : Skv_max;
                attention_row(q, k, v, dtype, Hq, Hkv, Sq, Skv_max, skv, d, scale, causal, b,
                              h, i, s_row, q_row, o + n * d, lse + n);
            }
        }
        free(s_row);
        free(q_row);
    }
    return bad ? -1 : 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
