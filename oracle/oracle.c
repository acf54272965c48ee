/*
 * oracle.c -- plain fp64 CPU oracle for grouped-query attention (GQA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant with the CUDA
 * library; the only thing both sides share is the seeded input generator.
 *
 * Sources (cited by page title and section):
 *   [GQA-BERT]  "3个GQA核心优化技巧：解决BERT模型内存效率与吞吐量瓶颈"
 *               (blog.gitcode.com), sections "GQA的分组共享机制" (query heads
 *               share one K/V head per group, Hq % Hkv == 0, group size
 *               Hq / Hkv) and "Flash-Attention的稀疏分组优化" (the K/V head of
 *               query head h is h / group_size); "阶段二" (softmax scale
 *               1/sqrt(d_head), causal off for BERT).
 *   [GQA-PAPER] "GQA: Training Generalized Multi-Query Transformer Models
 *               from Multi-Head Checkpoints" (azimuth.plus/paper/gqa),
 *               "Idea 2: grouped attention" (GQA-H = MHA, GQA-1 = MQA) and
 *               the mean-pooling code listing, whose slice g*hpg:(g+1)*hpg
 *               fixes contiguous groups of heads.
 *   [LOWRANK]   aifullclass.xyz article on BERT multi-head self-attention,
 *               code example: scores = QK^T / sqrt(d); masked_fill(mask==0);
 *               softmax over keys; weights times V.
 *   [FA-SERIES] "FlashAttention Serisi: Bellek G/Ç Tıkanıklığının Çözümü"
 *               (webturing.pages.dev), "Ana fikir" and FAQ: the tiled online
 *               softmax computes the mathematically identical result, so the
 *               oracle is the plain two-pass definition, not a tiled one.
 *
 * Definition computed, for every batch b, query head h, query row i:
 *   G   = Hq / Hkv ;  kvh = h / G                      [GQA-BERT], [GQA-PAPER]
 *   Lb  = seqlens_k ? seqlens_k[b] : Sk                (right padding of keys)
 *   J   = { j : 0 <= j < Lb and (!causal or j <= i + Sk - Sq) }
 *   s_j = scale * sum_d q[b,i,h,d] * k[b,j,kvh,d]       [LOWRANK]
 *   m   = max_{j in J} s_j ;  l = sum_{j in J} exp(s_j - m)
 *   out[b,i,h,:] = sum_{j in J} exp(s_j - m) / l * v[b,j,kvh,:]
 *   lse[b,h,i]   = m + ln(l)
 *   J empty  ->  out = 0, lse = -inf.
 * Masked keys are left out of J, which gives them exactly zero weight (the
 * page's -1e9 fill is read as "never attended").
 *
 * Layouts (row-major, contiguous):
 *   q   [B, Sq, Hq, D]          float32 holding the exact input values
 *   k,v [B, Skcap, Hkv, D]      float32; Skcap >= Sk is the row capacity per
 *                               batch entry (a KV cache has Skcap = Smax)
 *   out [B, Sq, Hq, D] double   (or [nrows, D] when rows != NULL)
 *   lse [B, Hq, Sq]    double   (or [nrows]    when rows != NULL)
 * All arithmetic is fp64 on the inputs widened from float32.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* One (b, h, i) row of the definition above, written out term by term. */
static void oracle_row(const float* q, const float* k, const float* v,
                       int Hq, int Hkv, int Sq, int Sk, int Skcap, int D,
                       double scale, int causal, int Lb,
                       int b, int h, int i, double* s_buf,
                       double* out_row, double* lse_out)
{
    const int G = Hq / Hkv;
    const int kvh = h / G;
    const float* qrow = q + (((int64_t)b * Sq + i) * Hq + h) * (int64_t)D;

    /* pass 1: scores over the admissible key set J, and their maximum */
    int nJ = 0;
    double m = -INFINITY;
    for (int j = 0; j < Lb; ++j) {
        if (causal && (int64_t)j > (int64_t)i + Sk - Sq) break;
        const float* krow = k + (((int64_t)b * Skcap + j) * Hkv + kvh) * (int64_t)D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)krow[d];
        double s = scale * dot;
        s_buf[j] = s;
        if (s > m) m = s;
        nJ = j + 1;
    }
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    if (nJ == 0) {              /* empty key set: zero output, lse = -inf */
        *lse_out = -INFINITY;
        return;
    }
    /* pass 2: normaliser l and the weighted sum of V rows */
    double l = 0.0;
    for (int j = 0; j < nJ; ++j) l += exp(s_buf[j] - m);
    for (int j = 0; j < nJ; ++j) {
        const double w = exp(s_buf[j] - m) / l;
        const float* vrow = v + (((int64_t)b * Skcap + j) * Hkv + kvh) * (int64_t)D;
        for (int d = 0; d < D; ++d) out_row[d] += w * (double)vrow[d];
    }
    *lse_out = m + log(l);
}

/*
 * Full or row-sampled GQA attention.  rows[r] = (b * Hq + h) * Sq + i picks
 * the rows to compute (same order as lse); rows == NULL computes all of them.
 * Returns ORACLE_OK or ORACLE_BAD_ARG (Hq % Hkv != 0 per [GQA-BERT], any
 * non-positive size, Skcap < Sk, or a key length outside [0, Sk]).
 */
int oracle_gqa_attention(const float* q, const float* k, const float* v,
                         double* out, double* lse,
                         int B, int Hq, int Hkv, int Sq, int Sk, int Skcap, int D,
                         double scale, int causal, const int* seqlens_k,
                         const int64_t* rows, int64_t nrows)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return ORACLE_BAD_ARG;
    if (Hq % Hkv != 0 || Skcap < Sk) return ORACLE_BAD_ARG;
    if (seqlens_k)
        for (int b = 0; b < B; ++b)
            if (seqlens_k[b] < 0 || seqlens_k[b] > Sk) return ORACLE_BAD_ARG;
    const int64_t total = (int64_t)B * Hq * Sq;
    const int64_t n = rows ? nrows : total;
    if (rows)
        for (int64_t r = 0; r < n; ++r)
            if (rows[r] < 0 || rows[r] >= total) return ORACLE_BAD_ARG;
    int failed = 0;
#pragma omp parallel
    {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)Sk);
        if (!s_buf) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < n; ++r) {
                const int64_t idx = rows ? rows[r] : r;
                const int i = (int)(idx % Sq);
                const int h = (int)((idx / Sq) % Hq);
                const int b = (int)(idx / ((int64_t)Sq * Hq));
                const int Lb = seqlens_k ? seqlens_k[b] : Sk;
                double* orow = rows ? out + r * (int64_t)D
                                    : out + (((int64_t)b * Sq + i) * Hq + h) * (int64_t)D;
                double* lrow = rows ? lse + r : lse + idx;
                oracle_row(q, k, v, Hq, Hkv, Sq, Sk, Skcap, D, scale, causal, Lb,
                           b, h, i, s_buf, orow, lrow);
            }
            free(s_buf);
        }
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Single-token decode over a per-sequence KV cache: the new token attends to
 * the whole cached prefix [0, cache_seqlens[b]) with no causal term
 * ([GQA-PAPER] "Problem"/"Bottleneck": every generation step reads all cached
 * keys and values).  It is the definition above with Sq = 1, Sk = Skcap =
 * Smax and seqlens_k = cache_seqlens.
 *   q [B, Hq, D]; kcache, vcache [B, Smax, Hkv, D]; out [B, Hq, D]; lse [B, Hq]
 */
int oracle_gqa_decode(const float* q, const float* kcache, const float* vcache,
                      const int* cache_seqlens, double* out, double* lse,
                      int B, int Hq, int Hkv, int D, int Smax, double scale)
{
    return oracle_gqa_attention(q, kcache, vcache, out, lse, B, Hq, Hkv, 1, Smax, Smax, D,
                                scale, 0, cache_seqlens, NULL, 0);
}
