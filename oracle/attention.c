/*
 * oracle/attention.c -- reference CPU attention for paged-KV grouped-query
 * attention.  TEST INFRASTRUCTURE ONLY: only tests/, __graft_entry__.smoke()
 * and bench.py's cpu_baseline / reference leg may load or call this code.
 * It shares no code, header, table or helper with the CUDA library, and
 * nothing in the library may call it.
 *
 * What it computes (the plain definition, written out):
 *
 *   "nx_f32_attn_paged.nx source", header comment: the paged path has the
 *   same math as the contiguous-cache path -- same attention core, same
 *   offset-causal query position q_pos = total_k - n_q + i, same GQA head
 *   grouping -- and only the K/V storage differs.  So the result the method
 *   reaches is dense attention over the sequence's logical K/V history.
 *
 *   "nx_f32_attn_paged.nx source", step 2 ("Total keys = past + new"):
 *   total_k = seq_len + n_tokens, the new rows already appended.
 *
 *   "nx_f32_attn_paged.nx source", step 3 (per-head loop) and
 *   "nx_f32_gqa_attention.nx source" (the GQA wrapper): query head h reads
 *   kv head h / (n_heads / n_kv_heads).
 *
 *   For each query row i and query head h:
 *     q_pos   = total_k - n_q + i
 *     visible = { j : 0 <= j <= q_pos }      (causal != 0)
 *             = { j : 0 <= j <  total_k }    (causal == 0, the bidirectional
 *                                             core of the GQA self-test)
 *     s_j     = scale * sum_d Q[i, h, d] * K[j, h/g, d]
 *     out[i, h, :] = sum_j exp(s_j - max s) V[j, h/g, :] / sum_j exp(s_j - max s)
 *
 * Precision: the pages store f32 values and do not show the core's
 * arithmetic order.  This oracle widens every f32 input to double, forms
 * each product exactly in double (24 + 24 significant bits fit in 53),
 * accumulates in double, uses exp() in double, and rounds once to f32 at the
 * end.  It is therefore the correctly computed result to well below f32
 * resolution, which is what a tolerance is measured against.
 *
 * Threads: the (query row, query head) pairs are independent, and each is
 * computed by one thread in the order written below, so the result does not
 * depend on the thread count (oracle_set_threads; OpenMP when the build has
 * it, else one thread).  The build turns off contraction of a*b+c into fused
 * multiply-adds, so every host gives the same bits.
 *
 * Validation order and return codes follow the argument checks at the top
 * of nx_f32_attn_with_paged ("nx_f32_attn_paged.nx source"): non-positive
 * sizes -> 1 (bad dim), n_heads not a multiple of n_kv_heads -> 2 (bad GQA).
 * A history shorter than the query block (total_k < n_q) is also a bad dim.
 *
 * Layouts (row-major f32, as in "nx_f32_gqa_attention.nx source", header):
 *   Q, out : [n_q, n_heads * head_dim]
 *   K, V   : [total_k, n_kv_heads * head_dim]  (the contiguous history)
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_BAD_DIM 1
#define ORACLE_ERR_BAD_GQA 2
#define ORACLE_ERR_NOMEM 9

static int g_threads = 1;

/* Threads used by oracle_attend from now on (n < 1: all the host offers);
 * returns the count in effect (1 without OpenMP). */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    g_threads = n < 1 ? omp_get_num_procs() : n;
#else
    (void)n;
    g_threads = 1;
#endif
    return g_threads;
}

int oracle_attend(const float *Q, const float *K, const float *V,
                  int n_q, int total_k, int n_heads, int n_kv_heads,
                  int head_dim, int causal, float scale, float *out)
{
    if (n_q <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_ERR_BAD_DIM;
    if (n_heads % n_kv_heads != 0)
        return ORACLE_ERR_BAD_GQA;
    if (total_k < n_q)
        return ORACLE_ERR_BAD_DIM;

    const int group = n_heads / n_kv_heads;
    const size_t q_dim = (size_t)n_heads * head_dim;
    const size_t kv_dim = (size_t)n_kv_heads * head_dim;

    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(g_threads) reduction(| : failed)
#endif
    {
        /* per-thread scratch; every thread takes part in the loop below
           (a thread whose allocation failed marks its pairs as failed) */
        double *s = (double *)malloc((size_t)total_k * sizeof(double));
        double *acc = (double *)malloc((size_t)head_dim * sizeof(double));
        {
#ifdef _OPENMP
#pragma omp for collapse(2) schedule(dynamic, 1)
#endif
            for (int i = 0; i < n_q; i++) {
                for (int h = 0; h < n_heads; h++) {
                    if (!s || !acc) {
                        failed = 1;
                        continue;
                    }
                    const int q_pos = total_k - n_q + i;
                    const int n_visible = causal ? q_pos + 1 : total_k;
                    const int kv_head = h / group;
                    const float *q = Q + (size_t)i * q_dim + (size_t)h * head_dim;

                    /* scores over the visible keys, and their maximum */
                    double m = -INFINITY;
                    for (int j = 0; j < n_visible; j++) {
                        const float *k = K + (size_t)j * kv_dim + (size_t)kv_head * head_dim;
                        double dot = 0.0;
                        for (int d = 0; d < head_dim; d++)
                            dot += (double)q[d] * (double)k[d];
                        s[j] = (double)scale * dot;
                        if (s[j] > m)
                            m = s[j];
                    }

                    /* softmax-weighted sum of the visible value rows */
                    double denom = 0.0;
                    for (int d = 0; d < head_dim; d++)
                        acc[d] = 0.0;
                    for (int j = 0; j < n_visible; j++) {
                        const double p = exp(s[j] - m);
                        const float *v = V + (size_t)j * kv_dim + (size_t)kv_head * head_dim;
                        denom += p;
                        for (int d = 0; d < head_dim; d++)
                            acc[d] += p * (double)v[d];
                    }

                    float *o = out + (size_t)i * q_dim + (size_t)h * head_dim;
                    for (int d = 0; d < head_dim; d++)
                        o[d] = (float)(acc[d] / denom);
                }
            }
        }
        free(s);
        free(acc);
    }
    if (failed)
        return ORACLE_ERR_NOMEM;
    return ORACLE_OK;
}
