/*
 * fp64 CPU oracle for attention forward — TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  It shares no code with the CUDA path.
 *
 * What it computes is the plain definition of scaled dot-product attention,
 *     O = softmax(Q K^T * scale + mask) V,
 * as stated on the jsqmd page "CANN Transformer算子库ops-transformer深度实践",
 * §二 "SelfAttention的基础实现与瓶颈" (the formula softmax(QK^T/sqrt(d))V) and in
 * its `naive_attention` sketch, and on the agent.csdn.net BERT walkthrough,
 * 第一章 (BertSelfAttention.forward: matmul, additive mask, softmax, matmul).
 * The softmax is the max-subtracted form exp(x - max) / sum exp(x - max) of the
 * hwcomputing.csdn.net page, §2.2 "数值稳定性优化".  Because FlashAttention is an
 * exact reformulation, the oracle is that definition written out row by row:
 * every score of a row is materialised in fp64, masked, and reduced.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - causal alignment is bottom-right: query row i of a sequence with Lq
 *    queries and Lk keys sits at absolute position p = i + Lk - Lq and may see
 *    key j iff j <= p (the jsqmd page, §二 "因果掩码与解码优化", says only that a
 *    position sees the ones before it);
 *  - sliding window w > 0: with causal, keys p - w < j <= p (the window holds
 *    the diagonal, so w = 1 keeps only key p); without causal, |p - j| < w;
 *    w <= 0 means no window (the jsqmd page, §一 "核心能力矩阵", names the mode only);
 *  - MQA/GQA: query head h reads KV head floor(h * Hkv / Hq) (contiguous groups);
 *  - a row with no allowed key has O = 0 and LSE = -inf (log of an empty sum);
 *  - LSE is the natural log of the row's normaliser in scaled-score units,
 *    LSE_i = M_i + ln(sum_j exp(s_ij - M_i)).
 *  - ALiBi (optional): the jsqmd page, §三 "ALiBi位置编码的线性偏置", adds -m * |i - j|
 *    to each scaled score, m a per-head slope; the pages give no slope values, so
 *    the caller passes them, and i is the query's absolute position p (the same
 *    bottom-right alignment as the causal mask): s_ij = scale q.k - m_h |p - j|.
 *
 * Inputs are raw bf16 bit patterns (uint16); bf16 -> fp64 is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Is key j visible from absolute query position p?  (readings above) */
static int key_allowed(long p, long j, int causal, int window) {
  if (causal) {
    if (j > p) return 0;
    if (window > 0 && j <= p - window) return 0;
    return 1;
  }
  if (window > 0) {
    long dist = p - j;
    if (dist < 0) dist = -dist;
    if (dist >= window) return 0;
  }
  return 1;
}

/*
 * Compute selected output rows.
 *
 *  q      bf16 bits, row r of sequence b at element ((q_off[b] + r) * Hq + h) * d
 *  k, v   bf16 bits, row j of sequence b at element ((k_off[b] + j) * Hkv + g) * d
 *  len_q, len_k   per-sequence valid lengths
 *  alibi_slopes  NULL, or Hq per-head slopes m_h (bias -m_h |p - j| on the scaled score)
 *  rows   n_rows triples (b, h, i)
 *  o_out  [n_rows, d] fp64;  lse_out [n_rows] fp64
 *  work   scratch of n_threads * max_len_k doubles is allocated internally
 *
 * Returns 0, or -1 if a scratch allocation failed or an index is out of range.
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          int B, int Hq, int Hkv, int d,
                          const long* q_off, const int* len_q,
                          const long* k_off, const int* len_k,
                          double scale, int causal, int window, const double* alibi_slopes,
                          int n_rows, const int* rows_bhi,
                          double* o_out, double* lse_out, int n_threads) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return -1;
  int max_lk = 0;
  for (int b = 0; b < B; ++b)
    if (len_k[b] > max_lk) max_lk = len_k[b];
  int bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel reduction(| : bad)
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
    char* ok = (char*)malloc((size_t)(max_lk > 0 ? max_lk : 1));
    if (!s || !ok) bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (int n = 0; n < n_rows; ++n) {
      if (!s || !ok) continue;
      int b = rows_bhi[3 * n], h = rows_bhi[3 * n + 1], i = rows_bhi[3 * n + 2];
      double* o = o_out + (size_t)n * d;
      if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= len_q[b]) {
        bad = 1;
        continue;
      }
      int g = h / (Hq / Hkv); /* = floor(h * Hkv / Hq) for contiguous groups */
      long Lq = len_q[b], Lk = len_k[b];
      long p = (long)i + Lk - Lq;
      const uint16_t* qi = q + ((size_t)(q_off[b] + i) * Hq + h) * d;
      /* scores of the row */
      double M = -INFINITY;
      int any = 0;
      for (long j = 0; j < Lk; ++j) {
        ok[j] = (char)key_allowed(p, j, causal, window);
        if (!ok[j]) continue;
        const uint16_t* kj = k + ((size_t)(k_off[b] + j) * Hkv + g) * d;
        double dot = 0.0;
        for (int t = 0; t < d; ++t) dot += bf16_to_f64(qi[t]) * bf16_to_f64(kj[t]);
        s[j] = scale * dot;
        if (alibi_slopes) s[j] -= alibi_slopes[h] * fabs((double)(p - j));
        if (!any || s[j] > M) M = s[j];
        any = 1;
      }
      for (int t = 0; t < d; ++t) o[t] = 0.0;
      if (!any) {
        lse_out[n] = -INFINITY;
        continue;
      }
      /* softmax with the row max subtracted, then P V */
      double Z = 0.0;
      for (long j = 0; j < Lk; ++j)
        if (ok[j]) Z += exp(s[j] - M);
      for (long j = 0; j < Lk; ++j) {
        if (!ok[j]) continue;
        double pj = exp(s[j] - M) / Z;
        const uint16_t* vj = v + ((size_t)(k_off[b] + j) * Hkv + g) * d;
        for (int t = 0; t < d; ++t) o[t] += pj * bf16_to_f64(vj[t]);
      }
      lse_out[n] = M + log(Z);
    }
    free(s);
    free(ok);
  }
  return bad ? -1 : 0;
}

/* Number of threads OpenMP would use (1 when built without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
