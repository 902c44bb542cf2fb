/*
 * fp64 CPU oracle for speculative-decoding verification attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may build, load or call it; the library
 * itself never does.  It shares no code, header or constant with the CUDA
 * sources.
 *
 * What it computes (LongSpec, section 2.C "Hybrid Tree Attention"): the
 * divide-and-aggregate split of verification attention -- an unmasked pass over
 * the cached history plus a masked pass over the speculative tokens, merged by
 * log-sum-exp -- is exact, so its result equals ordinary masked softmax
 * attention over the union of keys.  The oracle therefore evaluates that union
 * directly from an EXPLICIT full visibility matrix, one (query token, head) row
 * at a time, in double precision:
 *
 *     z_n   = scale * sum_d q[i,h,d] * k[n,kv(h),d]          n visible to i
 *     lse   = ln sum_n exp(z_n)        (as max + ln sum exp(z - max))
 *     out   = sum_n exp(z_n - lse) * v[n,kv(h),:]
 *
 * with kv(h) = h / (Hq / Hkv) (contiguous GQA groups).  A row that sees no key
 * gets out = 0 and lse = -inf.
 *
 * Inputs are widened exactly: bf16 bit patterns become fp32 by a 16-bit left
 * shift (the definition of bfloat16) and then fp64.
 *
 * Also here: the log-sum-exp merge of partial attentions (LongSpec 2.C, the
 * "Log-Sum-Exp fusion") and the ancestor-or-self visibility of a token tree
 * given by parent pointers (LongSpec 1.3 / 2.C: branch-specific tree masks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_BF16 = 0, ORACLE_F32 = 2, ORACLE_F64 = 3 };

static double widen(const void *base, int dtype, size_t i) {
  if (dtype == ORACLE_BF16) {
    uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  if (dtype == ORACLE_F32) return (double)((const float *)base)[i];
  return ((const double *)base)[i];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Masked attention of one sequence over an explicit key list.
 *   q        [T][Hq][D]        (dtype q_dtype)
 *   k, v     [n_keys][Hkv][D]  (dtype kv_dtype), key rows in any order
 *   visible  [T][n_keys]       1 = query token i may attend key n
 *   out      [T][Hq][D]  fp64
 *   lse      [Hq][T]     fp64 (natural log)
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_masked_attention(int T, int Hq, int Hkv, int D, double scale, long long n_keys,
                            const void *q, int q_dtype, const void *k, const void *v, int kv_dtype,
                            const unsigned char *visible, double *out, double *lse) {
  if (T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || n_keys < 0 || Hq % Hkv != 0) return -1;
  const int group = Hq / Hkv;
  int failed = 0;
#pragma omp parallel
  {
    double *z = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    if (!z || !acc) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for collapse(2) schedule(dynamic, 1)
    for (int h = 0; h < Hq; ++h) {
      for (int i = 0; i < T; ++i) {
        if (!z || !acc) continue;
        const int kvh = h / group;
        const unsigned char *vis = visible + (size_t)i * (size_t)n_keys;
        double zmax = -INFINITY;
        long long n_vis = 0;
        for (long long n = 0; n < n_keys; ++n) {
          if (!vis[n]) continue;
          double s = 0.0;
          for (int d = 0; d < D; ++d) {
            s += widen(q, q_dtype, ((size_t)i * Hq + h) * D + d) *
                 widen(k, kv_dtype, ((size_t)n * Hkv + kvh) * D + d);
          }
          z[n] = scale * s;
          if (z[n] > zmax) zmax = z[n];
          ++n_vis;
        }
        double *o = out + ((size_t)i * Hq + h) * D;
        if (n_vis == 0) {
          for (int d = 0; d < D; ++d) o[d] = 0.0;
          lse[(size_t)h * T + i] = -INFINITY;
          continue;
        }
        double sum = 0.0;
        for (long long n = 0; n < n_keys; ++n)
          if (vis[n]) sum += exp(z[n] - zmax);
        const double l = zmax + log(sum);
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (long long n = 0; n < n_keys; ++n) {
          if (!vis[n]) continue;
          const double p = exp(z[n] - l);
          for (int d = 0; d < D; ++d) acc[d] += p * widen(v, kv_dtype, ((size_t)n * Hkv + kvh) * D + d);
        }
        for (int d = 0; d < D; ++d) o[d] = acc[d];
        lse[(size_t)h * T + i] = l;
      }
    }
    free(z);
    free(acc);
  }
  return failed ? -1 : 0;
}

/*
 * Log-sum-exp merge of n_parts partial attentions of the same query rows.
 *   o_parts   [n_parts][n_rows][D]  each part normalised over its own keys
 *   lse_parts [n_parts][n_rows]     natural-log partition of each part
 *   out       [n_rows][D], lse [n_rows]
 * lse = ln sum_s exp(lse_s);  out = sum_s exp(lse_s - lse) * o_s.
 * A part with lse_s = -inf contributes nothing; if every part is empty the
 * row gets out = 0, lse = -inf.
 */
void oracle_lse_merge(int n_parts, long long n_rows, int D, const double *o_parts,
                      const double *lse_parts, double *out, double *lse) {
  for (long long r = 0; r < n_rows; ++r) {
    double m = -INFINITY;
    for (int s = 0; s < n_parts; ++s) {
      const double a = lse_parts[(size_t)s * n_rows + r];
      if (a > m) m = a;
    }
    double *o = out + (size_t)r * D;
    if (m == -INFINITY) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int s = 0; s < n_parts; ++s) sum += exp(lse_parts[(size_t)s * n_rows + r] - m);
    const double l = m + log(sum);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int s = 0; s < n_parts; ++s) {
      const double w = exp(lse_parts[(size_t)s * n_rows + r] - l);
      const double *os = o_parts + ((size_t)s * n_rows + r) * D;
      for (int d = 0; d < D; ++d) o[d] += w * os[d];
    }
    lse[r] = l;
  }
}

/*
 * Ancestor-or-self visibility of a token tree.
 *   parent   [T]  -1 for a root, otherwise 0 <= parent[i] < i (topological
 *                  order; node 0 is always a root, several roots make a forest)
 *   visible  [T][T]  visible[i][j] = 1 iff j lies on the path from i to its root
 * Returns 0, or -1 if parent is not in that form.
 */
int oracle_tree_visibility(int T, const int32_t *parent, unsigned char *visible) {
  for (int i = 0; i < T; ++i) {
    if (parent[i] < -1 || parent[i] >= i) return -1;
  }
  memset(visible, 0, (size_t)T * (size_t)T);
  for (int i = 0; i < T; ++i) {
    int j = i;
    while (j >= 0) {
      visible[(size_t)i * T + j] = 1;
      j = parent[j];
    }
  }
  return 0;
}
