/*
 * ORACLE -- plain fp64 CPU attention forward.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the bench's CPU-baseline leg may
 * load this file's library.  It shares no code, header, table or helper with the
 * CUDA library, and the product path never calls it.
 *
 * What it computes (the plain definition the FlashAttention-2 forward reaches
 * exactly, up to rounding order):
 *   for every batch b, head h and query row i,
 *     s_j  = scale * sum_d q[i,d] k[j,d]      for every visible key j
 *     m    = max_j s_j,   w_j = exp(s_j - m),   l = sum_j w_j
 *     O[i] = sum_j w_j v[j] / l,                L[i] = m + ln l
 *   Visible: j < N, and j <= i when causal (top-left aligned).
 * Sources: "From FlashAttention to FlashAttention 2", Background: FlashAttention 1
 * (standard attention softmax(QK^T/sqrt d)V and the stored logsumexp
 * L = m + log l); "FlashAttention-2 from PyTorch to Triton", introduction
 * (L_i = m_i + log l_i = log sum_k exp S_ik) and its test file's reference
 * (masked scores, logsumexp over the last axis); "Writing FlashAttention 2 in
 * Triton", Step 4 (causal: query row m sees key n iff m >= n).
 *
 * A second entry point, oracle_attn_fwd_tiled, runs the pages' tiled online
 * softmax recurrence in fp64 (query tiles outer, key tiles inner, running m, l
 * and unnormalised O rescaled by exp(m_old - m_new), one divide at the end;
 * "FlashAttention-2 from PyTorch to Triton", the PyTorch FlashAttentionPytorch
 * forward and the Triton kernel's inner loop).  It exists to pin the identity
 * "tiled recurrence == two-pass softmax" that the GPU path relies on.
 *
 * Inputs are the same host arrays the GPU receives: dtype 0 = bf16 bit
 * patterns, 1 = fp32, 2 = fp64 (oracle-only, for closed-form pins).  Every
 * element is widened to fp64 before use, so the oracle measures only the
 * kernel's arithmetic error.  Layouts: q [B,H,M,D], k and v [B,H,N,D],
 * o [B,H,M,D] fp64, lse [B,H,M] fp64, all contiguous.
 *
 * Grouped-query attention ("From FlashAttention to FlashAttention 2", Layer 8:
 * Multi-Query / Grouped-Query Attention): k and v hold Hkv heads, Hkv divides H,
 * and query head h reads key/value head h / (H / Hkv) of the same batch entry.
 * Hkv == H is ordinary multi-head attention.
 *
 * Return value: 0 on success, -1 on invalid sizes, -2 on allocation failure,
 * -3 if a row had no visible key (cannot happen for N >= 1).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen(const void* base, int64_t idx, int dtype) {
  if (dtype == 0) {
    uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
  }
  if (dtype == 1) return (double)((const float*)base)[idx];
  return ((const double*)base)[idx];
}

static int check_sizes(int B, int H, int Hkv, int M, int N, int D, int dtype) {
  if (B <= 0 || H <= 0 || Hkv <= 0 || M <= 0 || N <= 0 || D <= 0) return -1;
  if (H % Hkv != 0) return -1;
  if (dtype < 0 || dtype > 2) return -1;
  return 0;
}

/* Flat key/value head index read by flat query head bh = b*H + h. */
static int64_t kv_head(int64_t bh, int H, int Hkv) {
  return (bh / H) * Hkv + (bh % H) / (H / Hkv);
}

/* Number of keys visible to query row i. */
static int64_t visible_keys(int64_t i, int N, int causal) {
  if (!causal) return N;
  return (i + 1 < N) ? i + 1 : N;
}

/* One query row of one (b,h): the definition, with all scores of the row formed
 * explicitly.  w must hold N doubles. */
static int attn_row(const void* q, const void* k, const void* v, int dtype,
                    int64_t bh, int64_t kvh, int64_t i, int M, int N, int D, double scale,
                    int causal, double* o_row, double* lse, double* w) {
  const int64_t qoff = (bh * M + i) * (int64_t)D;
  const int64_t kvoff = kvh * (int64_t)N * D;
  const int64_t nvis = visible_keys(i, N, causal);
  if (nvis <= 0) return -3;

  double m = -INFINITY;
  for (int64_t j = 0; j < nvis; ++j) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += widen(q, qoff + d, dtype) * widen(k, kvoff + j * D + d, dtype);
    w[j] = scale * dot;
    if (w[j] > m) m = w[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    w[j] = exp(w[j] - m);
    l += w[j];
  }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int64_t j = 0; j < nvis; ++j) acc += w[j] * widen(v, kvoff + j * D + d, dtype);
    o_row[d] = acc / l;
  }
  *lse = m + log(l);
  return 0;
}

/* Every row of every (b,h); k and v hold Hkv heads. */
int oracle_attn_fwd_gqa(const void* q, const void* k, const void* v, double* o, double* lse,
                        int B, int H, int Hkv, int M, int N, int D, double scale, int causal,
                        int dtype) {
  if (check_sizes(B, H, Hkv, M, N, D, dtype)) return -1;
  const int64_t rows = (int64_t)B * H * M;
  int status = 0;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)N);
    if (!w) {
#pragma omp atomic write
      status = -2;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t r = 0; r < rows; ++r) {
        int64_t bh = r / M, i = r % M;
        int rc = attn_row(q, k, v, dtype, bh, kv_head(bh, H, Hkv), i, M, N, D, scale, causal,
                          o + r * D, lse + r, w);
        if (rc) {
#pragma omp atomic write
          status = rc;
        }
      }
      free(w);
    }
  }
  return status;
}

/* Only the listed rows; rows[t] is the flat row index (b*H + h)*M + i.
 * o is [nrows, D], lse is [nrows]. */
int oracle_attn_fwd_gqa_rows(const void* q, const void* k, const void* v,
                             const int64_t* rows, int64_t nrows, double* o, double* lse,
                             int B, int H, int Hkv, int M, int N, int D, double scale,
                             int causal, int dtype) {
  if (check_sizes(B, H, Hkv, M, N, D, dtype)) return -1;
  const int64_t total = (int64_t)B * H * M;
  for (int64_t t = 0; t < nrows; ++t)
    if (rows[t] < 0 || rows[t] >= total) return -1;
  int status = 0;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)N);
    if (!w) {
#pragma omp atomic write
      status = -2;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t t = 0; t < nrows; ++t) {
        int64_t r = rows[t];
        int rc = attn_row(q, k, v, dtype, r / M, kv_head(r / M, H, Hkv), r % M, M, N, D, scale,
                          causal, o + t * D, lse + t, w);
        if (rc) {
#pragma omp atomic write
          status = rc;
        }
      }
      free(w);
    }
  }
  return status;
}

/* The tiled online-softmax recurrence in fp64, query tiles of BM rows outer,
 * key tiles of BN rows inner.  Per query row the state is (m, l, O~):
 *   m_new = max(m, max_j s_j);  alpha = exp(m - m_new);  p_j = exp(s_j - m_new)
 *   l = alpha l + sum_j p_j;    O~ = alpha O~ + sum_j p_j v_j;   m = m_new
 * with masked keys (j >= N, or j > i when causal) excluded, and at the end
 * O = O~ / l, L = m + ln l.  With m = -inf before the first key the factor
 * alpha = exp(-inf) is 0, so the first tile needs no special case. */
int oracle_attn_fwd_tiled(const void* q, const void* k, const void* v, double* o, double* lse,
                          int B, int H, int M, int N, int D, double scale, int causal,
                          int dtype, int BM, int BN) {
  if (check_sizes(B, H, H, M, N, D, dtype) || BM <= 0 || BN <= 0) return -1;
  const int64_t n_qtiles = (M + BM - 1) / BM;
  const int64_t units = (int64_t)B * H * n_qtiles;
  int status = 0;
#pragma omp parallel
  {
    double* m_run = (double*)malloc(sizeof(double) * (size_t)BM);
    double* l_run = (double*)malloc(sizeof(double) * (size_t)BM);
    double* acc = (double*)malloc(sizeof(double) * (size_t)BM * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)BM * BN);
    if (!m_run || !l_run || !acc || !s) {
#pragma omp atomic write
      status = -2;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t u = 0; u < units; ++u) {
        const int64_t bh = u / n_qtiles, qt = u % n_qtiles;
        const int64_t i0 = qt * BM;
        const int rows = (int)((i0 + BM <= M) ? BM : (M - i0));
        const int64_t kvoff = bh * (int64_t)N * D;
        for (int r = 0; r < rows; ++r) {
          m_run[r] = -INFINITY;
          l_run[r] = 0.0;
          for (int d = 0; d < D; ++d) acc[(int64_t)r * D + d] = 0.0;
        }
        for (int64_t j0 = 0; j0 < N; j0 += BN) {
          const int cols = (int)((j0 + BN <= N) ? BN : (N - j0));
          for (int r = 0; r < rows; ++r) {
            const int64_t i = i0 + r;
            const int64_t qoff = (bh * M + i) * (int64_t)D;
            double tile_max = -INFINITY;
            for (int c = 0; c < cols; ++c) {
              const int64_t j = j0 + c;
              if (causal && j > i) {
                s[(int64_t)r * BN + c] = -INFINITY;
                continue;
              }
              double dot = 0.0;
              for (int d = 0; d < D; ++d)
                dot += widen(q, qoff + d, dtype) * widen(k, kvoff + j * D + d, dtype);
              s[(int64_t)r * BN + c] = scale * dot;
              if (s[(int64_t)r * BN + c] > tile_max) tile_max = s[(int64_t)r * BN + c];
            }
            const double m_new = (tile_max > m_run[r]) ? tile_max : m_run[r];
            if (m_new == -INFINITY) continue; /* no visible key yet: state unchanged */
            const double alpha = exp(m_run[r] - m_new);
            double rowsum = 0.0;
            for (int c = 0; c < cols; ++c) {
              double p = exp(s[(int64_t)r * BN + c] - m_new);
              s[(int64_t)r * BN + c] = p;
              rowsum += p;
            }
            l_run[r] = alpha * l_run[r] + rowsum;
            for (int d = 0; d < D; ++d) {
              double pv = 0.0;
              for (int c = 0; c < cols; ++c)
                pv += s[(int64_t)r * BN + c] * widen(v, kvoff + (j0 + c) * D + d, dtype);
              acc[(int64_t)r * D + d] = alpha * acc[(int64_t)r * D + d] + pv;
            }
            m_run[r] = m_new;
          }
        }
        for (int r = 0; r < rows; ++r) {
          const int64_t row = bh * M + i0 + r;
          if (l_run[r] <= 0.0) {
#pragma omp atomic write
            status = -3;
            continue;
          }
          for (int d = 0; d < D; ++d) o[row * D + d] = acc[(int64_t)r * D + d] / l_run[r];
          lse[row] = m_run[r] + log(l_run[r]);
        }
      }
    }
    free(m_run);
    free(l_run);
    free(acc);
    free(s);
  }
  return status;
}

/* ---------------------------------------------------------------------------
 * Score modifiers: sliding window, softcap and ALiBi.  The pages name these
 * options of the forward ("From FlashAttention to FlashAttention 2", Layer 1:
 * Python API: window_size, softcap, alibi_slopes) and describe the window as a
 * change of the causal mask formula and ALiBi as a bias added to the score
 * ("Writing FlashAttention 2 in Triton", What to do after your FA2 works, items
 * 3 and 4) without printing formulas.  The reading used, for query row i of
 * head (b, h) and key j:
 *   s_j = scale * q_i . k_j
 *   softcap c > 0:   s_j <- c * tanh(s_j / c)
 *   ALiBi slope a:   s_j <- s_j - a * |i - j|       (a = slopes[b*sb + h])
 *   visible:  0 <= j < N;  j <= i when causal;  j >= i - wl when wl >= 0;
 *             j <= i + wr when wr >= 0            (wl, wr < 0: unbounded)
 * then the plain softmax over the visible keys.  A window can leave a row with
 * no visible key ("Writing FlashAttention 2 in Triton", bug catalogue item 8);
 * such a row gets O = 0 and L = -inf. */
static int attn_row_mod(const void* q, const void* k, const void* v, int dtype, int64_t bh,
                        int64_t kvh, int64_t i, int H, int M, int N, int D, double scale,
                        int causal, int wl, int wr, double softcap, const double* slopes,
                        int64_t slope_bstride, double* o_row, double* lse, double* w) {
  const int64_t kvoff = kvh * (int64_t)N * D;
  const int64_t qoff = (bh * M + i) * (int64_t)D;
  int64_t lo = 0, hi = (int64_t)N - 1; /* visible keys: lo <= j <= hi */
  if (causal && i < hi) hi = i;
  if (wr >= 0 && i + wr < hi) hi = i + wr;
  if (wl >= 0 && i - wl > lo) lo = i - wl;
  if (lo > hi) {
    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    *lse = -INFINITY;
    return 0;
  }
  const double slope = slopes ? slopes[(bh / H) * slope_bstride + bh % H] : 0.0;

  double m = -INFINITY;
  for (int64_t j = lo; j <= hi; ++j) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += widen(q, qoff + d, dtype) * widen(k, kvoff + j * D + d, dtype);
    double s = scale * dot;
    if (softcap > 0.0) s = softcap * tanh(s / softcap);
    s -= slope * fabs((double)(i - j));
    w[j - lo] = s;
    if (s > m) m = s;
  }
  double lsum = 0.0;
  for (int64_t j = lo; j <= hi; ++j) {
    w[j - lo] = exp(w[j - lo] - m);
    lsum += w[j - lo];
  }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int64_t j = lo; j <= hi; ++j) acc += w[j - lo] * widen(v, kvoff + j * D + d, dtype);
    o_row[d] = acc / lsum;
  }
  *lse = m + log(lsum);
  return 0;
}

/* Rows of attention with score modifiers.  rows == NULL: every row, o [B,H,M,D]
 * and lse [B,H,M]; otherwise the nrows listed flat rows (b*H + h)*M + i, o
 * [nrows, D] and lse [nrows].  slopes: NULL (no ALiBi) or fp64 slopes read at
 * b*slope_bstride + h (slope_bstride 0: one slope per head for every batch
 * entry; H: one per (b, h)). */
int oracle_attn_fwd_mod(const void* q, const void* k, const void* v, const int64_t* rows,
                        int64_t nrows, double* o, double* lse, int B, int H, int Hkv, int M,
                        int N, int D, double scale, int causal, int wl, int wr, double softcap,
                        const double* slopes, int64_t slope_bstride, int dtype) {
  if (check_sizes(B, H, Hkv, M, N, D, dtype)) return -1;
  if (!(softcap >= 0.0) || isinf(softcap)) return -1;
  if (slopes && slope_bstride != 0 && slope_bstride != H) return -1;
  const int64_t total = (int64_t)B * H * M;
  if (rows == NULL) nrows = total;
  for (int64_t t = 0; rows && t < nrows; ++t)
    if (rows[t] < 0 || rows[t] >= total) return -1;
  int status = 0;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)N);
    if (!w) {
#pragma omp atomic write
      status = -2;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (int64_t t = 0; t < nrows; ++t) {
        const int64_t r = rows ? rows[t] : t;
        const int64_t bh = r / M;
        int rc = attn_row_mod(q, k, v, dtype, bh, kv_head(bh, H, Hkv), r % M, H, M, N, D, scale,
                              causal, wl, wr, softcap, slopes, slope_bstride, o + t * D, lse + t,
                              w);
        if (rc) {
#pragma omp atomic write
          status = rc;
        }
      }
      free(w);
    }
  }
  return status;
}

/* ---------------------------------------------------------------------------
 * Backward pass: the gradients of the forward above for an upstream gradient
 * dO = dloss/dO ("From FlashAttention to FlashAttention 2", Layer 7: The Backward
 * Kernel; "FlashAttention-2 from PyTorch to Triton", Known gaps item 5: the
 * backward recomputes P = exp(S - L) and uses D = rowsum(dO o O)).  With
 * P_ij = exp(s_ij - L_i) the attention weight of visible key j in row i (0 for a
 * hidden key):
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j,   D_i = dO_i . O_i,   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j,            dK_j = scale sum_i dS_ij q_i
 * (the scale appears because s = scale q.k).  With grouped-query attention the
 * dK and dV of a key/value head sum over the query heads that read it.  O and L
 * are recomputed here in fp64 from q, k, v: this is the exact gradient of the
 * exact function.  dout has the dtype of q; dq [B,H,M,D], dk and dv [B,Hkv,N,D]
 * are fp64. */
int oracle_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* dout, double* dq,
                        double* dk, double* dv, int B, int H, int Hkv, int M, int N, int D,
                        double scale, int causal, int dtype) {
  if (check_sizes(B, H, Hkv, M, N, D, dtype)) return -1;
  const int group = H / Hkv;
  const int64_t kv_heads = (int64_t)B * Hkv;
  const int64_t nd = (int64_t)N * D;
  int status = 0;
  /* key/value heads one after another; the rows of a head's query heads in
   * parallel, each thread summing its dK, dV contributions privately */
  for (int64_t kvh = 0; kvh < kv_heads && status == 0; ++kvh) {
    const int64_t kvoff = kvh * nd;
    for (int64_t e = 0; e < nd; ++e) {
      dk[kvoff + e] = 0.0;
      dv[kvoff + e] = 0.0;
    }
#pragma omp parallel
    {
      double* p = (double*)malloc(sizeof(double) * (size_t)N);
      double* ds = (double*)malloc(sizeof(double) * (size_t)N);
      double* dk_t = (double*)calloc((size_t)nd, sizeof(double));
      double* dv_t = (double*)calloc((size_t)nd, sizeof(double));
      if (!p || !ds || !dk_t || !dv_t) {
#pragma omp atomic write
        status = -2;
      } else {
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < (int64_t)group * M; ++r) {
          const int64_t g = r / M, i = r % M;
          const int64_t bh = (kvh / Hkv) * H + (kvh % Hkv) * group + g;
          const int64_t qoff = (bh * M + i) * (int64_t)D;
          const int64_t nvis = visible_keys(i, N, causal);
          /* scores, logsumexp, weights */
          double m = -INFINITY;
          for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
              dot += widen(q, qoff + d, dtype) * widen(k, kvoff + j * D + d, dtype);
            p[j] = scale * dot;
            if (p[j] > m) m = p[j];
          }
          double l = 0.0;
          for (int64_t j = 0; j < nvis; ++j) l += exp(p[j] - m);
          const double L = m + log(l);
          for (int64_t j = 0; j < nvis; ++j) p[j] = exp(p[j] - L);
          /* D_i = dO_i . O_i with O_i = sum_j P_ij v_j */
          double Di = 0.0;
          for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int64_t j = 0; j < nvis; ++j) acc += p[j] * widen(v, kvoff + j * D + d, dtype);
            Di += widen(dout, qoff + d, dtype) * acc;
          }
          /* dS_ij = P_ij (dO_i . v_j - D_i) */
          for (int64_t j = 0; j < nvis; ++j) {
            double dp = 0.0;
            for (int d = 0; d < D; ++d)
              dp += widen(dout, qoff + d, dtype) * widen(v, kvoff + j * D + d, dtype);
            ds[j] = p[j] * (dp - Di);
          }
          for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int64_t j = 0; j < nvis; ++j) acc += ds[j] * widen(k, kvoff + j * D + d, dtype);
            dq[qoff + d] = scale * acc;
          }
          for (int64_t j = 0; j < nvis; ++j)
            for (int d = 0; d < D; ++d) {
              dk_t[j * D + d] += scale * ds[j] * widen(q, qoff + d, dtype);
              dv_t[j * D + d] += p[j] * widen(dout, qoff + d, dtype);
            }
        }
#pragma omp critical
        for (int64_t e = 0; e < nd; ++e) {
          dk[kvoff + e] += dk_t[e];
          dv[kvoff + e] += dv_t[e];
        }
      }
      free(p);
      free(ds);
      free(dk_t);
      free(dv_t);
    }
  }
  return status;
}

/* Multi-head attention: the Hkv == H case of the entry points above. */
int oracle_attn_fwd(const void* q, const void* k, const void* v, double* o, double* lse,
                    int B, int H, int M, int N, int D, double scale, int causal, int dtype) {
  return oracle_attn_fwd_gqa(q, k, v, o, lse, B, H, H, M, N, D, scale, causal, dtype);
}

int oracle_attn_fwd_rows(const void* q, const void* k, const void* v,
                         const int64_t* rows, int64_t nrows, double* o, double* lse,
                         int B, int H, int M, int N, int D, double scale, int causal,
                         int dtype) {
  return oracle_attn_fwd_gqa_rows(q, k, v, rows, nrows, o, lse, B, H, H, M, N, D, scale,
                                  causal, dtype);
}

/* Threads an OpenMP parallel region of the entry points above runs with (the
 * count the CPU baseline reports; it changes no arithmetic). */
int oracle_omp_threads(void) { return omp_get_max_threads(); }
