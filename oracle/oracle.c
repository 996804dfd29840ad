/*
 * oracle.c -- plain fp64 CPU reference for decode-step KV page retrieval.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (FreeKV: Boosting KV Cache Retrieval for Efficient LLM
 * Inference, technical summary, section 2.1 "Algorithm side", and the
 * "Key-Value (KV) Cache" wiki page, sections on PagedAttention and GQA):
 *   - the KV cache is paged; each decode step selects, per KV head, the KV
 *     pages it needs and runs attention on the retrieved pages only;
 *   - the pages print no page-score formula.  The score used here is the
 *     per-channel upper bound of q.k over a page built from the page's
 *     per-channel key minimum and maximum:
 *         s_h(p) = sum_c max(q_hc * kmin_pc, q_hc * kmax_pc)
 *     and a KV head's score is the mean over the query heads of its group
 *     (section 2.1 keeps decisions group-consistent by averaging over the
 *     group's heads);
 *   - the k highest-scoring pages are selected, ties to the lower page id;
 *   - attention is ordinary scaled dot-product softmax attention of each
 *     query head over the tokens of its KV head's selected pages.
 *
 * Layouts (row-major, bf16 passed as raw uint16 bit patterns):
 *   k_pool, v_pool : [n_phys][P][H][D]   (token-major pages, all KV heads)
 *   page_table     : [B][N] int32 logical page -> physical page
 *   q              : [B][Hq][D], query head h belongs to KV head h / (Hq/H)
 *   kmin, kmax     : [B][H][N][D] double
 *   scores         : [B][H][N] double
 *   sel            : [B][H][k] int32 logical page ids, ascending
 *   out            : [B][Hq][D] double
 *
 * Everything is computed in double from the exactly widened bf16 inputs, in
 * the order the definitions are written; independent (b, head) units may run
 * on several OpenMP threads, which changes no result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static size_t pool_at(int P, int H, int D, int phys, int t, int g, int c) {
  return (((size_t)phys * P + t) * H + g) * D + c;
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Tokens of logical page p that a sequence of `len` tokens has written:
 * min(P, len - p P), at least 0 (decode-time append fills pages in order;
 * "Key-Value (KV) Cache" wiki page, PagedAttention).  len < 0 means every
 * page is full. */
static int page_tokens(int P, int p, long len) {
  if (len < 0) return P;
  long v = len - (long)p * P;
  return v <= 0 ? 0 : (v >= P ? P : (int)v);
}

/* Per (sequence, KV head, logical page): per-channel min and max of the keys
 * of the page's written tokens (all P when seq_len is NULL; a page with none
 * gets NaN).  Returns the number of out-of-range physical ids. */
int oracle_summaries(int B, int H, int D, int P, int N, int n_phys,
                     const uint16_t *k_pool, const int32_t *page_table,
                     const int32_t *seq_len, double *kmin, double *kmax) {
  int bad = 0;
#pragma omp parallel for collapse(2) reduction(+ : bad) schedule(static)
  for (int b = 0; b < B; b++)
    for (int g = 0; g < H; g++)
      for (int p = 0; p < N; p++) {
        int phys = page_table[(size_t)b * N + p];
        int nt = page_tokens(P, p, seq_len ? seq_len[b] : -1);
        double *mn = kmin + (((size_t)b * H + g) * N + p) * D;
        double *mx = kmax + (((size_t)b * H + g) * N + p) * D;
        if (nt == 0) {
          for (int c = 0; c < D; c++) mn[c] = mx[c] = NAN;
          continue;
        }
        if (phys < 0 || phys >= n_phys) {
          bad++;
          for (int c = 0; c < D; c++) mn[c] = mx[c] = NAN;
          continue;
        }
        for (int c = 0; c < D; c++) {
          double lo = INFINITY, hi = -INFINITY;
          for (int t = 0; t < nt; t++) {
            double v = bf(k_pool[pool_at(P, H, D, phys, t, g, c)]);
            if (v < lo) lo = v;
            if (v > hi) hi = v;
          }
          mn[c] = lo;
          mx[c] = hi;
        }
      }
  return bad;
}

/* KV-head page score: mean over the group's query heads of
 * sum_c max(q_c * kmin_c, q_c * kmax_c). */
void oracle_scores(int B, int Hq, int H, int D, int N, const uint16_t *q,
                   const double *kmin, const double *kmax, double *scores) {
  int G = Hq / H;
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; b++)
    for (int g = 0; g < H; g++)
      for (int p = 0; p < N; p++) {
        const double *mn = kmin + (((size_t)b * H + g) * N + p) * D;
        const double *mx = kmax + (((size_t)b * H + g) * N + p) * D;
        double group_sum = 0.0;
        for (int j = 0; j < G; j++) {
          const uint16_t *qh = q + ((size_t)b * Hq + (size_t)g * G + j) * D;
          double s = 0.0;
          for (int c = 0; c < D; c++) {
            double qc = bf(qh[c]);
            s += fmax(qc * mn[c], qc * mx[c]);
          }
          group_sum += s;
        }
        scores[((size_t)b * H + g) * N + p] = group_sum / G;
      }
}

typedef struct {
  double neg_score;
  int page;
} ranked;

static int by_rank(const void *a, const void *b) {
  const ranked *x = (const ranked *)a, *y = (const ranked *)b;
  if (x->neg_score < y->neg_score) return -1;
  if (x->neg_score > y->neg_score) return 1;
  return (x->page > y->page) - (x->page < y->page);
}

static int by_int(const void *a, const void *b) {
  int x = *(const int *)a, y = *(const int *)b;
  return (x > y) - (x < y);
}

/* The k pages with the largest score; among equal scores the lower page id
 * ranks first.  Output sorted by page id. */
void oracle_topk(int n, const double *s, int k, int32_t *sel) {
  ranked *r = (ranked *)malloc(sizeof(ranked) * (size_t)n);
  for (int p = 0; p < n; p++) {
    r[p].neg_score = -s[p];
    r[p].page = p;
  }
  qsort(r, (size_t)n, sizeof(ranked), by_rank);
  for (int i = 0; i < k; i++) sel[i] = r[i].page;
  qsort(sel, (size_t)k, sizeof(int32_t), by_int);
  free(r);
}

/* Per unit; n_valid (may be NULL) limits unit u to its pages 0 .. n_valid[u]-1.
 * A unit with fewer valid pages than k selects them all and pads with -1. */
void oracle_topk_all(int units, int n, const double *s, int k, const int32_t *n_valid,
                     int32_t *sel) {
#pragma omp parallel for schedule(static)
  for (int u = 0; u < units; u++) {
    int nv = n_valid ? (n_valid[u] < n ? n_valid[u] : n) : n;
    int kk = k < nv ? k : nv;
    int32_t *out = sel + (size_t)u * k;
    if (kk > 0) oracle_topk(nv, s + (size_t)u * n, kk, out);
    for (int i = kk; i < k; i++) out[i] = -1;
  }
}

/* Decode attention of every query head over the written tokens of its KV
 * head's selected logical pages (ascending page, then token order; all P
 * tokens of a page when seq_len is NULL; a -1 entry is no page):
 *   l_t = scale * q . K_t,  w_t = exp(l_t - max l),  o = sum w_t V_t / sum w_t.
 * Returns the number of out-of-range page ids met. */
int oracle_attention(int B, int Hq, int H, int D, int P, int N, int n_phys,
                     const uint16_t *q, const uint16_t *k_pool,
                     const uint16_t *v_pool, const int32_t *page_table,
                     const int32_t *sel, int k, const int32_t *seq_len, double scale,
                     double *out) {
  int G = Hq / H, bad = 0;
  int T = k * P;
#pragma omp parallel for collapse(2) reduction(+ : bad) schedule(static)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < Hq; h++) {
      int g = h / G;
      const uint16_t *qh = q + ((size_t)b * Hq + h) * D;
      const int32_t *pages = sel + ((size_t)b * H + g) * k;
      double *logit = (double *)malloc(sizeof(double) * (size_t)T);
      int *phys_of = (int *)malloc(sizeof(int) * (size_t)k);
      for (int i = 0; i < k; i++) {
        int lp = pages[i];
        if (lp == -1) {
          phys_of[i] = -1;
          continue;
        }
        int phys = (lp >= 0 && lp < N) ? page_table[(size_t)b * N + lp] : -1;
        if (phys < 0 || phys >= n_phys) {
          bad++;
          phys = -1;
        }
        phys_of[i] = phys;
      }
      long len = seq_len ? seq_len[b] : -1;
      double mx = -INFINITY;
      for (int i = 0; i < k; i++)
        for (int t = 0; t < P; t++) {
          double l = -INFINITY;
          if (phys_of[i] >= 0 && t < page_tokens(P, pages[i], len)) {
            double dot = 0.0;
            for (int c = 0; c < D; c++)
              dot += bf(qh[c]) * bf(k_pool[pool_at(P, H, D, phys_of[i], t, g, c)]);
            l = scale * dot;
          }
          logit[i * P + t] = l;
          if (l > mx) mx = l;
        }
      double *o = out + ((size_t)b * Hq + h) * D;
      for (int c = 0; c < D; c++) o[c] = 0.0;
      double wsum = 0.0;
      for (int i = 0; i < k; i++) {
        if (phys_of[i] < 0) continue;
        for (int t = 0; t < page_tokens(P, pages[i], len); t++) {
          double w = exp(logit[i * P + t] - mx);
          wsum += w;
          for (int c = 0; c < D; c++)
            o[c] += w * bf(v_pool[pool_at(P, H, D, phys_of[i], t, g, c)]);
        }
      }
      for (int c = 0; c < D; c++) o[c] = wsum > 0.0 ? o[c] / wsum : 0.0;
      free(logit);
      free(phys_of);
    }
  return bad;
}

/* Group-consistent query similarity of the speculative mode: per KV head, the
 * mean over its group's query heads of cos(q_t,h, q_prev,h).  A zero-norm
 * vector has cosine 0. */
void oracle_group_cosine(int B, int Hq, int H, int D, const uint16_t *q_t,
                         const uint16_t *q_prev, double *cbar) {
  int G = Hq / H;
  for (int b = 0; b < B; b++)
    for (int g = 0; g < H; g++) {
      double acc = 0.0;
      for (int j = 0; j < G; j++) {
        size_t base = ((size_t)b * Hq + (size_t)g * G + j) * D;
        double dot = 0.0, na = 0.0, nb = 0.0;
        for (int c = 0; c < D; c++) {
          double x = bf(q_t[base + c]), y = bf(q_prev[base + c]);
          dot += x * y;
          na += x * x;
          nb += y * y;
        }
        acc += (na > 0.0 && nb > 0.0) ? dot / (sqrt(na) * sqrt(nb)) : 0.0;
      }
      cbar[(size_t)b * H + g] = acc / G;
    }
}
