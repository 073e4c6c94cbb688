/*
 * tv_oracle.c -- plain, slow, float64 CPU oracle for tree-verify MLA-absorb attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file; only the test-suite, the smoke check and the CPU-baseline leg of the benchmark
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (the three web pages this project is built from):
 *   [RoPE]   "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA
 *             Inference Engine"
 *   [VERIFY] "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA
 *             Attention Kernel"
 *   [GOLDEN] "The Golden Reference: A Pivotal Moment in Building a Native DDTree
 *             Inference Engine"
 *
 * Every function is the plain definition written out, in double precision, with no
 * blocking, fusion or reordering:
 *   tvo_visibility   -- ancestor-or-self visibility of draft-tree nodes, found by walking
 *                       the parent chain of every node ([VERIFY] §Context: the kernel
 *                       applies a visibility mask over the draft tree; [GOLDEN]
 *                       §"Principled Abstraction": M query tokens against the cache with
 *                       an [M, kv_len] mask).
 *   tvo_rope_neox    -- NeoX rotate-half RoPE with angle, trigonometry and rotation in
 *                       float64, one rounding to float32 at the end ([RoPE] §"The
 *                       Message", §"The Float64 Decision", §"What Input Knowledge Is
 *                       Required" item 1).
 *   tvo_verify_attn  -- absorbed-MLA masked softmax attention in latent space
 *                       ([VERIFY] §"Input Knowledge Required": the query is projected
 *                       into the latent space before the dot product; [GOLDEN] §"The
 *                       Absorb Form of MLA"), plus the log-sum-exp of the scores.
 *
 * Readings taken where the pages are silent (each one is listed in the design notes):
 *   - NeoX pairs element k with element k + d_rope/2 ("split the input in half").
 *   - inverse frequency of pair k is 1 / base^(2k/d_rope).
 *   - tree node i has RoPE position prefix_len + depth(i) and cache slot prefix_len + i.
 *   - a node sees every prefix key and its ancestor-or-self tree keys; masked keys are
 *     left out of the max and the sum.
 *   - lse = max + ln(sum of exp(score - max)), natural logarithm.
 *   - bf16 storage is round-to-nearest-even of the float32 value.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (see oracle/__init__.py).
 * -ffp-contract=off keeps every a*b+c as two roundings, as written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TVO_OK 0
#define TVO_ERR_INVALID_ARG -1
#define TVO_ERR_INVALID_TREE -2
#define TVO_ERR_UNSUPPORTED -3

/* ------------------------------------------------------------------------------------ */
/* Visibility.                                                                          */
/* ------------------------------------------------------------------------------------ */

/*
 * parent : [B, Q] int32; parent[b*Q + 0] must be -1 (node 0 is the root of the draft
 *          tree), and for i > 0, 0 <= parent[b*Q + i] < i (nodes come in topological
 *          order).  Any other array is rejected with TVO_ERR_INVALID_TREE.
 * vis    : [B, Q, Q] uint8 out; vis[b][i][k] = 1 iff tree node k is node i or one of
 *          its ancestors.
 * depth  : [B, Q] int32 out; number of parent steps from node i to the root.
 * anc    : [B, Q] uint64 out, nullable; bit k set iff vis[b][i][k].  Only for Q <= 64.
 */
int tvo_visibility(const int32_t* parent, int B, int Q, uint8_t* vis, int32_t* depth,
                   uint64_t* anc) {
  if (B < 0 || Q < 0 || (B > 0 && Q > 0 && (!parent || !vis || !depth)))
    return TVO_ERR_INVALID_ARG;
  if (anc && Q > 64) return TVO_ERR_UNSUPPORTED;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (int64_t)b * Q;
    if (Q > 0 && par[0] != -1) return TVO_ERR_INVALID_TREE;
    for (int i = 1; i < Q; ++i)
      if (par[i] < 0 || par[i] >= i) return TVO_ERR_INVALID_TREE;
  }
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (int64_t)b * Q;
    for (int i = 0; i < Q; ++i) {
      uint8_t* row = vis + ((int64_t)b * Q + i) * Q;
      memset(row, 0, (size_t)Q);
      /* Walk from node i up to the root, marking every node on the way. */
      int k = i, steps = 0;
      for (;;) {
        row[k] = 1;
        if (k == 0) break;
        k = par[k];
        ++steps;
      }
      depth[(int64_t)b * Q + i] = steps;
      if (anc) {
        uint64_t bits = 0;
        for (int t = 0; t < Q; ++t)
          if (row[t]) bits |= ((uint64_t)1) << t;
        anc[(int64_t)b * Q + i] = bits;
      }
    }
  }
  return TVO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Rounding helpers (IEEE round-to-nearest-even).                                       */
/* ------------------------------------------------------------------------------------ */

/* float32 -> nearest bf16 value (ties to even), returned as a float32 holding it. */
static float tvo_round_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) { /* inf or nan: keep, quiet a nan */
    if (u & 0x007fffffu) u |= 0x00400000u;
    u &= 0xffff0000u;
  } else {
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    u &= 0xffff0000u;
  }
  float y;
  memcpy(&y, &u, 4);
  return y;
}

float tvo_bf16_round(float x) { return tvo_round_bf16(x); }

/* ------------------------------------------------------------------------------------ */
/* NeoX RoPE in float64.                                                                */
/* ------------------------------------------------------------------------------------ */

/*
 * x, y      : [B, Q, n_heads, d_rope] float32 (y may equal x).
 * prefix_len: [B]; depth: [B, Q].  Position of (b, i) is prefix_len[b] + depth[b*Q+i].
 * base      : RoPE base (10000 in every workload here).
 * out_bf16  : nonzero -> round the float32 result once more to bf16 (storage in a bf16
 *             cache); the float32 holding that value is written.
 *
 * For each pair k < d_rope/2:  inv = 1/base^(2k/d_rope), a = pos*inv,
 *   y[k]          = x[k]*cos(a) - x[k+d/2]*sin(a)
 *   y[k + d/2]    = x[k+d/2]*cos(a) + x[k]*sin(a)
 * all in double, then one round-to-nearest to float32.
 */
int tvo_rope_neox(const float* x, float* y, int B, int Q, int n_heads, int d_rope,
                  const int32_t* prefix_len, const int32_t* depth, double base,
                  int out_bf16) {
  if (B < 0 || Q < 0 || n_heads < 0 || d_rope <= 0 || (d_rope & 1)) return TVO_ERR_INVALID_ARG;
  const int half = d_rope / 2;
  const int64_t nrow = (int64_t)B * Q;
  int64_t r;
#pragma omp parallel for schedule(static)
  for (r = 0; r < nrow; ++r) {
    const int b = (int)(r / Q);
    const double pos = (double)prefix_len[b] + (double)depth[r];
    for (int h = 0; h < n_heads; ++h) {
      const float* xi = x + (r * n_heads + h) * d_rope;
      float* yo = y + (r * n_heads + h) * d_rope;
      for (int k = 0; k < half; ++k) {
        const double inv = 1.0 / pow(base, (2.0 * (double)k) / (double)d_rope);
        const double a = pos * inv;
        const double c = cos(a), s = sin(a);
        const double x0 = (double)xi[k], x1 = (double)xi[k + half];
        const double y0 = x0 * c - x1 * s;
        const double y1 = x1 * c + x0 * s;
        float f0 = (float)y0, f1 = (float)y1;
        if (out_bf16) {
          f0 = tvo_round_bf16(f0);
          f1 = tvo_round_bf16(f1);
        }
        yo[k] = f0;
        yo[k + half] = f1;
      }
    }
  }
  return TVO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Cache addressing (logical key j of sequence b -> physical row of the cache arrays).  */
/* ------------------------------------------------------------------------------------ */

typedef struct {
  const int32_t* page_table; /* [B, max_pages] or NULL */
  int page_size;
  int max_pages;
  int64_t kv_stride_b; /* rows per sequence when page_table is NULL */
} tvo_cache;

static int64_t tvo_row(const tvo_cache* c, int b, int64_t j) {
  if (c->page_table) {
    const int32_t page = c->page_table[(int64_t)b * c->max_pages + j / c->page_size];
    return (int64_t)page * c->page_size + j % c->page_size;
  }
  return (int64_t)b * c->kv_stride_b + j;
}

/*
 * Write the rotated draft-tree k_pe rows into the cache: row of (b, i) is the cache row
 * of logical key prefix_len[b] + i.  kpe_tree: [B, Q, d_rope] float32 (already rotated).
 */
int tvo_scatter_tree_kpe(const float* kpe_tree, int B, int Q, int d_rope, float* k_pe,
                         int64_t kpe_stride, const int32_t* page_table, int page_size,
                         int max_pages, int64_t kv_stride_b, const int32_t* prefix_len) {
  tvo_cache c = {page_table, page_size, max_pages, kv_stride_b};
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < Q; ++i) {
      const int64_t row = tvo_row(&c, b, (int64_t)prefix_len[b] + i);
      memcpy(k_pe + row * kpe_stride, kpe_tree + ((int64_t)b * Q + i) * d_rope,
             sizeof(float) * (size_t)d_rope);
    }
  return TVO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Tree-verify attention in latent space, float64.                                      */
/* ------------------------------------------------------------------------------------ */

/*
 * For every (b, i, h): the visible key set is
 *     V = { j : j < P_b }  U  { P_b + k : vis[b][i][k] = 1 }
 * and for j in V
 *     s_j = scale * ( sum_d qL[d]*c_kv[j][d] + sum_r qR[r]*k_pe[j][r] ).
 * Then m = max s_j, l = sum exp(s_j - m), out[d] = sum_j exp(s_j - m)/l * c_kv[j][d],
 * lse = m + ln l.  Keys outside V take no part at all.
 *
 * q_latent [B,Q,H,DL], q_pe [B,Q,H,DR] (RoPE already applied), float32 values.
 * c_kv / k_pe: cache arrays with row strides ckv_stride / kpe_stride (elements); key j of
 * sequence b lives in row page_table[b][j/page_size]*page_size + j%page_size, or in row
 * b*kv_stride_b + j when page_table is NULL.
 * rows_b: optional list of n_sel sequence indices to compute (NULL: all B).  Outputs are
 * written only for those sequences; out [B,Q,H,DL] and lse [B,Q,H] are float64.
 * nthreads <= 0: OpenMP default.
 */
int tvo_verify_attn(int B, int H, int Q, int DL, int DR, double scale,
                    const float* q_latent, const float* q_pe, const float* c_kv,
                    int64_t ckv_stride, const float* k_pe, int64_t kpe_stride,
                    const int32_t* page_table, int page_size, int max_pages,
                    int64_t kv_stride_b, const int32_t* prefix_len, const uint8_t* vis,
                    const int32_t* rows_b, int n_sel, double* out, double* lse,
                    int nthreads) {
  if (B < 0 || H < 0 || Q < 0 || DL <= 0 || DR < 0) return TVO_ERR_INVALID_ARG;
  if (page_table && page_size <= 0) return TVO_ERR_INVALID_ARG;
  tvo_cache c = {page_table, page_size, max_pages, kv_stride_b};
  const int nb = rows_b ? n_sel : B;
  const int64_t work = (int64_t)nb * Q * H;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int64_t w;
#pragma omp parallel for schedule(dynamic, 1)
  for (w = 0; w < work; ++w) {
    const int b = rows_b ? rows_b[w / ((int64_t)Q * H)] : (int)(w / ((int64_t)Q * H));
    const int i = (int)((w / H) % Q);
    const int h = (int)(w % H);
    const int64_t P = prefix_len[b];
    const int64_t kv_len = P + Q;
    const int64_t qrow = ((int64_t)b * Q + i) * H + h;
    const float* qL = q_latent + qrow * DL;
    const float* qR = q_pe + qrow * DR;
    const uint8_t* vrow = vis + ((int64_t)b * Q + i) * Q;

    double* s = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
    unsigned char* ok = (unsigned char*)malloc((size_t)(kv_len > 0 ? kv_len : 1));
    double m = -INFINITY;
    for (int64_t j = 0; j < kv_len; ++j) {
      ok[j] = (j < P) ? 1 : vrow[j - P];
      if (!ok[j]) continue;
      const int64_t row = tvo_row(&c, b, j);
      const float* ck = c_kv + row * ckv_stride;
      const float* kr = k_pe + row * kpe_stride;
      double dot = 0.0;
      for (int d = 0; d < DL; ++d) dot += (double)qL[d] * (double)ck[d];
      for (int r = 0; r < DR; ++r) dot += (double)qR[r] * (double)kr[r];
      s[j] = scale * dot;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < kv_len; ++j)
      if (ok[j]) l += exp(s[j] - m);
    double* o = out + qrow * DL;
    for (int d = 0; d < DL; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < kv_len; ++j) {
      if (!ok[j]) continue;
      const double p = exp(s[j] - m) / l;
      const float* ck = c_kv + tvo_row(&c, b, j) * ckv_stride;
      for (int d = 0; d < DL; ++d) o[d] += p * (double)ck[d];
    }
    lse[qrow] = m + log(l);
    free(s);
    free(ok);
  }
  return TVO_OK;
}

/* Threads of later parallel regions (n <= 0: leave as is); for the CPU-baseline timing. */
void tvo_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Number of OpenMP threads a parallel region would use (for the CPU-baseline report). */
int tvo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
