/*
 * tree_oracle.c -- plain, slow CPU oracle for the steps around tree verification:
 * greedy tree acceptance and post-verify KV-cache compaction.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file; only the test-suite, the smoke check and the CPU-baseline leg of the benchmark
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages about a native DDTree engine):
 *   [VERIFY] "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA
 *             Attention Kernel", §"The Context: What Led to This Moment": the first custom
 *             kernel was a GPU best-first tree builder replacing a per-request CPU heapq
 *             implementation; the draft tree has a budget of nodes.
 *   [RoPE]   "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA
 *             Inference Engine", §"The Broader Context: A Full Native Engine from
 *             Scratch": the engine wires a greedy
 *             tree-accept kernel into the DDTree decode loop and keeps a KV cache with
 *             post-verify compaction; greedy speculative output must match greedy
 *             autoregressive output token for token.
 *   [GOLDEN] "The Golden Reference: A Pivotal Moment in Building a Native DDTree
 *             Inference Engine", §"Context: The Quest for a Hyper-Optimized Inference
 *             Stack" (the greedy tree-accept kernel is one of the three custom kernels,
 *             checked bit-exact against a reference) and §"Recursive Refinement of the
 *             Decode Loop Design" (root, draft and bonus token positions in the cache).
 *
 * The pages give no formulas for these steps.  The readings taken (each is listed in the
 * design notes):
 *   - tree building: the drafter proposes, for each depth d = 1..L after the root, K
 *     candidate tokens with log-probabilities sorted in descending order (the same for
 *     every path: a block drafter predicts every position at once).  A tree node is a
 *     path of candidate ranks (r_1, ..., r_d); its score is the float32 sum of
 *     lp[1][r_1] + ... + lp[d][r_d] accumulated in depth order.  Best-first search pops the
 *     best candidate from a heap and pushes its K children, until `budget` nodes are taken;
 *     "best" is the larger score, then the smaller depth, then the lexicographically
 *     smaller rank path.  Nodes are numbered in the order they are taken (the root is
 *     node 0), which is topological.
 *   - target token of node i = argmax over the vocabulary of the target model's logits at
 *     node i (the prediction of the token that follows node i); ties go to the smallest
 *     token id.
 *   - acceptance walks down from the root: the next accepted node is a child c of the
 *     current node whose draft token equals the current node's target token; if several
 *     children qualify, the one with the smallest node index.  The walk stops when no
 *     child qualifies.  The bonus token is the target token of the last accepted node.
 *     (With distinct sibling tokens -- a well-formed draft tree -- this is the longest
 *     root path whose every draft token equals its parent's target token.)
 *   - compaction: node i's KV row sits at logical key prefix_len + i; the accepted node at
 *     depth d moves to logical key prefix_len + d (the root stays at prefix_len), so the
 *     accepted tokens follow the prefix contiguously and the new prefix length is
 *     prefix_len + 1 + accept_len.  Its rope key was rotated at position prefix_len +
 *     depth = its new key index, so it is moved unchanged.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared, together with tv_oracle.c.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TRO_OK 0
#define TRO_ERR_INVALID_ARG -1
#define TRO_ERR_INVALID_TREE -2

/*
 * Index of the largest of n float values; ties go to the smallest index.  NaN is never
 * the maximum (a comparison with it is false).
 */
static int64_t tro_argmax(const float* x, int64_t n) {
  int64_t best = 0;
  for (int64_t v = 1; v < n; ++v)
    if (x[v] > x[best]) best = v;
  return best;
}

/*
 * logits : [rows, V] float32, row r at logits + r * row_stride.
 * out    : [rows] int32 out, the argmax of each row (smallest index on ties).
 */
int tro_argmax_rows(const float* logits, int64_t rows, int64_t V, int64_t row_stride,
                    int32_t* out) {
  if (rows < 0 || V < 1 || row_stride < V || (rows > 0 && (!logits || !out)))
    return TRO_ERR_INVALID_ARG;
  int64_t r;
#pragma omp parallel for schedule(static)
  for (r = 0; r < rows; ++r) out[r] = (int32_t)tro_argmax(logits + r * row_stride, V);
  return TRO_OK;
}

/*
 * Greedy acceptance of one draft tree per sequence.
 *
 * parent     : [B, Q] int32, topologically ordered, parent[b*Q] == -1.
 * tokens     : [B, Q] int32, draft token of node i (node 0's entry, the root token, is not
 *              read).
 * target     : [B, Q] int32, target token of node i (argmax of the target's logits there).
 * accept_len : [B] int32 out, accepted draft nodes A (0 <= A <= Q-1).
 * path       : [B, Q] int32 out, path[0] = 0 (the root), path[d] = accepted node at depth
 *              d for d = 1..A, -1 after.
 * new_tokens : [B, Q] int32 out, the tokens this step emits: the accepted draft tokens
 *              (depth 1..A) then the bonus token target[path[A]], -1 after.
 */
int tro_tree_accept(const int32_t* parent, const int32_t* tokens, const int32_t* target,
                    int B, int Q, int32_t* accept_len, int32_t* path, int32_t* new_tokens) {
  if (B < 0 || Q < 1) return TRO_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (int64_t)b * Q;
    if (par[0] != -1) return TRO_ERR_INVALID_TREE;
    for (int i = 1; i < Q; ++i)
      if (par[i] < 0 || par[i] >= i) return TRO_ERR_INVALID_TREE;
  }
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (int64_t)b * Q;
    const int32_t* tok = tokens + (int64_t)b * Q;
    const int32_t* tgt = target + (int64_t)b * Q;
    int32_t* pth = path + (int64_t)b * Q;
    int32_t* emit = new_tokens + (int64_t)b * Q;
    for (int i = 0; i < Q; ++i) pth[i] = emit[i] = -1;
    pth[0] = 0;
    int cur = 0, a = 0;
    for (;;) {
      int next = -1;
      for (int c = 1; c < Q; ++c) {
        if (par[c] == cur && tok[c] == tgt[cur]) {
          next = c; /* the smallest qualifying child */
          break;
        }
      }
      if (next < 0) break;
      ++a;
      pth[a] = next;
      emit[a - 1] = tok[next];
      cur = next;
    }
    emit[a] = tgt[cur]; /* bonus token */
    accept_len[b] = a;
  }
  return TRO_OK;
}

/*
 * Post-verify compaction of the latent KV cache: for every sequence b and every accepted
 * depth d = 1..accept_len[b], the cache row of logical key prefix_len[b] + d receives the
 * row of logical key prefix_len[b] + path[b*Q + d] (c_kv and k_pe both).  Rows are moved
 * in increasing d; since path[d] >= d and the path's nodes increase along it, no row is
 * overwritten before it is read.  new_prefix_len[b] = prefix_len[b] + 1 + accept_len[b].
 *
 * c_kv [rows, ckv_stride] / k_pe [rows, kpe_stride]: float32 cache arrays (bf16 caches are
 * compared through their float32 values), d_latent / d_rope elements per row.
 * Key j of sequence b is row page_table[b][j/page_size]*page_size + j%page_size, or
 * b*kv_stride_b + j when page_table is NULL.
 */
static int64_t tro_row(const int32_t* page_table, int page_size, int max_pages,
                       int64_t kv_stride_b, int b, int64_t j) {
  if (page_table) {
    const int32_t page = page_table[(int64_t)b * max_pages + j / page_size];
    return (int64_t)page * page_size + j % page_size;
  }
  return (int64_t)b * kv_stride_b + j;
}

int tro_compact_kv(float* c_kv, int64_t ckv_stride, float* k_pe, int64_t kpe_stride,
                   int d_latent, int d_rope, const int32_t* page_table, int page_size,
                   int max_pages, int64_t kv_stride_b, const int32_t* prefix_len,
                   const int32_t* path, const int32_t* accept_len, int B, int Q,
                   int32_t* new_prefix_len) {
  if (B < 0 || Q < 1 || d_latent < 0 || d_rope < 0) return TRO_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int64_t P = prefix_len[b];
    const int a = accept_len[b];
    if (a < 0 || a >= Q) return TRO_ERR_INVALID_ARG;
    for (int d = 1; d <= a; ++d) {
      const int node = path[(int64_t)b * Q + d];
      if (node < d || node >= Q) return TRO_ERR_INVALID_ARG;
      const int64_t src = tro_row(page_table, page_size, max_pages, kv_stride_b, b, P + node);
      const int64_t dst = tro_row(page_table, page_size, max_pages, kv_stride_b, b, P + d);
      if (src == dst) continue;
      memcpy(c_kv + dst * ckv_stride, c_kv + src * ckv_stride, sizeof(float) * (size_t)d_latent);
      memcpy(k_pe + dst * kpe_stride, k_pe + src * kpe_stride, sizeof(float) * (size_t)d_rope);
    }
    new_prefix_len[b] = (int32_t)(P + 1 + a);
  }
  return TRO_OK;
}


/* ------------------------------------------------------------------------------------ */
/* Best-first draft-tree construction.                                                  */
/* ------------------------------------------------------------------------------------ */

/* A heap candidate: a node not yet taken. */
typedef struct {
  float score;    /* float32 sum of its log-probabilities */
  int depth;      /* 1..L */
  int rank;       /* candidate rank at its depth */
  int parent;     /* index (in the output) of its parent node */
  int path[16];   /* ranks from depth 1 to depth (lexicographic tie break) */
} tro_cand;

/* 1 if a comes before b: larger score, then smaller depth, then smaller rank path. */
static int tro_before(const tro_cand* a, const tro_cand* b) {
  if (a->score != b->score) return a->score > b->score;
  if (a->depth != b->depth) return a->depth < b->depth;
  for (int i = 0; i < a->depth; ++i)
    if (a->path[i] != b->path[i]) return a->path[i] < b->path[i];
  return 0;
}

static void tro_swap(tro_cand* a, tro_cand* b) {
  tro_cand t = *a;
  *a = *b;
  *b = t;
}

/* binary heap with the best candidate at h[0] */
static void tro_push(tro_cand* h, int* n, const tro_cand* c) {
  int i = (*n)++;
  h[i] = *c;
  while (i > 0 && tro_before(&h[i], &h[(i - 1) / 2])) {
    tro_swap(&h[i], &h[(i - 1) / 2]);
    i = (i - 1) / 2;
  }
}

static tro_cand tro_pop(tro_cand* h, int* n) {
  tro_cand top = h[0];
  h[0] = h[--(*n)];
  int i = 0;
  for (;;) {
    int l = 2 * i + 1, r = l + 1, m = i;
    if (l < *n && tro_before(&h[l], &h[m])) m = l;
    if (r < *n && tro_before(&h[r], &h[m])) m = r;
    if (m == i) break;
    tro_swap(&h[i], &h[m]);
    i = m;
  }
  return top;
}

/*
 * lp     : [B, L, K] float32 log-probabilities, lp[b][d-1][k] for depth d, sorted in
 *          descending order over k.
 * tok    : [B, L, K] int32 candidate tokens.
 * root   : [B] int32 root token (the last accepted token), nullable (then -1).
 * budget : draft nodes to take (the tree has budget + 1 nodes); at most the number of
 *          paths of depth 1..L, and at most 63.
 * parent, tokens, depth : [B, budget+1] int32 out (node 0: -1 / root / 0).
 * score  : [B, budget+1] float32 out, nullable (node 0: 0).
 */
int tro_build_tree(const float* lp, const int32_t* tok, const int32_t* root, int B, int L,
                   int K, int budget, int32_t* parent, int32_t* tokens, int32_t* depth,
                   float* score) {
  if (B < 0 || L < 1 || L > 16 || K < 1 || budget < 0 || budget > 63) return TRO_ERR_INVALID_ARG;
  double paths = 0.0, level = 1.0;
  for (int d = 1; d <= L; ++d) {
    level *= K;
    paths += level;
  }
  if ((double)budget > paths) return TRO_ERR_INVALID_ARG;
  const int Q = budget + 1;
  /* every pop pushes at most K candidates */
  tro_cand* heap = (tro_cand*)malloc(sizeof(tro_cand) * (size_t)(K * (budget + 1) + 1));
  if (!heap) return TRO_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const float* lpb = lp + (int64_t)b * L * K;
    const int32_t* tkb = tok + (int64_t)b * L * K;
    int32_t* par = parent + (int64_t)b * Q;
    int32_t* tks = tokens + (int64_t)b * Q;
    int32_t* dep = depth + (int64_t)b * Q;
    float* sc = score ? score + (int64_t)b * Q : NULL;
    par[0] = -1;
    tks[0] = root ? root[b] : -1;
    dep[0] = 0;
    if (sc) sc[0] = 0.0f;
    int n = 0;
    /* the root is taken: push its children */
    for (int k = 0; k < K; ++k) {
      tro_cand c;
      memset(&c, 0, sizeof(c));
      c.score = 0.0f + lpb[k];
      c.depth = 1;
      c.rank = k;
      c.parent = 0;
      c.path[0] = k;
      tro_push(heap, &n, &c);
    }
    for (int i = 1; i < Q; ++i) {
      if (n == 0) { /* fewer nodes than the budget (cannot happen for a valid budget) */
        free(heap);
        return TRO_ERR_INVALID_ARG;
      }
      const tro_cand w = tro_pop(heap, &n);
      par[i] = w.parent;
      tks[i] = tkb[(int64_t)(w.depth - 1) * K + w.rank];
      dep[i] = w.depth;
      if (sc) sc[i] = w.score;
      if (w.depth < L) {
        for (int k = 0; k < K; ++k) {
          tro_cand c = w;
          c.score = w.score + lpb[(int64_t)w.depth * K + k];
          c.depth = w.depth + 1;
          c.rank = k;
          c.parent = i;
          c.path[w.depth] = k;
          tro_push(heap, &n, &c);
        }
      }
    }
  }
  free(heap);
  return TRO_OK;
}
