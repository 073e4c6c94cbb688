// k_tree.cu -- best-first draft-tree construction (tv_build_tree).
//
// "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA Attention
// Kernel", §"The Context: What Led to This Moment": the engine's first custom kernel is a
// GPU best-first tree builder that replaces a per-request CPU heapq implementation and
// grows the draft tree up to a node budget.
//
// The drafter proposes, for each depth d = 1..L after the root, K candidate tokens with
// log-probabilities sorted in descending order.  A node is a path of candidate ranks; its
// score is the float32 sum of its log-probabilities, accumulated in depth order; the tree
// is the root plus the `budget` best nodes, taken best first: larger score, then smaller
// depth, then lexicographically smaller rank path.  Nodes are numbered in the order they
// are taken, which is topological (a node is offered only after its parent was taken).
//
// One warp per sequence.  The candidates' log-probabilities and tokens are staged in
// shared memory.  Instead of a heap of every child of every taken node, the warp keeps a
// frontier of at most budget + 1 candidates (two per lane): taking a node offers only its
// best child and its next sibling.  Since candidates are sorted at every depth, a node's
// next sibling and its children never come before it, so the best of this frontier is
// always the best of the full heap.  Each round is a warp-wide argmax under the total
// order (five butterfly steps over score, depth and the packed rank path, 4 bits per
// depth), after which the owner lane turns the taken slot into its next sibling and the
// node's first child takes the next free slot.
#include "tv_internal.h"

namespace tv {
namespace {

struct Cand {
  float score;   // float32 sum of the path's log-probabilities
  float pscore;  // the parent's score
  int depth;     // 1..L; 255 = empty slot
  int rank;      // candidate rank at its depth
  int parent;    // output index of its parent node
  uint64_t key;  // rank path, 4 bits per depth (first depth most significant)
};

__device__ __forceinline__ bool before(float sa, int da, uint64_t ka, float sb, int db,
                                       uint64_t kb) {
  if (sa != sb) return sa > sb;
  if (da != db) return da < db;
  return ka < kb;
}

__device__ __forceinline__ Cand empty_cand() {
  Cand c;
  c.score = -INFINITY;
  c.pscore = 0.f;
  c.depth = 255;
  c.rank = 0;
  c.parent = 0;
  c.key = ~0ull;
  return c;
}

__global__ void __launch_bounds__(128) build_tree_kernel(
    const float* __restrict__ lp_all, const int32_t* __restrict__ tok_all,
    const int32_t* __restrict__ root, int B, int L, int K, int budget, int32_t* __restrict__ parent,
    int32_t* __restrict__ tokens, int32_t* __restrict__ depth, float* __restrict__ score,
    int32_t* status) {
  extern __shared__ unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= B) return;  // whole warp
  const int LK = L * K;
  float* lp = reinterpret_cast<float*>(smem) + warp * 2 * LK;
  int* tk = reinterpret_cast<int*>(lp + LK);
  bool sorted = true;
  for (int i = lane; i < LK; i += 32) {
    lp[i] = lp_all[(int64_t)b * LK + i];
    tk[i] = tok_all[(int64_t)b * LK + i];
  }
  __syncwarp();
  for (int i = lane; i < LK; i += 32)
    if (i % K != K - 1 && !(lp[i] >= lp[i + 1])) sorted = false;
  if (!__all_sync(0xffffffffu, sorted) && lane == 0) report(status, TV_ERR_INVALID_ARG);

  const int Q = budget + 1;
  int32_t* par = parent + (int64_t)b * Q;
  int32_t* tks = tokens + (int64_t)b * Q;
  if (lane == 0) {
    par[0] = -1;
    tks[0] = root ? root[b] : -1;
    if (depth) depth[(int64_t)b * Q] = 0;
    if (score) score[(int64_t)b * Q] = 0.f;
  }
  // frontier slot f lives in lane f % 32, register slot f / 32
  Cand c[2] = {empty_cand(), empty_cand()};
  if (lane == 0) {
    c[0].score = __fadd_rn(0.f, lp[0]);
    c[0].pscore = 0.f;
    c[0].depth = 1;
    c[0].rank = 0;
    c[0].parent = 0;
    c[0].key = 0;
  }
  int n_front = 1;
  for (int i = 1; i < Q; ++i) {
    // this lane's better slot
    const int s = before(c[1].score, c[1].depth, c[1].key, c[0].score, c[0].depth, c[0].key) ? 1 : 0;
    float bs = c[s].score;
    int bd = c[s].depth;
    uint64_t bk = c[s].key;
    int bf = lane + 32 * s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int od = __shfl_xor_sync(0xffffffffu, bd, o);
      const uint64_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int of = __shfl_xor_sync(0xffffffffu, bf, o);
      if (before(os, od, ok, bs, bd, bk)) {
        bs = os;
        bd = od;
        bk = ok;
        bf = of;
      }
    }
    // every lane now holds the winner's slot index bf; its owner supplies the rest
    const int wl = bf & 31, ws = bf >> 5;
    const int rank = __shfl_sync(0xffffffffu, ws ? c[1].rank : c[0].rank, wl);
    const int wpar = __shfl_sync(0xffffffffu, ws ? c[1].parent : c[0].parent, wl);
    const float wps = __shfl_sync(0xffffffffu, ws ? c[1].pscore : c[0].pscore, wl);
    if (lane == 0) {
      par[i] = wpar;
      tks[i] = tk[(bd - 1) * K + rank];
      if (depth) depth[(int64_t)b * Q + i] = bd;
      if (score) score[(int64_t)b * Q + i] = bs;
    }
    // the taken slot becomes the node's next sibling
    if (lane == wl) {
      Cand& w = c[ws];
      if (rank + 1 < K) {
        w.rank = rank + 1;
        w.key = bk + 1;
        w.score = __fadd_rn(wps, lp[(bd - 1) * K + rank + 1]);
      } else {
        w = empty_cand();
      }
    }
    // the node's best child takes the next free slot
    if (bd < L) {
      const int f = n_front++;
      if (lane == (f & 31)) {
        Cand& n = c[f >> 5];
        n.depth = bd + 1;
        n.rank = 0;
        n.parent = i;
        n.key = bk << 4;
        n.pscore = bs;
        n.score = __fadd_rn(bs, lp[bd * K]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_build_tree(const float* lp, const int32_t* tok, const int32_t* root, int B,
                              int L, int K, int budget, int32_t* parent, int32_t* tokens,
                              int32_t* depth, float* score, int32_t* status, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const int warps = 4;
  const size_t smem = (size_t)warps * 2 * L * K * 4;
  build_tree_kernel<<<(unsigned)((B + warps - 1) / warps), warps * 32, smem, st>>>(
      lp, tok, root, B, L, K, budget, parent, tokens, depth, score, status);
  return cudaGetLastError();
}

}  // namespace tv
