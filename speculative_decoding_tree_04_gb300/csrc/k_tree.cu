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
// order: one warp reduction over the scores' order-preserving integer codes finds the best
// score, and only when several lanes hold it do five butterfly steps over (score, depth,
// packed rank path, 4 bits per depth) decide; then the owner lane turns the taken slot into
// its next sibling and the node's first child takes the next free slot.
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

// float -> unsigned with the same order (finite values and infinities)
__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= B) return;  // whole warp
  const int LK = L * K;
  const int Q = budget + 1;
  // per warp: log-probs and tokens (LKp words each, LKp even so that rec is 16-byte
  // aligned), then the nodes taken, written out together at the end:
  // {parent, candidate index, depth, score}
  const int LKp = (LK + 1) & ~1;
  float* lp = reinterpret_cast<float*>(smem) + warp * (2 * LKp + 4 * Q);
  int* tk = reinterpret_cast<int*>(lp + LKp);
  int4* rec = reinterpret_cast<int4*>(tk + LKp);
  bool sorted = true;
  for (int i = lane; i < LK; i += 32) {
    lp[i] = lp_all[(int64_t)b * LK + i];
    tk[i] = tok_all[(int64_t)b * LK + i];
  }
  __syncwarp();
  for (int i = lane; i < LK; i += 32)
    if (i % K != K - 1 && !(lp[i] >= lp[i + 1])) sorted = false;
  if (!__all_sync(0xffffffffu, sorted) && lane == 0) report(status, TV_ERR_INVALID_ARG);

  int32_t* par = parent + (int64_t)b * Q;
  int32_t* tks = tokens + (int64_t)b * Q;
  if (lane == 0) {
    par[0] = -1;
    tks[0] = root ? root[b] : -1;
    if (depth) depth[(int64_t)b * Q] = 0;
    if (score) score[(int64_t)b * Q] = 0.f;
  }
  // frontier slot f lives in lane f % 32, register slot f / 32 (c0 or c1: named, so that
  // they stay in registers)
  Cand c0 = empty_cand(), c1 = empty_cand();
  if (lane == 0) {
    c0.score = __fadd_rn(0.f, lp[0]);
    c0.pscore = 0.f;
    c0.depth = 1;
    c0.rank = 0;
    c0.parent = 0;
    c0.key = 0;
  }
  int n_front = 1;
  for (int i = 1; i < Q; ++i) {
    // this lane's better slot
    const bool s1 = before(c1.score, c1.depth, c1.key, c0.score, c0.depth, c0.key);
    float bs = s1 ? c1.score : c0.score;
    int bd = s1 ? c1.depth : c0.depth;
    uint64_t bk = s1 ? c1.key : c0.key;
    int bf = lane + (s1 ? 32 : 0);
    int rank = s1 ? c1.rank : c0.rank;
    int wpar = s1 ? c1.parent : c0.parent;
    float wps = s1 ? c1.pscore : c0.pscore;
    const uint32_t code = ordered(bs);
    const uint32_t top = __reduce_max_sync(0xffffffffu, code);
    const unsigned holders = __ballot_sync(0xffffffffu, code == top);
    if (__popc(holders) == 1) {
      // one lane holds the best score: it is the winner, and all its fields come at once
      const int wl0 = __ffs(holders) - 1;
      bs = __shfl_sync(0xffffffffu, bs, wl0);
      bd = __shfl_sync(0xffffffffu, bd, wl0);
      bk = __shfl_sync(0xffffffffu, bk, wl0);
      bf = __shfl_sync(0xffffffffu, bf, wl0);
      rank = __shfl_sync(0xffffffffu, rank, wl0);
      wpar = __shfl_sync(0xffffffffu, wpar, wl0);
      wps = __shfl_sync(0xffffffffu, wps, wl0);
    } else {
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
      const int wl1 = bf & 31, ws1 = bf >> 5;
      rank = __shfl_sync(0xffffffffu, ws1 ? c1.rank : c0.rank, wl1);
      wpar = __shfl_sync(0xffffffffu, ws1 ? c1.parent : c0.parent, wl1);
      wps = __shfl_sync(0xffffffffu, ws1 ? c1.pscore : c0.pscore, wl1);
    }
    const int wl = bf & 31, ws = bf >> 5;
    if (lane == 0) rec[i] = make_int4(wpar, (bd - 1) * K + rank, bd, __float_as_int(bs));
    // the taken slot becomes the node's next sibling
    if (lane == wl) {
      Cand w = empty_cand();
      if (rank + 1 < K) {
        w = ws ? c1 : c0;
        w.rank = rank + 1;
        w.key = bk + 1;
        w.score = __fadd_rn(wps, lp[(bd - 1) * K + rank + 1]);
      }
      if (ws) c1 = w; else c0 = w;
    }
    // the node's best child takes the next free slot
    if (bd < L) {
      const int f = n_front++;
      if (lane == (f & 31)) {
        Cand n;
        n.depth = bd + 1;
        n.rank = 0;
        n.parent = i;
        n.key = bk << 4;
        n.pscore = bs;
        n.score = __fadd_rn(bs, lp[bd * K]);
        if (f >> 5) c1 = n; else c0 = n;
      }
    }
  }
  __syncwarp();
  for (int i = 1 + lane; i < Q; i += 32) {
    const int4 r = rec[i];
    par[i] = r.x;
    tks[i] = tk[r.y];
    if (depth) depth[(int64_t)b * Q + i] = r.z;
    if (score) score[(int64_t)b * Q + i] = __int_as_float(r.w);
  }
}

}  // namespace

cudaError_t launch_build_tree(const float* lp, const int32_t* tok, const int32_t* root, int B,
                              int L, int K, int budget, int32_t* parent, int32_t* tokens,
                              int32_t* depth, float* score, int32_t* status, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const int warps = 4;
  const size_t smem = (size_t)warps * (2 * (size_t)((L * K + 1) & ~1) + 4 * (size_t)(budget + 1)) * 4;
  build_tree_kernel<<<(unsigned)((B + warps - 1) / warps), warps * 32, smem, st>>>(
      lp, tok, root, B, L, K, budget, parent, tokens, depth, score, status);
  return cudaGetLastError();
}

}  // namespace tv
