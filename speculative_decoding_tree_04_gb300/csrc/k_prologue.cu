// k_prologue.cu -- the steps before verify attention in one launch (tv_verify_prologue):
// draft-tree visibility, NeoX RoPE of the queries' rope part, RoPE of the draft tokens' k_pe
// rows written into their cache slots, and the append of the draft tokens' latent rows.
//
// "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference Engine":
// §"The Thinking Process" (cos/sin are computed once and reused), §"The Float64 Decision"
// (angle and trigonometry in double), §"The Broader Context: A Full Native Engine from
// Scratch" (the engine's KV cache management).  "The Precision Imperative: Validating
// Numerical Accuracy in a Custom CUDA Attention Kernel", §Context (the visibility mask).
//
// Separately these are three launches (visibility, RoPE of the queries, RoPE of the keys)
// plus a copy; each RoPE launch recomputes the node's cos/sin.  Here one CTA serves one
// (tree node, sequence): warp 0 resolves the sequence's tree by pointer jumping (the same
// algorithm as tv_build_visibility: every node starts with {itself} and a jump to its
// parent; six rounds OR in the jumped-to node's set and double the jump) and writes node
// i's ancestor bitset and depth; the CTA then computes the node's d_rope/2 cos/sin pairs
// once, in double, and uses them for all H query heads (four rotate-half pairs per thread
// per pass, 8- or 16-byte loads) and for the draft key row, which goes straight into cache
// slot P + i together with the node's latent row.  The rotation arithmetic is the one of
// tv_rope_neox (rope_math.h), so the results are the same bits.
#include <cuda_bf16.h>

#include <cmath>

#include "rope_math.h"
#include "tv_internal.h"

namespace tv {
namespace {

using namespace rope;

struct ProParams {
  const int32_t* parent;      // [B, Q]
  const int32_t* prefix_len;  // [B]
  int B, Q, H, DR, DL;
  const void* q_in;  // [B, Q, H, DR]
  void* q_out;
  const void* kpe_tree;  // [B, Q, DR]
  const void* ckv_tree;  // [B, Q, DL] or null
  void* c_kv;
  void* k_pe;
  int64_t ckv_stride, kpe_stride;  // elements
  CacheGeom cache;
  int64_t num_rows;  // 0: unknown
  uint64_t* anc;     // [B, Q]
  int32_t* depth;    // [B, Q]
  int32_t* status;
};

constexpr int kThreads = 128;       // small CTAs: one wave of (node, sequence) CTAs
constexpr int kQuadsPerThread = 4;  // query quads a thread loads before the angles exist

template <typename Tq, typename Tkv>
__global__ void __launch_bounds__(kThreads, 7) prologue_kernel(const ProParams p,
                                                       const __grid_constant__ InvFreq inv) {
  __shared__ float4 csf[kMaxHalf];
  __shared__ double2 csd[kMaxHalf];
  __shared__ int s_dep;
  // a programmatic dependent launched after this kernel (the attention call's preparation,
  // which reads none of this kernel's outputs) may start as soon as every CTA is running
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int i = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Q = p.Q;
  // ---- loads that do not wait for the tree or the angles: issued first ----
  const int P = p.prefix_len[b];
  const int half = p.DR / 2;
  const int quads = half / 4;
  const int64_t row = (int64_t)b * Q + i;
  const Tq* qi = static_cast<const Tq*>(p.q_in) + row * p.H * p.DR;
  Tq* qo = static_cast<Tq*>(p.q_out) + row * p.H * p.DR;
  const int nq = p.H * quads;
  Quad qv[kQuadsPerThread];
#pragma unroll
  for (int u = 0; u < kQuadsPerThread; ++u) {
    const int idx = threadIdx.x + u * blockDim.x;
    if (idx < nq) {
      const int h = idx / quads;
      load_quad<Tq>(qi + (int64_t)h * p.DR, idx - h * quads, half, qv[u]);
    }
  }
  // the draft token's cache slot P + i (skipped when outside the geometry)
  int64_t crow = -1;
  if (P >= 0) {
    const int64_t j = (int64_t)P + i;
    bool in = true;
    if (p.cache.page_table)
      in = j / p.cache.page_size < p.cache.max_pages &&
           p.cache.page_table[(int64_t)b * p.cache.max_pages + j / p.cache.page_size] >= 0;
    else
      in = j < p.cache.kv_stride_b;
    if (in) crow = cache_row(p.cache, b, j);
    if (p.num_rows > 0 && crow >= p.num_rows) crow = -1;
  }
  Quad kv;
  if (crow >= 0 && (int)threadIdx.x < quads)
    load_quad<Tkv>(static_cast<const Tkv*>(p.kpe_tree) + row * p.DR, threadIdx.x, half, kv);
  if (warp == 0) {
    // ---- visibility of the whole tree; this CTA publishes node i's entries ----
    const int32_t* par = p.parent + (int64_t)b * Q;
    int pp[2];
    bool valid = true;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int n = lane + 32 * s;
      pp[s] = -1;
      if (n < Q) {
        pp[s] = par[n];
        valid = valid && (n == 0 ? pp[s] == -1 : (pp[s] >= 0 && pp[s] < n));
      }
    }
    const bool ok = __all_sync(0xffffffffu, valid);
    uint64_t A[2];
    int J[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int n = lane + 32 * s;
      A[s] = n < Q ? (1ull << n) : 0ull;
      J[s] = (n < Q && ok) ? pp[s] : -1;
    }
#pragma unroll
    for (int round = 0; round < 6; ++round) {
      uint64_t nA[2];
      int nJ[2];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int src = J[s] < 0 ? lane : J[s];
        const uint64_t a0 = __shfl_sync(0xffffffffu, A[0], src & 31);
        const uint64_t a1 = __shfl_sync(0xffffffffu, A[1], src & 31);
        const int j0 = __shfl_sync(0xffffffffu, J[0], src & 31);
        const int j1 = __shfl_sync(0xffffffffu, J[1], src & 31);
        nA[s] = (src >> 5) ? a1 : a0;
        nJ[s] = (src >> 5) ? j1 : j0;
      }
#pragma unroll
      for (int s = 0; s < 2; ++s)
        if (J[s] >= 0) {
          A[s] |= nA[s];
          J[s] = nJ[s];
        }
    }
    const uint64_t ai0 = __shfl_sync(0xffffffffu, A[0], i & 31);
    const uint64_t ai1 = __shfl_sync(0xffffffffu, A[1], i & 31);
    const uint64_t ai = (i >> 5) ? ai1 : ai0;
    if (lane == 0) {
      const int d = ok ? __popcll(ai) - 1 : -1;
      s_dep = d;
      p.anc[(int64_t)b * Q + i] = ok ? ai : 0ull;
      p.depth[(int64_t)b * Q + i] = d;
      if (!ok && i == 0) report(p.status, TV_ERR_INVALID_TREE);
    }
  }
  __syncthreads();
  const int dep = s_dep;
  if (dep < 0) return;  // invalid tree: this node is left alone, as by tv_rope_neox
  // the latent row needs no rotation: copy it while the angles are computed
  if (crow >= 0 && p.ckv_tree) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const Tkv*>(p.ckv_tree) + row * p.DL);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<Tkv*>(p.c_kv) + crow * p.ckv_stride);
    const int words = p.DL * (int)sizeof(Tkv) / 16;
    for (int w = threadIdx.x; w < words; w += blockDim.x) dst[w] = src[w];
  }
  // ---- the node's cos/sin, once, in double ----
  const double pos = (double)P + (double)dep;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const CosSin t = make_cossin(__dmul_rn(pos, inv.v[k]));
    csf[(k & 3) * quads + (k >> 2)] = make_float4(t.ch, t.cl, t.sh, t.sl);
    csd[k] = make_double2(t.c, t.s);
  }
  __syncthreads();
  // ---- every query head of the node, then the draft key row into its cache slot ----
#pragma unroll
  for (int u = 0; u < kQuadsPerThread; ++u) {
    const int idx = threadIdx.x + u * blockDim.x;
    if (idx < nq) {
      const int h = idx / quads;
      rotate_store<Tq>(qv[u], qo + (int64_t)h * p.DR, idx - h * quads, half, csf, csd);
    }
  }
  // heads beyond what the first pass held (H * d_rope / 8 > 512)
  for (int idx = threadIdx.x + kQuadsPerThread * blockDim.x; idx < nq; idx += blockDim.x) {
    const int h = idx / quads, kq = idx - h * quads;
    Quad x;
    load_quad<Tq>(qi + (int64_t)h * p.DR, kq, half, x);
    rotate_store<Tq>(x, qo + (int64_t)h * p.DR, kq, half, csf, csd);
  }
  if (crow >= 0 && (int)threadIdx.x < quads)
    rotate_store<Tkv>(kv, static_cast<Tkv*>(p.k_pe) + crow * p.kpe_stride, threadIdx.x, half, csf, csd);
}

}  // namespace

cudaError_t launch_prologue(const tv_prologue_args* a, cudaStream_t st) {
  ProParams p{};
  p.parent = a->parent;
  p.prefix_len = a->prefix_len;
  p.B = a->B;
  p.Q = a->Q;
  p.H = a->H;
  p.DR = a->d_rope;
  p.DL = a->d_latent;
  p.q_in = a->q_pe_in;
  p.q_out = a->q_pe_out;
  p.kpe_tree = a->kpe_tree;
  p.ckv_tree = a->ckv_tree;
  p.c_kv = a->c_kv;
  p.k_pe = a->k_pe;
  p.ckv_stride = a->ckv_row_stride;
  p.kpe_stride = a->kpe_row_stride;
  p.cache = CacheGeom{a->cache.page_table, a->cache.page_size, a->cache.max_pages,
                      a->cache.kv_stride_b};
  p.num_rows = a->cache.num_rows;
  p.anc = a->anc;
  p.depth = a->depth;
  p.status = a->status;
  if (a->B == 0) return cudaSuccess;
  // the table of the last (base, d_rope) a thread used is kept
  thread_local InvFreq inv{};
  thread_local double inv_base = 0.0;
  thread_local int inv_d = 0;
  if (inv_base != a->rope_base || inv_d != a->d_rope) {
    for (int k = 0; k < a->d_rope / 2; ++k)
      inv.v[k] = 1.0 / std::pow(a->rope_base, (2.0 * (double)k) / (double)a->d_rope);
    inv_base = a->rope_base;
    inv_d = a->d_rope;
  }
  const dim3 grid((unsigned)a->Q, (unsigned)a->B);
  if (a->q_dt == TV_BF16 && a->kv_dt == TV_BF16)
    prologue_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, kThreads, 0, st>>>(p, inv);
  else if (a->q_dt == TV_BF16)
    prologue_kernel<__nv_bfloat16, float><<<grid, kThreads, 0, st>>>(p, inv);
  else if (a->kv_dt == TV_BF16)
    prologue_kernel<float, __nv_bfloat16><<<grid, kThreads, 0, st>>>(p, inv);
  else
    prologue_kernel<float, float><<<grid, kThreads, 0, st>>>(p, inv);
  return cudaGetLastError();
}

}  // namespace tv
