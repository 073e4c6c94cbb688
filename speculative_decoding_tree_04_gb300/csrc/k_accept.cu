// k_accept.cu -- greedy tree acceptance (tv_tree_accept) and post-verify KV compaction
// (tv_compact_kv).
//
// "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference Engine",
// §"The Broader Context: A Full Native Engine from Scratch": the DDTree decode loop wires a
// greedy tree-accept kernel after verification and keeps a KV cache with post-verify
// compaction; greedy speculative output must equal greedy autoregressive output.
// "The Golden Reference: A Pivotal Moment in Building a Native DDTree Inference Engine",
// §"Recursive Refinement of the Decode Loop Design": root, draft and bonus tokens and
// their cache positions.
//
// Acceptance.  The target token of node i is the argmax of the target model's logits at
// node i (smallest token id on ties).  Starting at the root, the walk moves to the child
// (smallest node index among several) whose draft token equals the current node's target
// token, until no child does; the bonus token is the last node's target token.
//
// The work is the argmax: B*Q rows of a vocabulary-sized logit vector (B32 Q33 with a
// 163840-token vocabulary is 692 MB of float32), read once -- an HBM-bound stream.
// argmax_chunks_kernel splits every row into `chunks` contiguous pieces so that the grid
// fills the GPU whatever B*Q is; each CTA streams its piece with 16-byte loads (eight in
// flight per thread; an unaligned head and a ragged tail take scalar loads), keeps a
// per-thread best (value, index) in index order for each of the eight slots, and reduces
// the block to one 64-bit key: high word the value mapped to an order-preserving unsigned
// integer, low word the bitwise complement of the index, so that the largest key is the
// largest value with, among equal values, the smallest index.  accept_kernel (one warp
// per sequence) takes the largest key of each row's chunks, validates the tree and walks
// it with ballots over the children.  It is launched with programmatic stream
// serialisation and waits for the argmax grid only before it reads the keys.
//
// Compaction.  The accepted node at depth d moves from logical key P + path[d] to key
// P + d.  Since path[d] >= d and the path's node indices increase, no source row is the
// destination of a move at a smaller depth; a source may be the destination of a move at
// a larger depth, which is why each CTA (one per sequence) first loads every row it moves
// into shared memory, synchronises, and only then stores them (in batches that fit in
// shared memory, loads of a batch before its stores and batches in increasing depth).
#include <cuda_bf16.h>

#include <algorithm>

#include "sm100_ptx.h"
#include "tv_internal.h"

namespace tv {
namespace {

using namespace ptx;

constexpr int kAmThreads = 256;
constexpr int kUnroll = 8;           // 16-byte loads in flight per thread
constexpr uint32_t kNone = 0xFFFFFFFFu;

// float -> unsigned integer with the same order (-0 is taken as +0, so that equal values
// compare equal as the argmax rule needs)
__device__ __forceinline__ uint32_t ordered(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t pack_key(float v, uint32_t idx) {
  return ((uint64_t)ordered(v) << 32) | (uint64_t)(kNone - idx);
}

__device__ __forceinline__ void take(float v, uint32_t i, float& best, uint32_t& bi) {
  // indices arrive in increasing order per thread: a strictly larger value wins, so the
  // first of equal values stays
  if (v > best || bi == kNone) {
    best = v;
    bi = i;
  }
}

__device__ __forceinline__ void take4(const uint4& w, uint32_t i0, float& best, uint32_t& bi,
                                      const float*) {
  take(__uint_as_float(w.x), i0, best, bi);
  take(__uint_as_float(w.y), i0 + 1, best, bi);
  take(__uint_as_float(w.z), i0 + 2, best, bi);
  take(__uint_as_float(w.w), i0 + 3, best, bi);
}
__device__ __forceinline__ void take4(const uint4& w, uint32_t i0, float& best, uint32_t& bi,
                                      const __nv_bfloat16*) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    take(__uint_as_float(ws[k] << 16), i0 + 2 * k, best, bi);
    take(__uint_as_float(ws[k] & 0xFFFF0000u), i0 + 2 * k + 1, best, bi);
  }
}

__device__ __forceinline__ float load_scalar(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_scalar(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}

// One CTA per (row, chunk): the largest key of logits[row][v0 .. v1).
template <typename T>
__global__ void __launch_bounds__(kAmThreads) argmax_chunks_kernel(
    const T* __restrict__ logits, int64_t V, int64_t stride, int chunks, int64_t chunk,
    uint64_t* __restrict__ keys) {
  griddep_launch_dependents();  // the walk kernel may start its launch now
  constexpr int kPer = 16 / sizeof(T);  // elements per 16-byte vector
  const int64_t row = blockIdx.x / chunks;
  const int c = (int)(blockIdx.x - row * chunks);
  const int64_t v0 = (int64_t)c * chunk;
  const int64_t v1 = min(V, v0 + chunk);
  const T* x = logits + row * stride;
  // one (best, index) pair per unrolled slot: independent compare chains, merged by key
  float best[kUnroll];
  uint32_t bi[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    best[u] = -INFINITY;
    bi[u] = kNone;
  }
  static_assert(kUnroll >= 3, "slots 0-2 take the remainder, tail and head");
  if (v0 < v1) {
    // elements before the first 16-byte boundary (rows need not be aligned), then whole
    // 16-byte vectors, then the ragged tail
    const int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)(x + v0) & 15u)) & 15u) /
                                   (uint32_t)sizeof(T));
    const int64_t a0 = min(v1, v0 + head);
    if (v0 + threadIdx.x < a0) take(load_scalar(x + v0 + threadIdx.x), (uint32_t)(v0 + threadIdx.x),
                                    best[2], bi[2]);
    const int64_t nvec = (v1 - a0) / kPer;
    const uint4* xv = reinterpret_cast<const uint4*>(x + a0);
    int64_t k = threadIdx.x;
    for (; k + (kUnroll - 1) * kAmThreads < nvec; k += kUnroll * kAmThreads) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) w[u] = __ldcs(xv + k + u * kAmThreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        take4(w[u], (uint32_t)(a0 + (k + u * kAmThreads) * kPer), best[u], bi[u], x);
    }
    for (; k < nvec; k += kAmThreads)
      take4(__ldcs(xv + k), (uint32_t)(a0 + k * kPer), best[0], bi[0], x);
    for (int64_t v = a0 + nvec * kPer + threadIdx.x; v < v1; v += kAmThreads)
      take(load_scalar(x + v), (uint32_t)v, best[1], bi[1]);
  }
  uint64_t key = 0ull;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const uint64_t ku = bi[u] == kNone ? 0ull : pack_key(best[u], bi[u]);
    key = ku > key ? ku : key;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t other = __shfl_xor_sync(0xffffffffu, key, o);
    key = other > key ? other : key;
  }
  __shared__ uint64_t part[kAmThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) part[warp] = key;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t m = part[0];
#pragma unroll
    for (int w = 1; w < kAmThreads / 32; ++w) m = part[w] > m ? part[w] : m;
    keys[blockIdx.x] = m;
  }
}

// One warp per sequence: targets from the chunk keys, then the greedy walk.
__global__ void __launch_bounds__(128) accept_kernel(
    const uint64_t* __restrict__ keys, int chunks, const int32_t* __restrict__ parent,
    const int32_t* __restrict__ tokens, int B, int Q, int32_t* __restrict__ target,
    int32_t* __restrict__ accept_len, int32_t* __restrict__ path,
    int32_t* __restrict__ new_tokens, int32_t* status) {
  const int b = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;  // whole warp
  const int32_t* par = parent + (int64_t)b * Q;
  const int32_t* tok = tokens + (int64_t)b * Q;
  // the tree and the draft tokens do not depend on the argmax grid: read them first
  int p[2], t[2];
  bool valid = true;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    p[s] = -2;
    t[s] = 0;
    if (i < Q) {
      p[s] = par[i];
      t[s] = tok[i];
      valid = valid && (i == 0 ? p[s] == -1 : (p[s] >= 0 && p[s] < i));
    }
  }
  const bool ok = __all_sync(0xffffffffu, valid);
  griddep_wait();  // the argmax keys are complete and visible from here on
  int g[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    g[s] = -1;
    if (i < Q) {
      const uint64_t* kr = keys + ((int64_t)b * Q + i) * chunks;
      uint64_t m = 0;
      for (int c = 0; c < chunks; ++c) {
        const uint64_t k = kr[c];
        m = k > m ? k : m;
      }
      g[s] = (int)(kNone - (uint32_t)m);
      if (target) target[(int64_t)b * Q + i] = g[s];
    }
  }
  int32_t* pth = path + (int64_t)b * Q;
  int32_t* emit = new_tokens + (int64_t)b * Q;
  if (!ok) {
    for (int i = lane; i < Q; i += 32) {
      pth[i] = i == 0 ? 0 : -1;
      emit[i] = -1;
    }
    if (lane == 0) {
      accept_len[b] = 0;
      report(status, TV_ERR_INVALID_TREE);
    }
    return;
  }
  int cur = 0, a = 0;
  for (;;) {
    const int tc = __shfl_sync(0xffffffffu, (cur >> 5) ? g[1] : g[0], cur & 31);
    const bool m0 = lane >= 1 && lane < Q && p[0] == cur && t[0] == tc;
    const bool m1 = lane + 32 < Q && p[1] == cur && t[1] == tc;
    const uint32_t b0 = __ballot_sync(0xffffffffu, m0);
    const uint32_t b1 = __ballot_sync(0xffffffffu, m1);
    if (!(b0 | b1)) {
      if (lane == 0) emit[a] = tc;  // bonus token
      break;
    }
    // children have larger indices than their parent, so the walk ends within Q steps
    const int next = b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
    const int tn = __shfl_sync(0xffffffffu, (next >> 5) ? t[1] : t[0], next & 31);
    ++a;
    if (lane == 0) {
      pth[a] = next;
      emit[a - 1] = tn;
    }
    cur = next;
  }
  if (lane == 0) {
    pth[0] = 0;
    accept_len[b] = a;
  }
  for (int i = a + 1 + lane; i < Q; i += 32) pth[i] = -1;
  for (int i = a + 1 + lane; i < Q; i += 32) emit[i] = -1;
}

// One CTA per sequence: move the accepted rows (c_kv and k_pe, as 16-byte words) to
// their compacted keys, through shared memory in batches of `batch` rows.
__global__ void __launch_bounds__(256) compact_kernel(
    uint4* c_kv, int64_t ckv_stride16, uint4* k_pe, int64_t kpe_stride16, int ckv_words,
    int kpe_words, CacheGeom cache, int64_t num_rows, const int32_t* __restrict__ prefix_len,
    const int32_t* __restrict__ path, const int32_t* __restrict__ accept_len, int Q,
    int32_t* __restrict__ new_prefix_len, int batch, int32_t* status) {
  extern __shared__ uint4 buf[];
  __shared__ int64_t src_row[64], dst_row[64];
  __shared__ unsigned char s_move[64];
  __shared__ int s_n;
  const int b = blockIdx.x;
  const int P = prefix_len[b];
  const int a = accept_len[b];
  const int words = ckv_words + kpe_words;
  // every accepted depth d = threadIdx.x + 1 (at most 63) checks its move in parallel
  const bool ok_seq = !(P < 0 || a < 0 || a >= Q);
  const int d = threadIdx.x + 1;
  bool bad = threadIdx.x == 0 && !ok_seq;
  if (threadIdx.x < 64) s_move[threadIdx.x] = 0;
  if (ok_seq && d <= a) {
    const int node = path[(int64_t)b * Q + d];
    const int64_t js = (int64_t)P + node, jd = (int64_t)P + d;
    if (node < d || node >= Q ||
        (cache.page_table ? js / cache.page_size >= cache.max_pages : js >= cache.kv_stride_b)) {
      bad = true;
    } else {
      const int64_t rs = cache_row(cache, b, js), rd = cache_row(cache, b, jd);
      bad = rs < 0 || rd < 0 || rs >= num_rows || rd >= num_rows;
      src_row[threadIdx.x] = rs;
      dst_row[threadIdx.x] = rd;
      s_move[threadIdx.x] = !bad && rs != rd;
    }
  }
  const bool any_bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    if (any_bad) report(status, TV_ERR_BOUNDS);
    new_prefix_len[b] = any_bad ? P : P + 1 + a;
    // the rows that move, in depth order
    int n = 0;
    for (int e = 0; !any_bad && e < a; ++e)
      if (s_move[e]) {
        src_row[n] = src_row[e];
        dst_row[n] = dst_row[e];
        ++n;
      }
    s_n = n;
  }
  __syncthreads();
  const int n = s_n;
  for (int r0 = 0; r0 < n; r0 += batch) {
    const int nr = min(batch, n - r0);
    for (int idx = threadIdx.x; idx < nr * words; idx += blockDim.x) {
      const int r = idx / words, w = idx - r * words;
      const int64_t row = src_row[r0 + r];
      buf[idx] = w < ckv_words ? c_kv[row * ckv_stride16 + w]
                               : k_pe[row * kpe_stride16 + (w - ckv_words)];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nr * words; idx += blockDim.x) {
      const int r = idx / words, w = idx - r * words;
      const int64_t row = dst_row[r0 + r];
      if (w < ckv_words)
        c_kv[row * ckv_stride16 + w] = buf[idx];
      else
        k_pe[row * kpe_stride16 + (w - ckv_words)] = buf[idx];
    }
    __syncthreads();
  }
}

}  // namespace

AcceptPlan accept_plan(int B, int Q, int64_t V, int sm_count) {
  AcceptPlan p{};
  const int64_t rows = (int64_t)B * Q;
  // about four CTAs per SM in one wave, chunks of whole 2048-element pieces
  const int64_t want = 4 * (int64_t)sm_count;
  int64_t chunks = rows >= want ? 1 : (want + rows - 1) / std::max<int64_t>(rows, 1);
  int64_t chunk = (V + chunks - 1) / chunks;
  chunk = (chunk + 2047) / 2048 * 2048;
  chunks = (V + chunk - 1) / chunk;
  p.chunks = (int)std::max<int64_t>(1, chunks);
  p.chunk = chunk;
  return p;
}

size_t accept_workspace(int B, int Q, const AcceptPlan& p) {
  return ((size_t)B * Q * p.chunks * sizeof(uint64_t) + 255) / 256 * 256;
}

cudaError_t launch_accept(const void* logits, tv_dtype dt, int64_t V, int64_t stride,
                          const int32_t* parent, const int32_t* tokens, int B, int Q,
                          int32_t* target, int32_t* accept_len, int32_t* path,
                          int32_t* new_tokens, int32_t* status, const AcceptPlan& p,
                          void* ws, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  uint64_t* keys = (uint64_t*)ws;
  const int64_t blocks = (int64_t)B * Q * p.chunks;
  if (dt == TV_BF16)
    argmax_chunks_kernel<__nv_bfloat16><<<(unsigned)blocks, kAmThreads, 0, st>>>(
        (const __nv_bfloat16*)logits, V, stride, p.chunks, p.chunk, keys);
  else
    argmax_chunks_kernel<float><<<(unsigned)blocks, kAmThreads, 0, st>>>(
        (const float*)logits, V, stride, p.chunks, p.chunk, keys);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((B + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_kernel, (const uint64_t*)keys, p.chunks, parent, tokens,
                            B, Q, target, accept_len, path, new_tokens, status);
}

cudaError_t launch_compact(void* c_kv, int64_t ckv_stride_bytes, void* k_pe,
                           int64_t kpe_stride_bytes, int ckv_row_bytes, int kpe_row_bytes,
                           const CacheGeom& g, int64_t num_rows, const int32_t* prefix_len,
                           const int32_t* path, const int32_t* accept_len, int B, int Q,
                           int32_t* new_prefix_len, int32_t* status, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const int words = (ckv_row_bytes + kpe_row_bytes) / 16;
  // as many rows per batch as fit in 96 KB of shared memory (all Q - 1 when they do)
  int batch = std::max(1, std::min(Q - 1, (96 * 1024) / std::max(words * 16, 16)));
  const size_t smem = (size_t)batch * words * 16;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  compact_kernel<<<(unsigned)B, 256, smem, st>>>(
      (uint4*)c_kv, ckv_stride_bytes / 16, (uint4*)k_pe, kpe_stride_bytes / 16, ckv_row_bytes / 16,
      kpe_row_bytes / 16, g, num_rows, prefix_len, path, accept_len, Q, new_prefix_len, batch,
      status);
  return cudaGetLastError();
}

}  // namespace tv
