// k_attn_simt.cu -- CUDA-core path of tv_verify_attn (float32 caches and small shapes).
//
// Method: "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA
// Attention Kernel" (§Context, §"Input Knowledge Required") and "The Golden Reference: A
// Pivotal Moment in Building a Native DDTree Inference Engine" (§"The Absorb Form of
// MLA"): scores in latent space, q_latent.c_kv + q_pe.k_pe, softmax over the visible keys,
// softmax-weighted sum of c_kv rows.  The pages' kernel used one block per (batch, head,
// query) and kept every score in shared memory in three phases; that re-reads the KV rows
// once per head and caps kv_len by shared memory.  This kernel instead:
//   * gives one block to (sequence, tree node, 32-head group, KV split): all heads of a
//     node share both the KV rows and the visibility mask, so each KV tile is staged once
//     in shared memory (cp.async, 16-byte pieces, double-buffered) and used by 32 heads;
//   * uses a single pass with an online softmax (running max and sum per row), so kv_len
//     is unbounded, and splits long KV ranges across blocks (flash-decoding style) with a
//     log-sum-exp combine when one wave of blocks would not fill the GPU;
//   * has each warp own 4 heads: lanes split the 4-element chunks of the (d_latent +
//     d_rope) vector, dot products finish with a reduce-scatter of the 4 partial sums
//     over the warp (6 shuffles for 4 rows), and the latent output stays in registers.
// Arithmetic is float32 (FFMA) with exp2 of log2e-prescaled scores.
#include <cuda_bf16.h>

#include <algorithm>

#include "tv_internal.h"

namespace tv {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTileKeys = 32;
constexpr int kRowsPerWarp = 4;
constexpr int kHeadsPerBlock = kWarps * kRowsPerWarp;  // 32

struct SimtArgs {
  const void* q_latent;
  const void* q_pe;
  const void* c_kv;
  const void* k_pe;
  int64_t ckv_stride, kpe_stride;
  CacheGeom cache;
  const int32_t* prefix_len;
  const uint64_t* anc;
  float* out;
  float* lse;
  float* ws_out;
  float* ws_lse;
  int32_t* status;
  int B, H, Q, DL, DR, max_prefix;
  int splits, chunk, head_blocks;
  int causal;  // TV_MASK_CAUSAL: row i sees keys 0 .. P + i
  float scale_log2;
};

__device__ __forceinline__ float4 load4(const float* p) { return *(const float4*)p; }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *(const uint2*)p;
  float4 r;
  r.x = __uint_as_float(u.x << 16);
  r.y = __uint_as_float(u.x & 0xffff0000u);
  r.z = __uint_as_float(u.y << 16);
  r.w = __uint_as_float(u.y & 0xffff0000u);
  return r;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Stage keys [base, base+32) of sequence b into tile (row-major [32][DL+DR] of T); keys at
// or beyond `end` are zero-filled.  8 threads per key, 16-byte pieces.
template <typename T>
__device__ __forceinline__ void stage_tile(const SimtArgs& a, T* tile, int b, int64_t base,
                                           int64_t end) {
  const int E = a.DL + a.DR;
  const int per_row_l = a.DL * (int)sizeof(T) / 16;
  const int per_row = E * (int)sizeof(T) / 16;
  const int kk = threadIdx.x >> 3;
  const int sub = threadIdx.x & 7;
  const int64_t j = base + kk;
  const bool live = j < end;
  const int64_t row = live ? cache_row(a.cache, b, j) : 0;
  const char* ck = (const char*)a.c_kv + row * a.ckv_stride * (int64_t)sizeof(T);
  const char* kp = (const char*)a.k_pe + row * a.kpe_stride * (int64_t)sizeof(T);
  char* dst = (char*)(tile + (int64_t)kk * E);
  for (int p = sub; p < per_row; p += 8) {
    const char* src = p < per_row_l ? ck + 16 * p : kp + 16 * (p - per_row_l);
    cp_async16(dst + 16 * p, live ? src : (const char*)a.c_kv, live ? 16 : 0);
  }
}

template <typename T, int TMAX, int VMAX>
__global__ void __launch_bounds__(kThreads, 1) attn_simt_kernel(const SimtArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int E = a.DL + a.DR;
  const int E4 = E >> 2, DL4 = a.DL >> 2;
  T* tiles = (T*)smem_raw;  // [2][32][E]
  float* sc = (float*)(smem_raw + 2 * kTileKeys * E * sizeof(T));  // [warps][4][32]
  float4* ps = (float4*)(sc + kWarps * kRowsPerWarp * kTileKeys);   // [warps][32]

  int idx = blockIdx.x;
  const int hb = idx % a.head_blocks;
  idx /= a.head_blocks;
  const int i = idx % a.Q;
  idx /= a.Q;
  const int s = idx % a.splits;
  const int b = idx / a.splits;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows_total = (int64_t)a.B * a.Q * a.H;

  const int P = a.prefix_len[b];
  const int64_t kv_len = (int64_t)P + a.Q;
  bool bad = P < 0 || P > a.max_prefix;
  if (!bad) {
    if (a.cache.page_table)
      bad = kv_len > (int64_t)a.cache.max_pages * a.cache.page_size;
    else
      bad = kv_len > a.cache.kv_stride_b;
  }
  const int64_t k0 = (int64_t)s * a.chunk;
  // causal rows see keys up to their own (P + i); tree rows up to the last tree key
  const int64_t k_end = a.causal ? (int64_t)P + i + 1 : kv_len;
  const int64_t k1 = bad ? k0 : (k0 + a.chunk < k_end ? k0 + a.chunk : k_end);
  const uint64_t anc = a.causal ? 0ull : a.anc[(int64_t)b * a.Q + i];
  // every key below pvis is visible (the prefix; for causal rows all keys up to P + i)
  const int64_t pvis = a.causal ? k_end : (int64_t)P;
  if (bad && threadIdx.x == 0 && s == 0 && hb == 0 && i == 0) report(a.status, TV_ERR_BOUNDS);

  // Query rows of this warp in registers: chunk c = lane + 32 t covers elements 4c..4c+3
  // of [q_latent | q_pe].
  float4 q[kRowsPerWarp][TMAX];
  int hrow[kRowsPerWarp];
#pragma unroll
  for (int g = 0; g < kRowsPerWarp; ++g) {
    const int h = hb * kHeadsPerBlock + warp * kRowsPerWarp + g;
    hrow[g] = h;
    const int64_t qrow = ((int64_t)b * a.Q + i) * a.H + h;
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      const int c = lane + 32 * t;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (h < a.H && c < E4) {
        if (c < DL4)
          v = load4((const T*)a.q_latent + qrow * a.DL + 4 * c);
        else
          v = load4((const T*)a.q_pe + qrow * a.DR + 4 * (c - DL4));
      }
      q[g][t] = v;
    }
  }
  const bool warp_live = hb * kHeadsPerBlock + warp * kRowsPerWarp < a.H;

  float m[kRowsPerWarp], l[kRowsPerWarp];
  float4 o[kRowsPerWarp][VMAX];
#pragma unroll
  for (int g = 0; g < kRowsPerWarp; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int v = 0; v < VMAX; ++v) o[g][v] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const int ntiles = k1 > k0 ? (int)((k1 - k0 + kTileKeys - 1) / kTileKeys) : 0;
  if (ntiles > 0) {
    stage_tile<T>(a, tiles, b, k0, k1);
    cp_async_commit();
  }
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles) stage_tile<T>(a, tiles + (buf ^ 1) * kTileKeys * E, b,
                                      k0 + (int64_t)(t + 1) * kTileKeys, k1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const T* tile = tiles + buf * kTileKeys * E;
    const int64_t base = k0 + (int64_t)t * kTileKeys;
    const int64_t j = base + lane;
    const bool vis = j < k1 && (j < pvis || (!a.causal && ((anc >> (int)(j - P)) & 1ull)));
    const unsigned vm = __ballot_sync(0xffffffffu, vis);
    if (warp_live && vm) {
      // ---- scores of the visible keys (log2 domain) ----
      unsigned mm = vm;
      while (mm) {
        const int kk = __ffs(mm) - 1;
        mm &= mm - 1;
        const T* krow = tile + kk * E;
        float part[kRowsPerWarp] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int tt = 0; tt < TMAX; ++tt) {
          const int c = lane + 32 * tt;
          if (c < E4) {
            const float4 kv = load4(krow + 4 * c);
#pragma unroll
            for (int g = 0; g < kRowsPerWarp; ++g)
              part[g] = fmaf(q[g][tt].x, kv.x, fmaf(q[g][tt].y, kv.y,
                        fmaf(q[g][tt].z, kv.z, fmaf(q[g][tt].w, kv.w, part[g]))));
          }
        }
        const bool hi = lane & 16;
        float keep0 = hi ? part[2] : part[0];
        float keep1 = hi ? part[3] : part[1];
        keep0 += __shfl_xor_sync(0xffffffffu, hi ? part[0] : part[2], 16);
        keep1 += __shfl_xor_sync(0xffffffffu, hi ? part[1] : part[3], 16);
        const bool b3 = lane & 8;
        float keep = b3 ? keep1 : keep0;
        keep += __shfl_xor_sync(0xffffffffu, b3 ? keep0 : keep1, 8);
        keep += __shfl_xor_sync(0xffffffffu, keep, 4);
        keep += __shfl_xor_sync(0xffffffffu, keep, 2);
        keep += __shfl_xor_sync(0xffffffffu, keep, 1);
        if ((lane & 7) == 0) {
          const int g = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
          sc[(warp * kRowsPerWarp + g) * kTileKeys + kk] = keep * a.scale_log2;
        }
      }
      __syncwarp();
      // ---- online softmax, one key per lane ----
      float pv[kRowsPerWarp];
#pragma unroll
      for (int g = 0; g < kRowsPerWarp; ++g) {
        const float sv = vis ? sc[(warp * kRowsPerWarp + g) * kTileKeys + lane] : -INFINITY;
        const float mnew = fmaxf(m[g], warp_max(sv));
        const float alpha = exp2f(m[g] - mnew);
        const float p = vis ? exp2f(sv - mnew) : 0.f;
        l[g] = l[g] * alpha + warp_sum(p);
        m[g] = mnew;
        pv[g] = p;
#pragma unroll
        for (int v = 0; v < VMAX; ++v) {
          o[g][v].x *= alpha;
          o[g][v].y *= alpha;
          o[g][v].z *= alpha;
          o[g][v].w *= alpha;
        }
      }
      ps[warp * kTileKeys + lane] = make_float4(pv[0], pv[1], pv[2], pv[3]);
      __syncwarp();
      // ---- weighted sum of latent rows ----
      mm = vm;
      while (mm) {
        const int kk = __ffs(mm) - 1;
        mm &= mm - 1;
        const float4 p4 = ps[warp * kTileKeys + kk];
        const T* krow = tile + kk * E;
#pragma unroll
        for (int v = 0; v < VMAX; ++v) {
          const int c = lane + 32 * v;
          if (c < DL4) {
            const float4 x = load4(krow + 4 * c);
            o[0][v].x = fmaf(p4.x, x.x, o[0][v].x); o[0][v].y = fmaf(p4.x, x.y, o[0][v].y);
            o[0][v].z = fmaf(p4.x, x.z, o[0][v].z); o[0][v].w = fmaf(p4.x, x.w, o[0][v].w);
            o[1][v].x = fmaf(p4.y, x.x, o[1][v].x); o[1][v].y = fmaf(p4.y, x.y, o[1][v].y);
            o[1][v].z = fmaf(p4.y, x.z, o[1][v].z); o[1][v].w = fmaf(p4.y, x.w, o[1][v].w);
            o[2][v].x = fmaf(p4.z, x.x, o[2][v].x); o[2][v].y = fmaf(p4.z, x.y, o[2][v].y);
            o[2][v].z = fmaf(p4.z, x.z, o[2][v].z); o[2][v].w = fmaf(p4.z, x.w, o[2][v].w);
            o[3][v].x = fmaf(p4.w, x.x, o[3][v].x); o[3][v].y = fmaf(p4.w, x.y, o[3][v].y);
            o[3][v].z = fmaf(p4.w, x.z, o[3][v].z); o[3][v].w = fmaf(p4.w, x.w, o[3][v].w);
          }
        }
      }
    }
    __syncthreads();  // tile buffer is refilled two iterations later
  }

  // ---- finalise: this split's normalised output and log-sum-exp ----
#pragma unroll
  for (int g = 0; g < kRowsPerWarp; ++g) {
    const int h = hrow[g];
    if (h >= a.H) continue;
    const int64_t row = ((int64_t)b * a.Q + i) * a.H + h;
    const bool any = l[g] > 0.f;
    const float inv = any ? 1.f / l[g] : 0.f;
    const float lse = any ? (m[g] + log2f(l[g])) * 0.69314718055994531f : -INFINITY;
    float* dst = a.splits == 1 ? a.out + row * a.DL
                               : a.ws_out + ((int64_t)s * rows_total + row) * a.DL;
#pragma unroll
    for (int v = 0; v < VMAX; ++v) {
      const int c = lane + 32 * v;
      if (c < DL4) {
        float4 r = o[g][v];
        r.x *= inv; r.y *= inv; r.z *= inv; r.w *= inv;
        *(float4*)(dst + 4 * c) = r;
      }
    }
    if (lane == 0) {
      if (a.splits == 1)
        a.lse[row] = lse;
      else
        a.ws_lse[(int64_t)s * rows_total + row] = lse;
    }
  }
}

// One warp per row.  Lane s < splits forms split s's weight; the weights are then summed
// and applied in split order (the same arithmetic per element as a serial merge), each
// lane merging four float4 columns at a time so that their loads overlap.  More than 32
// splits take a plain serial merge.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws_out,
                                                      const float* __restrict__ ws_lse,
                                                      int splits, int64_t rows, int DL,
                                                      float* __restrict__ out,
                                                      float* __restrict__ lse) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  if (splits > 32) {  // many splits (forced by the caller): plain serial merge
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, ws_lse[(int64_t)s * rows + row]);
    float sum = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float l = ws_lse[(int64_t)s * rows + row];
      sum += (m == -INFINITY) ? 0.f : expf(l - m);
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int d4 = lane; d4 < DL / 4; d4 += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < splits; ++s) {
        const float l = ws_lse[(int64_t)s * rows + row];
        if (l == -INFINITY) continue;
        const float wt = expf(l - m) * inv;
        const float4 v = *(const float4*)(ws_out + ((int64_t)s * rows + row) * DL + 4 * d4);
        acc.x = fmaf(wt, v.x, acc.x);
        acc.y = fmaf(wt, v.y, acc.y);
        acc.z = fmaf(wt, v.z, acc.z);
        acc.w = fmaf(wt, v.w, acc.w);
      }
      *(float4*)(out + row * DL + 4 * d4) = acc;
    }
    if (lane == 0) lse[row] = sum > 0.f ? m + logf(sum) : -INFINITY;
    return;
  }
  const float ls = lane < splits ? ws_lse[(int64_t)lane * rows + row] : -INFINITY;
  float mx = ls;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float e = (lane < splits && mx != -INFINITY) ? expf(ls - mx) : 0.f;
  float wsum = 0.f;
  for (int s = 0; s < splits; ++s) wsum += __shfl_sync(0xffffffffu, e, s);
  const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
  const float w = e * winv;
  const int n4 = DL / 4;
  for (int base = 0; base < n4; base += 128) {
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < splits; ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      const float lss = __shfl_sync(0xffffffffu, ls, s);
      if (lss == -INFINITY) continue;  // uniform over the warp
      const float4* src = (const float4*)(ws_out + ((int64_t)s * rows + row) * DL);
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int d4 = base + lane + 32 * i;
        v[i] = d4 < n4 ? src[d4] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i].x = fmaf(ws, v[i].x, acc[i].x);
        acc[i].y = fmaf(ws, v[i].y, acc[i].y);
        acc[i].z = fmaf(ws, v[i].z, acc[i].z);
        acc[i].w = fmaf(ws, v[i].w, acc[i].w);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d4 = base + lane + 32 * i;
      if (d4 < n4) *(float4*)(out + row * DL + 4 * d4) = acc[i];
    }
  }
  if (lane == 0) lse[row] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

template <typename T, int TMAX, int VMAX>
cudaError_t launch_tv(const SimtArgs& sa, int blocks, size_t smem, cudaStream_t st) {
  auto k = attn_simt_kernel<T, TMAX, VMAX>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, kThreads, smem, st>>>(sa);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const SimtArgs& sa, int tmax, int vmax, int blocks, size_t smem,
                     cudaStream_t st) {
#define TV_CASE(TM, VM) \
  if (tmax == TM && vmax == VM) return launch_tv<T, TM, VM>(sa, blocks, smem, st);
  TV_CASE(1, 1)
  TV_CASE(2, 1) TV_CASE(2, 2)
  TV_CASE(3, 1) TV_CASE(3, 2) TV_CASE(3, 3)
  TV_CASE(4, 1) TV_CASE(4, 2) TV_CASE(4, 3) TV_CASE(4, 4)
  TV_CASE(5, 1) TV_CASE(5, 2) TV_CASE(5, 3) TV_CASE(5, 4) TV_CASE(5, 5)
#undef TV_CASE
  return cudaErrorInvalidValue;
}

size_t smem_bytes(const tv_attn_args* a) {
  const size_t es = a->kv_dt == TV_BF16 ? 2 : 4;
  return 2 * kTileKeys * (size_t)(a->d_latent + a->d_rope) * es +
         kWarps * kRowsPerWarp * kTileKeys * sizeof(float) + kWarps * kTileKeys * 16;
}

}  // namespace

bool simt_supported(const tv_attn_args* a) {
  const int E = a->d_latent + a->d_rope;
  return a->q_dt == a->kv_dt && E <= 5 * 128 && a->d_latent % 8 == 0 && a->d_rope % 8 == 0 &&
         smem_bytes(a) <= 227 * 1024;
}

SimtPlan simt_plan(const tv_attn_args* a, int sm_count) {
  SimtPlan p;
  p.head_blocks = (a->H + kHeadsPerBlock - 1) / kHeadsPerBlock;
  const int64_t kv_max = (int64_t)a->max_prefix_len + a->Q;
  const int64_t base = (int64_t)a->B * a->Q * p.head_blocks;
  int splits = a->num_splits;
  if (splits <= 0) {
    // aim for about two waves of one-block-per-SM launches, keep >= 64 keys per split
    const int64_t want = (2LL * sm_count + base - 1) / std::max<int64_t>(base, 1);
    const int64_t cap = std::max<int64_t>(1, (kv_max + 63) / 64);
    splits = (int)std::max<int64_t>(1, std::min(want, cap));
  }
  int64_t chunk = (kv_max + splits - 1) / splits;
  chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
  if (chunk < kTileKeys) chunk = kTileKeys;
  p.chunk = (int)chunk;
  p.splits = (int)((kv_max + chunk - 1) / chunk);
  if (p.splits < 1) p.splits = 1;
  return p;
}

size_t simt_workspace(const tv_attn_args* a, const SimtPlan& p) {
  if (p.splits <= 1) return 0;
  const size_t rows = (size_t)a->B * a->Q * a->H;
  const size_t out_b = ((size_t)p.splits * rows * a->d_latent * 4 + 255) / 256 * 256;
  const size_t lse_b = ((size_t)p.splits * rows * 4 + 255) / 256 * 256;
  return out_b + lse_b;
}

cudaError_t launch_attn_simt(const tv_attn_args* a, const SimtPlan& p, void* ws,
                             cudaStream_t st) {
  SimtArgs sa;
  sa.q_latent = a->q_latent;
  sa.q_pe = a->q_pe;
  sa.c_kv = a->c_kv;
  sa.k_pe = a->k_pe;
  sa.ckv_stride = a->ckv_row_stride;
  sa.kpe_stride = a->kpe_row_stride;
  sa.cache = CacheGeom{a->cache.page_table, a->cache.page_size, a->cache.max_pages,
                       a->cache.kv_stride_b};
  sa.prefix_len = a->prefix_len;
  sa.anc = a->anc;
  sa.out = a->out;
  sa.lse = a->lse;
  sa.status = a->status;
  sa.B = a->B;
  sa.H = a->H;
  sa.Q = a->Q;
  sa.DL = a->d_latent;
  sa.DR = a->d_rope;
  sa.max_prefix = a->max_prefix_len;
  sa.splits = p.splits;
  sa.chunk = p.chunk;
  sa.head_blocks = p.head_blocks;
  sa.scale_log2 = (float)((double)a->scale * 1.4426950408889634);
  sa.causal = a->mask_mode == TV_MASK_CAUSAL ? 1 : 0;
  const size_t rows = (size_t)a->B * a->Q * a->H;
  sa.ws_out = (float*)ws;
  sa.ws_lse = ws ? (float*)((char*)ws + ((size_t)p.splits * rows * a->d_latent * 4 + 255) /
                                            256 * 256)
                 : nullptr;
  const int E = a->d_latent + a->d_rope;
  const int tmax = (E / 4 + 31) / 32;
  const int vmax = (a->d_latent / 4 + 31) / 32;
  const int64_t blocks = (int64_t)a->B * a->Q * p.head_blocks * p.splits;
  if (blocks == 0) return cudaSuccess;
  const size_t smem = smem_bytes(a);
  cudaError_t e = a->kv_dt == TV_BF16
                      ? dispatch<__nv_bfloat16>(sa, tmax, vmax, (int)blocks, smem, st)
                      : dispatch<float>(sa, tmax, vmax, (int)blocks, smem, st);
  if (e != cudaSuccess || p.splits == 1) return e;
  return launch_combine(sa.ws_out, sa.ws_lse, p.splits, (int64_t)rows, a->d_latent, a->out,
                        a->lse, st);
}

cudaError_t launch_combine(const float* ws_out, const float* ws_lse, int splits, int64_t rows,
                           int DL, float* out, float* lse, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  combine_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(ws_out, ws_lse, splits, rows, DL,
                                                              out, lse);
  return cudaGetLastError();
}

}  // namespace tv
