// k_rope.cu -- NeoX RoPE with a float64 angle (tv_rope_neox).
//
// "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference
// Engine": §"The Message" (split the input in half, rotate with cos/sin), §"The Float64
// Decision" (angle and trigonometry in double, converted to float32 at the end),
// §"The Thinking Process" (cos/sin computed once and reused).
//
// One block per (sequence, tree node) row and group of heads.  The block computes cos/sin
// of the node's angles for the d_rope/2 frequencies in double (the frequencies themselves
// come from the host, where they are computed with the same libm pow the float64
// reference uses) and keeps them in shared memory; every head of the group (all H query
// heads share the node's position) then reuses them.  When the layout allows 8- or
// 16-byte accesses (d_rope a multiple of 8, strides of four elements, aligned bases), each
// thread loads its rows' pairs four at a time before the angles exist, so that the loads
// and the float64 trigonometry overlap; otherwise an element-wise kernel does the same
// arithmetic.
//
// GB300's float64 pipe retires about two operations per clock per SM, so the rotation is
// not done in double.  Each of cos and sin is split into two floats (hi + lo, 48 bits
// together); x0*c - x1*s is then formed from exact fp32 products (fma gives each product's
// rounding error), an exact difference (TwoSum) and the small cross terms, which leaves an
// error below 2^-44 of |x0*c| + |x1*s| before the one rounding to float32.  Where the
// result is smaller than 2^-19 of that sum (heavy cancellation, where this bound would not
// be below a quarter ulp), the element is recomputed in double.  Either way the float32
// value is within one ulp of the float64 formula rounded once.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>
#include <cmath>

#include "rope_math.h"
#include "tv_internal.h"

namespace tv {
namespace {

using namespace rope;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(128) rope_kernel(const Tin* in, int64_t isr, int64_t ish,
                                                   Tout* out, int64_t osr, int64_t osh,
                                                   CacheGeom cache, int use_cache, int Q,
                                                   int NH, int D, int heads_per_block,
                                                   const int32_t* __restrict__ prefix_len,
                                                   const int32_t* __restrict__ depth,
                                                   const __grid_constant__ InvFreq inv) {
  __shared__ CosSin cs[kMaxHalf];
  const int64_t r = blockIdx.x;  // b*Q + i
  const int b = (int)(r / Q);
  const int i = (int)(r % Q);
  const int dep = depth ? depth[r] : i;  // no depth array: a chain, position P + i
  if (dep < 0) return;  // invalid tree: leave the row alone
  const int P = prefix_len[b];
  const int half = D / 2;
  const double pos = (double)P + (double)dep;
  for (int k = threadIdx.x; k < half; k += blockDim.x) cs[k] = make_cossin(__dmul_rn(pos, inv.v[k]));
  __syncthreads();
  int64_t orow = r;
  if (use_cache) {
    // skip rows whose cache slot lies outside the declared geometry
    const int64_t j = (int64_t)P + i;
    if (P < 0) return;
    if (cache.page_table) {
      if (j / cache.page_size >= cache.max_pages) return;
      if (cache.page_table[(int64_t)b * cache.max_pages + j / cache.page_size] < 0) return;
    } else if (j >= cache.kv_stride_b) {
      return;
    }
    orow = cache_row(cache, b, j);
  }
  const int h0 = (int)blockIdx.y * heads_per_block;
  const int nh = min(heads_per_block, NH - h0);
  const Tin* src = in + r * isr + (int64_t)h0 * ish;
  Tout* dst = out + orow * osr + (int64_t)h0 * osh;
  for (int idx = threadIdx.x; idx < nh * half; idx += blockDim.x) {
    const int h = idx / half;
    const int k = idx - h * half;
    const float x0 = to_float(src[h * ish + k]);
    const float x1 = to_float(src[h * ish + k + half]);
    const CosSin t = cs[k];
    store_float(dst + h * osh + k, rot_out<Tout>(x0, x1, t));         // x0 cos - x1 sin
    store_float(dst + h * osh + k + half, rot_out<Tout>(x1, -x0, t));  // x1 cos + x0 sin
  }
}

// Vector form: four rotate-half pairs per load, loads issued before the angles exist.
constexpr int kVecThreads = 128;
constexpr int kVecQuads = 4;  // quads a thread loads before the angles exist

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kVecThreads) rope_vec_kernel(
    const Tin* in, int64_t isr, int64_t ish, Tout* out, int64_t osr, int64_t osh,
    CacheGeom cache, int use_cache, int Q, int NH, int D, int heads_per_block,
    const int32_t* __restrict__ prefix_len, const int32_t* __restrict__ depth,
    const __grid_constant__ InvFreq inv) {
  __shared__ float4 csf[kMaxHalf];
  __shared__ double2 csd[kMaxHalf];
  const int64_t r = blockIdx.x;  // b*Q + i
  const int b = (int)(r / Q);
  const int i = (int)(r % Q);
  const int half = D / 2, quads = half / 4;
  const int h0 = (int)blockIdx.y * heads_per_block;
  const int nh = min(heads_per_block, NH - h0);
  const int nq = nh * quads;
  const Tin* src = in + r * isr + (int64_t)h0 * ish;
  // ---- loads that wait for nothing: issued first ----
  const int dep = depth ? depth[r] : i;  // no depth array: a chain, position P + i
  const int P = prefix_len[b];
  Quad qv[kVecQuads];
#pragma unroll
  for (int u = 0; u < kVecQuads; ++u) {
    const int idx = threadIdx.x + u * blockDim.x;
    if (idx < nq) {
      const int h = idx / quads;
      load_quad<Tin>(src + (int64_t)h * ish, idx - h * quads, half, qv[u]);
    }
  }
  if (dep < 0) return;  // invalid tree: leave the row alone (the whole block agrees)
  int64_t orow = r;
  if (use_cache) {
    // skip rows whose cache slot lies outside the declared geometry
    const int64_t j = (int64_t)P + i;
    if (P < 0) return;
    if (cache.page_table) {
      if (j / cache.page_size >= cache.max_pages) return;
      if (cache.page_table[(int64_t)b * cache.max_pages + j / cache.page_size] < 0) return;
    } else if (j >= cache.kv_stride_b) {
      return;
    }
    orow = cache_row(cache, b, j);
  }
  Tout* dst = out + orow * osr + (int64_t)h0 * osh;
  // ---- the node's cos/sin, once, in double (conflict-free layout, as in the prologue) ----
  const double pos = (double)P + (double)dep;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const CosSin t = make_cossin(__dmul_rn(pos, inv.v[k]));
    csf[(k & 3) * quads + (k >> 2)] = make_float4(t.ch, t.cl, t.sh, t.sl);
    csd[k] = make_double2(t.c, t.s);
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kVecQuads; ++u) {
    const int idx = threadIdx.x + u * blockDim.x;
    if (idx < nq) {
      const int h = idx / quads;
      rotate_store<Tout>(qv[u], dst + (int64_t)h * osh, idx - h * quads, half, csf, csd);
    }
  }
  for (int idx = threadIdx.x + kVecQuads * blockDim.x; idx < nq; idx += blockDim.x) {
    const int h = idx / quads, kq = idx - h * quads;
    Quad x;
    load_quad<Tin>(src + (int64_t)h * ish, kq, half, x);
    rotate_store<Tout>(x, dst + (int64_t)h * osh, kq, half, csf, csd);
  }
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const void* in, int64_t isr, int64_t ish, void* out, int64_t osr,
                     int64_t osh, const CacheGeom* cache, int B, int Q, int NH, int D,
                     const int32_t* prefix_len, const int32_t* depth, double base,
                     cudaStream_t st) {
  CacheGeom g{};
  if (cache) g = *cache;
  const int64_t rows = (int64_t)B * Q;
  if (rows == 0) return cudaSuccess;
  // the table of the last (base, d_rope) a thread used is kept
  thread_local InvFreq inv{};
  thread_local double inv_base = 0.0;
  thread_local int inv_d = 0;
  if (inv_base != base || inv_d != D) {
    for (int k = 0; k < D / 2; ++k)
      inv.v[k] = 1.0 / std::pow(base, (2.0 * (double)k) / (double)D);
    inv_base = base;
    inv_d = D;
  }
  // few rows: split each row's heads over several blocks, so that about two blocks per SM
  // share the work
  const int64_t want = 2 * (int64_t)current_sm_count();
  int groups = rows >= want ? 1 : (int)std::min<int64_t>(NH, (want + rows - 1) / rows);
  if (groups < 1) groups = 1;
  const int hpb = (NH + groups - 1) / groups;
  groups = (NH + hpb - 1) / hpb;
  const bool vec = D % 8 == 0 && isr % 4 == 0 && ish % 4 == 0 && osr % 4 == 0 &&
                   osh % 4 == 0 && reinterpret_cast<uintptr_t>(in) % (4 * sizeof(Tin)) == 0 &&
                   reinterpret_cast<uintptr_t>(out) % (4 * sizeof(Tout)) == 0;
  if (vec)
    rope_vec_kernel<Tin, Tout><<<dim3((unsigned)rows, (unsigned)groups), kVecThreads, 0, st>>>(
        (const Tin*)in, isr, ish, (Tout*)out, osr, osh, g, cache ? 1 : 0, Q, NH, D, hpb,
        prefix_len, depth, inv);
  else
    rope_kernel<Tin, Tout><<<dim3((unsigned)rows, (unsigned)groups), 128, 0, st>>>(
        (const Tin*)in, isr, ish, (Tout*)out, osr, osh, g, cache ? 1 : 0, Q, NH, D, hpb,
        prefix_len, depth, inv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(const void* in, tv_dtype in_dt, int64_t isr, int64_t ish, void* out,
                        tv_dtype out_dt, int64_t osr, int64_t osh, const CacheGeom* cache,
                        int B, int Q, int NH, int D, const int32_t* prefix_len,
                        const int32_t* depth, double base, cudaStream_t st) {
  using bf = __nv_bfloat16;
  if (in_dt == TV_F32 && out_dt == TV_F32)
    return launch_t<float, float>(in, isr, ish, out, osr, osh, cache, B, Q, NH, D, prefix_len,
                                  depth, base, st);
  if (in_dt == TV_F32 && out_dt == TV_BF16)
    return launch_t<float, bf>(in, isr, ish, out, osr, osh, cache, B, Q, NH, D, prefix_len,
                               depth, base, st);
  if (in_dt == TV_BF16 && out_dt == TV_F32)
    return launch_t<bf, float>(in, isr, ish, out, osr, osh, cache, B, Q, NH, D, prefix_len,
                               depth, base, st);
  return launch_t<bf, bf>(in, isr, ish, out, osr, osh, cache, B, Q, NH, D, prefix_len, depth,
                          base, st);
}

}  // namespace tv
