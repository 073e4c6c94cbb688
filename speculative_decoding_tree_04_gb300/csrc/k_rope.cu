// k_rope.cu -- NeoX RoPE with a float64 angle (tv_rope_neox).
//
// "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference
// Engine": §"The Message" (split the input in half, rotate with cos/sin), §"The Float64
// Decision" (angle and trigonometry in double, converted to float32 at the end),
// §"The Thinking Process" (cos/sin computed once and reused).
//
// One block per (sequence, tree node) row.  The block first computes cos/sin of the
// node's angles for the d_rope/2 frequencies in double and keeps them in shared memory;
// every head of that row (all H query heads share the node's position) then reuses them.
// The rotation is done in double with explicit round-to-nearest multiplies and adds (no
// contraction), then rounded once to float32 (and once more to bf16 for bf16 storage).
// GB300's float64 rate is low, so the trigonometry is kept to d_rope/2 calls per row;
// the per-element work is four double multiplies and two adds.
#include <cuda_bf16.h>

#include "tv_internal.h"

namespace tv {
namespace {

template <typename T>
__device__ __forceinline__ double load_as_double(const T* p);
template <>
__device__ __forceinline__ double load_as_double<float>(const float* p) {
  return (double)*p;
}
template <>
__device__ __forceinline__ double load_as_double<__nv_bfloat16>(const __nv_bfloat16* p) {
  return (double)__bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store_from_double(T* p, double v);
template <>
__device__ __forceinline__ void store_from_double<float>(float* p, double v) {
  *p = __double2float_rn(v);
}
template <>
__device__ __forceinline__ void store_from_double<__nv_bfloat16>(__nv_bfloat16* p, double v) {
  *p = __float2bfloat16_rn(__double2float_rn(v));
}

constexpr int kMaxHalf = 256;  // d_rope <= 512

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(128) rope_kernel(const Tin* in, int64_t isr, int64_t ish,
                                                   Tout* out, int64_t osr, int64_t osh,
                                                   CacheGeom cache, int use_cache, int Q,
                                                   int NH, int D,
                                                   const int32_t* __restrict__ prefix_len,
                                                   const int32_t* __restrict__ depth,
                                                   double base) {
  __shared__ double cs[kMaxHalf][2];
  const int64_t r = blockIdx.x;  // b*Q + i
  const int b = (int)(r / Q);
  const int i = (int)(r % Q);
  const int dep = depth[r];
  if (dep < 0) return;  // invalid tree: leave the row alone
  const int P = prefix_len[b];
  const int half = D / 2;
  const double pos = (double)P + (double)dep;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const double inv = 1.0 / pow(base, (2.0 * (double)k) / (double)D);
    double s, c;
    sincos(__dmul_rn(pos, inv), &s, &c);
    cs[k][0] = c;
    cs[k][1] = s;
  }
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
  const Tin* src = in + r * isr;
  Tout* dst = out + orow * osr;
  for (int idx = threadIdx.x; idx < NH * half; idx += blockDim.x) {
    const int h = idx / half;
    const int k = idx - h * half;
    const double x0 = load_as_double(src + h * ish + k);
    const double x1 = load_as_double(src + h * ish + k + half);
    const double c = cs[k][0], s = cs[k][1];
    const double y0 = __dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s));
    const double y1 = __dadd_rn(__dmul_rn(x1, c), __dmul_rn(x0, s));
    store_from_double(dst + h * osh + k, y0);
    store_from_double(dst + h * osh + k + half, y1);
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
  rope_kernel<Tin, Tout><<<(unsigned)rows, 128, 0, st>>>(
      (const Tin*)in, isr, ish, (Tout*)out, osr, osh, g, cache ? 1 : 0, Q, NH, D, prefix_len,
      depth, base);
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
