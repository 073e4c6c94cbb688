// rope_math.h -- the NeoX rotation arithmetic shared by the RoPE kernels (tv_rope_neox and
// the fused verify prologue), so that both give identical bits.
//
// "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference Engine",
// §"The Float64 Decision": the angle and the trigonometry run in double precision and the
// result is converted to float32 at the end.  cos/sin of an angle are taken in double and
// each split into two floats (hi + lo); x0*c - x1*s is formed from exact fp32 products
// (fma gives each product's rounding error), an exact difference (TwoSum) and the small
// cross terms, leaving an error below 2^-44 of |x0*c| + |x1*s| before the one rounding;
// where the result is under 2^-19 of that sum it is recomputed in double.  Either way the
// float32 value is within one ulp of the float64 formula rounded once.  For bf16 storage a
// plain float32 evaluation is kept whenever it already decides the bf16 rounding (RotOut),
// which stores the same bits with about half the arithmetic.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace tv {
namespace rope {

__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void store_float(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_float(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

constexpr int kMaxHalf = 256;  // d_rope <= 512

// cos and sin of one angle: in double, and each split into float hi + lo
struct CosSin {
  double c, s;
  float ch, cl, sh, sl;
};

__device__ __forceinline__ CosSin make_cossin(double angle) {
  CosSin t;
  sincos(angle, &t.s, &t.c);
  t.ch = __double2float_rn(t.c);
  t.cl = __double2float_rn(__dsub_rn(t.c, (double)t.ch));
  t.sh = __double2float_rn(t.s);
  t.sl = __double2float_rn(__dsub_rn(t.s, (double)t.sh));
  return t;
}

// The double-precision recomputation, kept out of line: inlined, the compiler evaluates it
// unconditionally (predication), which puts five float64-pipe operations on every element.
static __device__ __noinline__ float rot_out_double(float a, float b, double c, double s) {
  return __double2float_rn(__fma_rn((double)a, c, -__dmul_rn((double)b, s)));
}

// float32 rounding of a*C - b*S, where C ~ ch + cl ~ c and S ~ sh + sl ~ s (see above);
// cs points at the double pair {c, s}, read only by the fallback
__device__ __forceinline__ float rot_out_parts(float a, float b, float ch, float cl, float sh,
                                               float sl, const double* cs) {
  const float p = __fmul_rn(a, ch), ep = __fmaf_rn(a, ch, -p);
  const float q = __fmul_rn(b, sh), eq = __fmaf_rn(b, sh, -q);
  const float d = __fsub_rn(p, q);
  const float bb = __fsub_rn(d, p);  // TwoSum(p, -q): p - q = d + ed exactly
  const float ed = __fadd_rn(__fsub_rn(p, __fsub_rn(d, bb)), __fsub_rn(-q, bb));
  const float cross = __fmaf_rn(a, cl, -__fmul_rn(b, sl));
  const float tail = __fadd_rn(__fadd_rn(ed, __fsub_rn(ep, eq)), cross);
  const float y = __fadd_rn(d, tail);
  if (fabsf(y) >= 0x1p-19f * __fadd_rn(fabsf(p), fabsf(q))) return y;
  return rot_out_double(a, b, cs[0], cs[1]);
}

// The same value for storage type T.  float: rot_out_parts.  bfloat16: the stored value
// is the bf16 rounding of the float32 result, and plain float32 arithmetic already decides
// it unless the result lies near a bf16 rounding boundary.  y = fma(a, ch, -(b*sh)) is within
// 3 * 2^-24 (|a| + |b|) of the exact a*c - b*s (cos/sin cut to float: 2^-24 each; two
// roundings), and the float32 rounding of the exact value adds 2^-24 (|a| + |b|) more; so
// when y - m and y + m, m = 2^-21 (|a| + |b|), round to the same bf16 value, that value is the
// bf16 rounding of the correctly rounded float32 result, and y is returned.  Otherwise (about
// one element in 10^4, and near cancellation) the exact path above decides.  Either way the
// stored bits are those of rot_out_parts, at about half the arithmetic.
template <typename T>
struct RotOut {
  __device__ static __forceinline__ float f(float a, float b, float ch, float cl, float sh,
                                            float sl, const double* cs) {
    return rot_out_parts(a, b, ch, cl, sh, sl, cs);
  }
};
template <>
struct RotOut<__nv_bfloat16> {
  __device__ static __forceinline__ float f(float a, float b, float ch, float cl, float sh,
                                            float sl, const double* cs) {
    const float y = __fmaf_rn(a, ch, -__fmul_rn(b, sh));
    const float m = __fmul_rn(0x1p-21f, __fadd_rn(fabsf(a), fabsf(b)));
    const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(y, m));
    const __nv_bfloat16 hi = __float2bfloat16_rn(__fadd_rn(y, m));
    if (__bfloat16_as_ushort(lo) == __bfloat16_as_ushort(hi)) return y;
    return rot_out_parts(a, b, ch, cl, sh, sl, cs);
  }
};

template <typename T>
__device__ __forceinline__ float rot_out(float a, float b, const CosSin& t) {
  return RotOut<T>::f(a, b, t.ch, t.cl, t.sh, t.sl, &t.c);
}

// ---- vector form: four rotate-half pairs at a time -----------------------------------
template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  using type = float4;
  __device__ static void load(const float* p, float* x) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  }
  __device__ static void store(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};
template <>
struct Vec4<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float* x) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(u.x << 16), x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16), x[3] = __uint_as_float(u.y & 0xffff0000u);
  }
  __device__ static void store(__nv_bfloat16* p, const float* x) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

// Pairs (k, k + half) for k in 4kq .. 4kq+3 of one rope vector: loaded early (before the
// node's cos/sin exist), rotated and stored later.
struct Quad {
  float x0[4], x1[4];
};
template <typename T>
__device__ __forceinline__ void load_quad(const T* src, int kq, int half, Quad& q) {
  Vec4<T>::load(src + 4 * kq, q.x0);
  Vec4<T>::load(src + half + 4 * kq, q.x1);
}
// The node's cos/sin in shared memory: csf[e * quads + kq] holds the float parts (hi, lo of
// cos, hi, lo of sin) of frequency 4kq + e -- consecutive quads in consecutive 16-byte slots,
// so a warp's reads are free of bank conflicts -- and csd[k] the doubles {cos, sin} that
// only the rare double fallback reads.
template <typename T>
__device__ __forceinline__ void rotate_store(const Quad& q, T* dst, int kq, int half,
                                             const float4* csf, const double2* csd) {
  const int quads = half / 4;
  float y0[4], y1[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 f = csf[e * quads + kq];
    const double* dp = &csd[4 * kq + e].x;
    y0[e] = RotOut<T>::f(q.x0[e], q.x1[e], f.x, f.y, f.z, f.w, dp);   // x0 cos - x1 sin
    y1[e] = RotOut<T>::f(q.x1[e], -q.x0[e], f.x, f.y, f.z, f.w, dp);  // x1 cos + x0 sin
  }
  Vec4<T>::store(dst + 4 * kq, y0);
  Vec4<T>::store(dst + half + 4 * kq, y1);
}
// inverse frequencies 1 / base^(2k / d_rope), k < d_rope / 2 (computed on the host with the
// C library's pow)
struct InvFreq {
  double v[kMaxHalf];
};

}  // namespace rope
}  // namespace tv
