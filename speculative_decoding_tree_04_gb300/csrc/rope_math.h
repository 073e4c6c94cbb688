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
// float32 value is within one ulp of the float64 formula rounded once.
#pragma once

#include <cuda_bf16.h>

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

__device__ __forceinline__ float rot_out(float a, float b, const CosSin& t) {
  return rot_out_parts(a, b, t.ch, t.cl, t.sh, t.sl, &t.c);
}

// inverse frequencies 1 / base^(2k / d_rope), k < d_rope / 2 (computed on the host with the
// C library's pow)
struct InvFreq {
  double v[kMaxHalf];
};

}  // namespace rope
}  // namespace tv
