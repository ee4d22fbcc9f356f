// Rotation of one channel pair rounded to bf16 exactly as the rotation with fp64 cos/sin would
// round (nearest-even), for the 3D RoPE prologue of the bf16 path.
//
// The attention of a bf16 pipeline reads its rotated q and k as bf16 tensors ("Accelerating
// Video Generation Inference with Sequential-Parallel 3D Positional Encoding Using a Global
// Time Index", section 2: the fused projection + RoPE step hands bf16 tensors to attention), so
// the value to produce is RN_bf16(x0 cos - x1 sin) and RN_bf16(x0 sin + x1 cos) of the exact
// rotation. cos and sin come as fp32 tables plus fp32 residual tables (cos = c + c_lo to about
// 48 bits).
//
// Fast path (fp32): y0 = fma(x0, c, -fl(x1 s)), y1 = fma(x0, s, fl(x1 c)). With u = 2^-24 its
// distance to the rotation with fp64 cos/sin is at most u |y| (the fma) + u |x1| (the product)
// + u (|x0| + |x1|) (the fp32 tables) + 2^-52 (|x0| + |x1|), i.e. just over 3 u (|x0| + |x1|),
// below E = 3.25 u (|x0| + |x1|) as computed in fp32.
// Rounding y to bf16 gives the exact result unless a bf16 rounding midpoint lies within E of
// y. Within y's binade the nearest midpoint is the fp32 value with y's upper 16 bits and low
// half 0x8000 (|y - m| is exact: same binade); the midpoints of the neighbouring bf16 intervals
// are at least a quarter bf16 ulp (2^14 fp32 ulps) away, more than E whenever E < 2^-10 |y|.
// So the fast path is kept when |y - m| > E and 2^10 E <= |y| for both outputs; otherwise (about
// one pair in a few thousand) the slow path below recomputes both.
//
// Slow path: the products are split exactly (x c_hi = p + e with e = fma(x, c_hi, -p)), their
// sum is taken with Knuth's two-sum, the small terms (the two product errors, x0 c_lo, x1 s_lo)
// are added in fp32, and the final two-sum gives the result as r + err exactly. Rounding
// r + err to fp32 by round-to-odd (truncate, then set the last bit if inexact) and that to
// bf16 by nearest-even equals the direct nearest-even rounding to bf16 (round-to-odd with at
// least two extra bits is innocuous for a later nearest rounding; fp32 has 16 more than bf16).
// The slow path's own error is about 2^-46 (|x0| + |x1|).
#pragma once
#include <cstdint>

namespace ditango {

// Round-to-odd fp32 value of a (bh + bl) + q (dh + dl), computed with error-free transforms.
static __device__ __noinline__ float rope_dot2_odd(float a, float bh, float bl, float q, float dh,
                                            float dl) {
  const float p1 = __fmul_rn(a, bh);
  const float e1 = __fmaf_rn(a, bh, -p1);
  const float p2 = __fmul_rn(q, dh);
  const float e2 = __fmaf_rn(q, dh, -p2);
  const float s = __fadd_rn(p1, p2);  // two-sum: s + t = p1 + p2 exactly
  const float sb = __fsub_rn(s, p1);
  const float t = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, sb)), __fsub_rn(p2, sb));
  const float tail = __fmaf_rn(a, bl, __fmaf_rn(q, dl, __fadd_rn(__fadd_rn(t, e1), e2)));
  const float r = __fadd_rn(s, tail);  // two-sum: r + err = s + tail exactly
  const float rb = __fsub_rn(r, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(r, rb)), __fsub_rn(tail, rb));
  uint32_t u = __float_as_uint(r);
  if (err != 0.f && (u & 1u) == 0u)  // inexact with an even last bit: step toward err
    u = ((__float_as_uint(err) ^ u) >> 31) ? u - 1u : u + 1u;
  return __uint_as_float(u);
}

// True when the fp32 value y may round to bf16 differently from a value within e of it.
__device__ __forceinline__ bool bf16_rounding_unsure(float y, float e) {
  const float mid = __uint_as_float((__float_as_uint(y) & 0xFFFF0000u) | 0x8000u);
  return fabsf(__fsub_rn(y, mid)) <= e || __fmul_rn(e, 1024.f) > fabsf(y);
}

// Fast path alone: (x0, x1) rotated with the fp32 table values c, s and rounded to bf16
// (nearest-even), packed with y0 in the low half; `sure` is false when a rounding midpoint is
// too close for that rounding to be the exact one (the caller then uses the exact path).
__device__ __forceinline__ uint32_t rope_rotate_bf16x2_fast(float x0, float x1, float c, float s,
                                                            bool& sure) {
  const float2 p = __fmul2_rn(make_float2(x1, x1), make_float2(s, c));
  const float y0 = __fmaf_rn(x0, c, -p.x);
  const float y1 = __fmaf_rn(x0, s, p.y);
  const float e = __fmul_rn(__fadd_rn(fabsf(x0), fabsf(x1)), 0x1.ap-23f);  // 3.25 * 2^-24
  sure = !(bf16_rounding_unsure(y0, e) || bf16_rounding_unsure(y1, e));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y1), "f"(y0));
  return r;
}

// Exact path alone: the rotation with cos = c + c_lo, sin = s + s_lo rounded to bf16.
__device__ __forceinline__ uint32_t rope_rotate_bf16x2_exact(float x0, float x1, float c, float s,
                                                             float c_lo, float s_lo) {
  const float y0 = rope_dot2_odd(x0, c, c_lo, -x1, s, s_lo);
  const float y1 = rope_dot2_odd(x0, s, s_lo, x1, c, c_lo);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y1), "f"(y0));
  return r;
}

// (x0, x1) rotated by the angle whose cosine and sine are c + c_lo and s + s_lo, each output
// rounded to bf16 (nearest-even), packed with y0 in the low half. c_lo and s_lo are read
// through `lo(c_lo, s_lo)` only on the slow path.
template <class LoFn>
__device__ __forceinline__ uint32_t rope_rotate_bf16x2(float x0, float x1, float c, float s,
                                                       LoFn lo) {
  bool sure;
  const uint32_t r = rope_rotate_bf16x2_fast(x0, x1, c, s, sure);
  if (sure) return r;
  float c_lo, s_lo;
  lo(c_lo, s_lo);
  return rope_rotate_bf16x2_exact(x0, x1, c, s, c_lo, s_lo);
}

}  // namespace ditango
