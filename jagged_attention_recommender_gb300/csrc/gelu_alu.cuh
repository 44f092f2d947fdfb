// gelu_alu.cuh -- tanh-GELU evaluated with FMA-pipe and integer instructions
// only (no special-function-unit instruction).
//
// The GDPA section of the techfeed summary of "GEM Training" replaces the tanh
// inside GELU, a special-function-unit bottleneck, by a 6th-order Taylor
// expansion and notes that QK-norm bounds the inputs, so accuracy holds.  A
// Taylor series of tanh itself diverges long before |s| = 16, so this file
// takes the reading that keeps both statements true:
//
//   gelu(x) = x/2 (1 + tanh u) = x * sigma(2u),   u = sqrt(2/pi) (x + 0.044715 x^3)
//   sigma(z) = 1 / (1 + e^-z)        (and sigma(-a) = e^-a * sigma(a))
//
//   e^-a,  a = |z| clamped to 18:  a = k ln2 + r with integer k = round(a/ln2)
//          and |r| <= ln2/2 (two-part ln2, Cody and Waite), then
//          e^-a = 2^-k * T6(-r),  T6 = the degree-6 Taylor polynomial of exp,
//          with 2^-k built directly in the exponent field;
//   1/(1+e^-a), the divisor d in (1, 2]:  Newton-Raphson on d/2 in (1/2, 1]
//          from the linear seed 48/17 - 32/17 (d/2) (maximum relative error
//          1/17), three steps.
//
// Truncation error of T6 on |r| <= ln2/2 is below 2e-7 relative; the clamp at
// |z| = 18 changes sigma by less than 2e-8.  The whole evaluation is within
// about 1e-6 of the exact tanh-GELU for |x| <= 17 (tested against an fp64
// reference on a dense grid) and saturates to x or 0 beyond.
#pragma once

#include "sm103_ptx.cuh"

namespace gdpa {

__device__ __forceinline__ float gelu_tanh_alu(float x) {
  const float two_c = 1.5957691216057308f;        // 2 * sqrt(2/pi)
  const float two_c3 = 0.0713548162726f;          // 2 * sqrt(2/pi) * 0.044715
  const float z = x * fmaf(two_c3, x * x, two_c);  // z = 2u
  const float a = fminf(fabsf(z), 18.0f);
  // k = round(a / ln 2) by the add-magic-number trick (1.5 * 2^23)
  const float t = fmaf(a, 1.4426950408889634f, 12582912.0f);
  const float kf = t - 12582912.0f;
  const int k = __float_as_int(t) - 0x4B400000;    // 0 <= k <= 26
  float r = fmaf(kf, -0.693145751953125f, a);     // ln2 high part (exact product)
  r = fmaf(kf, -1.4286068203094173e-06f, r);      // ln2 low part
  const float y = -r;                              // e^-a = 2^-k e^y
  float p = fmaf(y, 1.0f / 720.0f, 1.0f / 120.0f);
  p = fmaf(p, y, 1.0f / 24.0f);
  p = fmaf(p, y, 1.0f / 6.0f);
  p = fmaf(p, y, 0.5f);
  p = fmaf(p, y, 1.0f);
  p = fmaf(p, y, 1.0f);
  const float e = __int_as_float((127 - k) << 23) * p;  // e^-a
  const float h = fmaf(0.5f, e, 0.5f);                   // (1 + e^-a) / 2 in (1/2, 1]
  float inv = fmaf(-1.8823529411764706f, h, 2.8235294117647059f);
  float err = fmaf(-h, inv, 1.0f);
  inv = fmaf(inv, err, inv);
  err = fmaf(-h, inv, 1.0f);
  inv = fmaf(inv, err, inv);
  err = fmaf(-h, inv, 1.0f);
  inv = fmaf(inv, err, inv);
  const float sig_pos = 0.5f * inv;                      // sigma(a) = 1 / (1 + e^-a)
  const float sig = (z >= 0.0f) ? sig_pos : e * sig_pos;
  return x * sig;
}

// The same evaluation for two arguments at once, with the packed fp32x2 FMA
// pipe instructions (fma/mul/add.rn.f32x2) wherever both lanes do the same
// arithmetic; exp(-r) uses the Taylor polynomial in r with alternating signs
// (the same polynomial as above, T6(-r)).  Identical results to calling
// gelu_tanh_alu on each argument up to the order of roundings.
__device__ __forceinline__ void gelu_tanh_alu2(float x0, float x1, float& y0, float& y1) {
  const uint64_t x = ptx::f2_pack(x0, x1);
  const uint64_t xx = ptx::f2_mul(x, x);
  const uint64_t z = ptx::f2_mul(x, ptx::f2_fma(ptx::f2_splat(0.0713548162726f), xx, ptx::f2_splat(1.5957691216057308f)));
  float z0, z1;
  ptx::f2_unpack(z, z0, z1);
  const uint64_t a = ptx::f2_pack(fminf(fabsf(z0), 18.0f), fminf(fabsf(z1), 18.0f));
  const uint64_t magic = ptx::f2_splat(12582912.0f);
  const uint64_t t = ptx::f2_fma(a, ptx::f2_splat(1.4426950408889634f), magic);
  const uint64_t kf = ptx::f2_sub(t, magic);
  uint64_t r = ptx::f2_fma(kf, ptx::f2_splat(-0.693145751953125f), a);
  r = ptx::f2_fma(kf, ptx::f2_splat(-1.4286068203094173e-06f), r);
  uint64_t p = ptx::f2_fma(ptx::f2_splat(1.0f / 720.0f), r, ptx::f2_splat(-1.0f / 120.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(1.0f / 24.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(-1.0f / 6.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(0.5f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(-1.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(1.0f));
  float t0, t1;
  ptx::f2_unpack(t, t0, t1);
  const int k0 = __float_as_int(t0) - 0x4B400000, k1 = __float_as_int(t1) - 0x4B400000;
  const uint64_t e = ptx::f2_mul(ptx::f2_pack(__int_as_float((127 - k0) << 23), __int_as_float((127 - k1) << 23)), p);
  const uint64_t h = ptx::f2_fma(ptx::f2_splat(0.5f), e, ptx::f2_splat(0.5f));
  const uint64_t one = ptx::f2_splat(1.0f);
  const uint64_t nh = ptx::f2_mul(h, ptx::f2_splat(-1.0f));
  uint64_t inv = ptx::f2_fma(ptx::f2_splat(-1.8823529411764706f), h, ptx::f2_splat(2.8235294117647059f));
  uint64_t err = ptx::f2_fma(nh, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  err = ptx::f2_fma(nh, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  err = ptx::f2_fma(nh, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  const uint64_t sp = ptx::f2_mul(ptx::f2_splat(0.5f), inv);  // sigma(a)
  const uint64_t sn = ptx::f2_mul(e, sp);                      // sigma(-a)
  float sp0, sp1, sn0, sn1;
  ptx::f2_unpack(sp, sp0, sp1);
  ptx::f2_unpack(sn, sn0, sn1);
  y0 = x0 * (z0 >= 0.0f ? sp0 : sn0);
  y1 = x1 * (z1 >= 0.0f ? sp1 : sn1);
}

}  // namespace gdpa
