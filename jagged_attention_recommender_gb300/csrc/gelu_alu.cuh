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

}  // namespace gdpa
