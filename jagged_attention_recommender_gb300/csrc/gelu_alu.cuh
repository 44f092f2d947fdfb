// gelu_alu.cuh -- tanh-GELU (and SiLU, x sigma(x), through the same sigma
// with other constants) by two routes: gelu_tanh_alu2 / gelu_tanh_grad_alu2
// with FMA-pipe and integer instructions only (no special-function-unit
// instruction), and gelu_tanh_sfu2 / gelu_tanh_val_grad_sfu2 with the
// special-function unit's exp2 and reciprocal; act_eval2 picks one per
// launch (gdpa_set_act_route).
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
//   1/(1+e^-a), the divisor d in (1, 2]:  Newton-Raphson from a quadratic
//          seed fitted to 1/d on [1, 2] by iteratively reweighted least
//          squares in relative error (maximum relative error 1.01e-2), two
//          steps (1e-8).
//
// The score scale folds into the cubic: for x = scale * s,
// z = s * (A + C s^2) with A = 2 sqrt(2/pi) scale and C = A * 0.044715 scale^2,
// and the routine returns s * sigma(z) = gelu(x) / scale; the caller applies
// the scale once per output row (any sign, and scale = 0 gives 0).
//
// Truncation error of T6 on |r| <= ln2/2 is below 2e-7 relative; the clamp at
// |z| = 18 changes sigma by less than 2e-8.  Emulated in fp32 the whole
// evaluation is within 5.2e-7 of the exact tanh-GELU for |x| <= 17, and it
// saturates to x or 0 beyond.
#pragma once

#include "sm103_ptx.cuh"

namespace gdpa {

// Two arguments at once with the packed fp32x2 FMA-pipe instructions
// (fma/mul/add.rn.f32x2) wherever both lanes do the same arithmetic.
// Returns y = s * sigma(z(s)) for each lane; see the header for A and C.
__device__ __forceinline__ void gelu_tanh_alu2(float s0, float s1, uint64_t A2, uint64_t C2, float& y0, float& y1) {
  const uint64_t s = ptx::f2_pack(s0, s1);
  const uint64_t z = ptx::f2_mul(s, ptx::f2_fma(C2, ptx::f2_mul(s, s), A2));
  float z0, z1;
  ptx::f2_unpack(z, z0, z1);
  const uint64_t a = ptx::f2_pack(fminf(fabsf(z0), 18.0f), fminf(fabsf(z1), 18.0f));
  const uint64_t magic = ptx::f2_splat(12582912.0f);  // 1.5 * 2^23: round to nearest integer
  const uint64_t t = ptx::f2_fma(a, ptx::f2_splat(1.4426950408889634f), magic);
  const uint64_t kf = ptx::f2_sub(t, magic);
  uint64_t r = ptx::f2_fma(kf, ptx::f2_splat(-0.693145751953125f), a);  // ln2 high part (exact product)
  r = ptx::f2_fma(kf, ptx::f2_splat(-1.4286068203094173e-06f), r);      // ln2 low part
  // e^-r = T6(-r), Horner in r with alternating signs
  uint64_t p = ptx::f2_fma(ptx::f2_splat(1.0f / 720.0f), r, ptx::f2_splat(-1.0f / 120.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(1.0f / 24.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(-1.0f / 6.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(0.5f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(-1.0f));
  p = ptx::f2_fma(p, r, ptx::f2_splat(1.0f));
  float t0, t1;
  ptx::f2_unpack(t, t0, t1);
  const int k0 = __float_as_int(t0) - 0x4B400000, k1 = __float_as_int(t1) - 0x4B400000;  // 0 <= k <= 26
  const uint64_t e = ptx::f2_mul(ptx::f2_pack(__int_as_float((127 - k0) << 23), __int_as_float((127 - k1) << 23)), p);
  // sigma(a) = 1/d, d = 1 + e^-a in (1, 2]; nd = -d
  const uint64_t nd = ptx::f2_fma(e, ptx::f2_splat(-1.0f), ptx::f2_splat(-1.0f));
  uint64_t inv = ptx::f2_fma(ptx::f2_fma(ptx::f2_splat(0.3232244551181793f), nd, ptx::f2_splat(1.4545105695724487f)), nd,
                             ptx::f2_splat(2.1211774349212646f));
  const uint64_t one = ptx::f2_splat(1.0f);
  uint64_t err = ptx::f2_fma(nd, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  err = ptx::f2_fma(nd, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  // sigma(z) = sigma(a) for z >= 0, e^-a sigma(a) otherwise
  float e0, e1;
  ptx::f2_unpack(e, e0, e1);
  const uint64_t sel = ptx::f2_pack(z0 >= 0.0f ? 1.0f : e0, z1 >= 0.0f ? 1.0f : e1);
  ptx::f2_unpack(ptx::f2_mul(s, ptx::f2_mul(inv, sel)), y0, y1);
}

// The same y = s * sigma(z(s)) with sigma taken on the special-function
// unit: sigma(z) = 1 / (1 + 2^(-z log2 e)), one ex2.approx and one
// rcp.approx per argument.  NA2 and NC2 are -log2(e) A and -log2(e) C, so
// that the cubic gives t = -z log2 e directly.  Both instructions keep about
// 22 bits, so the result matches gelu_tanh_alu2 to fp32 level; a large
// positive t gives 2^t = inf and sigma = 0, a large negative one sigma = 1.
// The forward kernels evaluate part of each row with this form and the rest
// with gelu_tanh_alu2, so that the special-function unit and the FMA pipe
// share the work.
__device__ __forceinline__ void gelu_tanh_sfu2(float s0, float s1, uint64_t NA2, uint64_t NC2, float& y0,
                                               float& y1) {
  const uint64_t s = ptx::f2_pack(s0, s1);
  const uint64_t t = ptx::f2_mul(s, ptx::f2_fma(NC2, ptx::f2_mul(s, s), NA2));
  float t0, t1;
  ptx::f2_unpack(t, t0, t1);
  const uint64_t d = ptx::f2_add(ptx::f2_pack(ptx::ex2_approx(t0), ptx::ex2_approx(t1)), ptx::f2_splat(1.0f));
  float d0, d1;
  ptx::f2_unpack(d, d0, d1);
  ptx::f2_unpack(ptx::f2_mul(s, ptx::f2_pack(ptx::rcp_approx(d0), ptx::rcp_approx(d1))), y0, y1);
}

// Derivative for the backward: with x = scale * s and z = s (A + C s^2),
// gelu'(x) = sigma(z) + sigma(z) sigma(-z) s (A + 3 C s^2), where
// sigma(z) sigma(-z) = e^-a sigma(a)^2 (a = |z|) is formed without the
// cancellation of sigma(1 - sigma).  Same evaluation of e^-a and sigma(a)
// as gelu_tanh_alu2; returns gelu'(x) for each lane.
__device__ __forceinline__ void gelu_tanh_grad_alu2(float s0, float s1, uint64_t A2, uint64_t C2, float& g0, float& g1) {
  const uint64_t s = ptx::f2_pack(s0, s1);
  const uint64_t ss = ptx::f2_mul(s, s);
  const uint64_t z = ptx::f2_mul(s, ptx::f2_fma(C2, ss, A2));
  float z0, z1;
  ptx::f2_unpack(z, z0, z1);
  const uint64_t a = ptx::f2_pack(fminf(fabsf(z0), 18.0f), fminf(fabsf(z1), 18.0f));
  const uint64_t magic = ptx::f2_splat(12582912.0f);  // 1.5 * 2^23: round to nearest integer
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
  const uint64_t nd = ptx::f2_fma(e, ptx::f2_splat(-1.0f), ptx::f2_splat(-1.0f));
  uint64_t inv = ptx::f2_fma(ptx::f2_fma(ptx::f2_splat(0.3232244551181793f), nd, ptx::f2_splat(1.4545105695724487f)), nd,
                             ptx::f2_splat(2.1211774349212646f));
  const uint64_t one = ptx::f2_splat(1.0f);
  uint64_t err = ptx::f2_fma(nd, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  err = ptx::f2_fma(nd, inv, one);
  inv = ptx::f2_fma(inv, err, inv);
  float e0, e1;
  ptx::f2_unpack(e, e0, e1);
  const uint64_t sig = ptx::f2_mul(inv, ptx::f2_pack(z0 >= 0.0f ? 1.0f : e0, z1 >= 0.0f ? 1.0f : e1));
  const uint64_t sig2 = ptx::f2_mul(e, ptx::f2_mul(inv, inv));                       // sigma(z) sigma(-z)
  const uint64_t dz = ptx::f2_mul(s, ptx::f2_fma(ptx::f2_mul(C2, ptx::f2_splat(3.0f)), ss, A2));  // s (A + 3 C s^2)
  ptx::f2_unpack(ptx::f2_fma(sig2, dz, sig), g0, g1);
}

// Value and derivative for the backward with sigma on the special-function
// unit: a = |z|, e = 2^(-a log2 e) (ex2.approx), sigma(a) = 1/(1+e)
// (rcp.approx); sigma(z) = sigma(a) for z >= 0, e sigma(a) otherwise;
// sigma(z) sigma(-z) = e sigma(a)^2.  Returns y = s sigma(z) (the forward's
// value) and gelu'(x) = sigma(z) + sigma(z) sigma(-z) s (A + 3 C s^2), as
// gelu_tanh_alu2 and gelu_tanh_grad_alu2 do.
__device__ __forceinline__ void gelu_tanh_val_grad_sfu2(float s0, float s1, uint64_t A2, uint64_t C2, float& y0,
                                                        float& y1, float& g0, float& g1) {
  const uint64_t s = ptx::f2_pack(s0, s1);
  const uint64_t ss = ptx::f2_mul(s, s);
  const uint64_t z = ptx::f2_mul(s, ptx::f2_fma(C2, ss, A2));
  float z0, z1;
  ptx::f2_unpack(z, z0, z1);
  const uint64_t t = ptx::f2_mul(ptx::f2_pack(fabsf(z0), fabsf(z1)), ptx::f2_splat(-1.4426950408889634f));
  float t0, t1;
  ptx::f2_unpack(t, t0, t1);
  const uint64_t e = ptx::f2_pack(ptx::ex2_approx(t0), ptx::ex2_approx(t1));
  float d0, d1;
  ptx::f2_unpack(ptx::f2_add(e, ptx::f2_splat(1.0f)), d0, d1);
  const uint64_t inv = ptx::f2_pack(ptx::rcp_approx(d0), ptx::rcp_approx(d1));
  float e0, e1;
  ptx::f2_unpack(e, e0, e1);
  const uint64_t sig = ptx::f2_mul(inv, ptx::f2_pack(z0 >= 0.0f ? 1.0f : e0, z1 >= 0.0f ? 1.0f : e1));
  ptx::f2_unpack(ptx::f2_mul(s, sig), y0, y1);
  const uint64_t sig2 = ptx::f2_mul(e, ptx::f2_mul(inv, inv));
  const uint64_t dz = ptx::f2_mul(s, ptx::f2_fma(ptx::f2_mul(C2, ptx::f2_splat(3.0f)), ss, A2));
  ptx::f2_unpack(ptx::f2_fma(sig2, dz, sig), g0, g1);
}

// One launch's activation constants and route: sfu selects gelu_tanh_sfu2
// (sigma on the special-function unit), otherwise gelu_tanh_alu2 (the
// FMA-pipe polynomial).  Both return s sigma(s (A + C s^2)).
struct ActK {
  uint64_t A2, C2, NA2, NC2;
  bool sfu;
};
__device__ __forceinline__ ActK act_k(float A, float C, int sfu) {
  ActK k;
  k.A2 = ptx::f2_splat(A);
  k.C2 = ptx::f2_splat(C);
  k.NA2 = ptx::f2_splat(-1.4426950408889634f * A);
  k.NC2 = ptx::f2_splat(-1.4426950408889634f * C);
  k.sfu = sfu != 0;
  return k;
}
__device__ __forceinline__ void act_eval2(const ActK& k, float s0, float s1, float& y0, float& y1) {
  if (k.sfu)
    gelu_tanh_sfu2(s0, s1, k.NA2, k.NC2, y0, y1);
  else
    gelu_tanh_alu2(s0, s1, k.A2, k.C2, y0, y1);
}

// The folded constants of the ALU activations, for which the routines above
// return y = s sigma(s (A + C s^2)) = act(scale s) / scale:
//   tanh-GELU: A = 2 sqrt(2/pi) scale, C = 0.044715 A scale^2
//   SiLU:      A = scale, C = 0           (silu(x) = x sigma(x))
// gelu_tanh_grad_alu2 then returns act'(scale s) for either.
__host__ __device__ inline void alu_act_consts(bool silu, float scale, float& A, float& C) {
  A = silu ? scale : 1.5957691216057308f * scale;
  C = silu ? 0.0f : A * 0.044715f * scale * scale;
}

}  // namespace gdpa
