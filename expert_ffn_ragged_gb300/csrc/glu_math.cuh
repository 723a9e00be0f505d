// glu_math.cuh -- the SiLU-GLU arithmetic of the fused epilogues and of the
// standalone GLU kernels.
//
// MaxText PR #5760 ("MoE wo FSDP sharding and valid-rows-only MoE kernels",
// commit message, kernels/ragged/glu_rows.py) fixes the forward op sequence:
// negate, exp, +1, divide, multiply, in f32, rounding only the output.  The
// backward sequence (the page gives none) is
//   e = exp(-g), den = 1 + e, sig = 1 / den, silu = g / den,
//   d_up = d * silu, d_gate = (d * u) * (sig * (1 + g * (1 - sig))),
// and any result that rounds to bf16 -0 is stored as +0 (the page's
// "-0 -> +0 fix").
//
// Results are held to the float64 values within a bf16 ulp; the standalone
// kernels must in addition give the sequence's bits wherever a result is
// special (an infinity or NaN, or a gate whose exp(-g) overflows binary32).
// Neither needs the sequence's own divisions: both evaluate the logistic in
// its two-sided stable form,
//   t = exp(-|g|) in (0, 1],  r = 1 / (1 + t) in [1/2, 1),
//   g >= 0: sig = r,    1 - sig = t r
//   g <  0: sig = t r,  1 - sig = r,
// so the reciprocal never sees a denominator above 2 and 1 - sig never
// cancels.  exp comes from the hardware base-2 exponential,
// exp(x) = 2^(x log2 e), and 1/x from the hardware reciprocal, both the
// .approx forms without flush-to-zero, so t keeps its subnormal values down
// to 2^-149.  Relative error of sig, silu and their products: a few f32 ulps.
// +-inf, NaN and -0 gates give the sequence's results.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace rd {

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Fused epilogues (compared with float64 only).  Gates between -103 and
// -88.7, where exp(-g) overflows in the sequence and silu comes out zero,
// keep their tiny silu here.

// sig = logistic(g) and 1 - sig
__device__ __forceinline__ void sigmoid_two_sided(float g, float& sig, float& one_minus_sig) {
  const float t = exp2_approx(-fabsf(g) * 1.44269504088896341f);  // exp(-|g|)
  const float r = rcp_approx(1.0f + t);
  const float tr = t * r;
  const bool pos = g >= 0.0f;
  sig = pos ? r : tr;
  one_minus_sig = pos ? tr : r;
}

__device__ __forceinline__ float glu_fwd_fast(float g, float u) {
  float sig, om;
  sigmoid_two_sided(g, sig, om);
  return (g * sig) * u;
}

__device__ __forceinline__ void glu_bwd_fast(float g, float u, float d, float& d_gate,
                                             float& d_up) {
  float sig, om;
  sigmoid_two_sided(g, sig, om);
  d_up = d * (g * sig);
  d_gate = (d * u) * (sig * (1.0f + g * om));
}

// ---------------------------------------------------------------------------
// Standalone kernels (special results bit for bit).  Two selects reproduce
// the sequence's exact intermediates: when 1 + t rounds to 1 (|g| above 16.6)
// the reciprocal is taken as exactly 1, as the sequence divides by exactly 1
// there; when exp(-g) overflows (g below -ln(FLT_MAX), and g = -inf) sig is 0
// and 1 - sig is 1, as 1 / inf and 1 - 0 in the sequence, so silu = g * 0 is
// -0 (NaN for g = -inf) like g / inf.  Products of bf16 values never fall
// within an ulp of binary32's overflow threshold, so the remaining few-ulp
// differences never move a result across it.
__device__ __forceinline__ void sigmoid_two_sided_seq(float g, float& sig, float& one_minus_sig) {
  const float t = exp2_approx(-fabsf(g) * 1.44269504088896341f);
  const float den = 1.0f + t;
  const float r = den == 1.0f ? 1.0f : rcp_approx(den);
  const float tr = t * r;
  const bool pos = g >= 0.0f;
  const bool over = g < -88.7228394f;  // exp(-g) > FLT_MAX
  sig = over ? 0.0f : (pos ? r : tr);
  one_minus_sig = over ? 1.0f : (pos ? tr : r);
}

__device__ __forceinline__ float glu_fwd_seq(float g, float u) {
  float sig, om;
  sigmoid_two_sided_seq(g, sig, om);
  return (g * sig) * u;
}

__device__ __forceinline__ void glu_bwd_seq(float g, float u, float d, float& d_gate,
                                            float& d_up) {
  float sig, om;
  sigmoid_two_sided_seq(g, sig, om);
  d_up = d * (g * sig);
  d_gate = (d * u) * (sig * (1.0f + g * om));
}

// two floats -> packed bf16x2 (round to nearest even), lower half first
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// packed bf16x2 with every -0 half replaced by +0
__device__ __forceinline__ uint32_t bf16x2_neg_zero_to_pos(uint32_t v) {
  if ((v & 0xFFFFu) == 0x8000u) v &= 0xFFFF0000u;
  if ((v >> 16) == 0x8000u) v &= 0x0000FFFFu;
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace rd
