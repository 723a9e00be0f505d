// glu_math.cuh -- the SiLU-GLU arithmetic of the fused epilogue and of the
// standalone GLU kernels.
//
// MaxText PR #5760 ("MoE wo FSDP sharding and valid-rows-only MoE kernels",
// commit message, kernels/ragged/glu_rows.py) fixes the forward op sequence:
// negate, exp, +1, divide, multiply, in f32, rounding only the output.  Each
// step uses an explicitly rounded intrinsic so the compiler cannot contract
// a multiply and an add into one FMA, which would change the rounding of
// the sequence.  The backward sequence (the page gives none) is
//   e = exp(-g), den = 1 + e, sig = 1 / den, silu = g / den,
//   d_up = d * silu, d_gate = (d * u) * (sig * (1 + g * (1 - sig))),
// and any result that rounds to bf16 -0 is stored as +0 (the page's
// "-0 -> +0 fix").
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace rd {

__device__ __forceinline__ float glu_fwd_f32(float g, float u) {
  const float e = expf(-g);
  const float den = __fadd_rn(1.0f, e);
  const float s = __fdiv_rn(g, den);
  return __fmul_rn(s, u);
}

__device__ __forceinline__ void glu_bwd_f32(float g, float u, float d, float& d_gate,
                                            float& d_up) {
  const float e = expf(-g);
  const float den = __fadd_rn(1.0f, e);
  const float sig = __fdiv_rn(1.0f, den);
  const float silu = __fdiv_rn(g, den);
  d_up = __fmul_rn(d, silu);
  const float dsil = __fmul_rn(sig, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sig))));
  d_gate = __fmul_rn(__fmul_rn(d, u), dsil);
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
