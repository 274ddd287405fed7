// fsa_mx.cuh -- MX (OCP microscaling) quantisation of one 32-element block,
// shared by the quantisation kernels (fsa_quant.cu) and the attention kernel's
// fused quantisation of Q (fsa_attn.cu), so both write the same codes and scales.
//
// Blocks of 32 elements share one E8M0 scale 2^E with
// E = clamp(floor(log2 amax) - emax, -127, 127) (emax 8 for E4M3, 4 for E3M2, 2 for
// E2M3 and E2M1); element codes are x * 2^-E rounded to nearest even with saturation
// (cvt.rn.satfinite); a block with a non-finite element gets scale 0xFF.
#pragma once
#include <cstdint>
#include "fsa_ptx.cuh"

namespace fsa {

// Storage formats (fsa.h numbering): 0 E4M3, 1 E2M3, 2 E2M1, 4 E3M2.
__host__ __device__ constexpr int mx_emax(int fmt) { return fmt == 0 ? 8 : (fmt == 4 ? 4 : 2); }
__host__ __device__ constexpr bool mx_six_bit(int fmt) { return fmt == 1 || fmt == 4; }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Block exponent from the fp32 bit pattern of amax (exact for bf16 inputs).
// Returns the scale byte; 0xFF for a non-finite block.
__device__ __forceinline__ uint32_t block_scale_byte(float amax, int emax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  if (ef == 0xFF) return 0xFFu;
  int E = ef - 127 - emax;      // zero and subnormal amax fall below -127 and clamp
  E = E < -127 ? -127 : (E > 127 ? 127 : E);
  return (uint32_t)(E + 127);
}

// 2^-E as fp32 for E in [-127, 127] (2^-127..2^127, exact).
__device__ __forceinline__ float pow2_neg(int E) {
  return E == 127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(127 - E) << 23);
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  if constexpr (FMT == 0) return cvt_e4m3x2(lo, hi);
  else if constexpr (FMT == 1) return cvt_e2m3x2(lo, hi);
  else if constexpr (FMT == 4) return cvt_e3m2x2(lo, hi);
  else return cvt_e2m1x2(lo, hi);
}

// Codes of one 32-element block held by one thread, v[0..32): 8 words (E4M3:
// one code per byte; E2M3: two 16-code groups of 12 packed bytes and 4 zero
// bytes) or 4 words (E2M1, two codes per byte, even index in the low nibble).
// Returns the scale byte (0xFF and NaN / zero codes for a non-finite block).
template <int FMT>
__device__ __forceinline__ uint32_t quant_block32(const float* v, uint32_t* w) {
  constexpr int emax = mx_emax(FMT);
  float amax = 0.f;
  bool nonfinite = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = fabsf(v[i]);
    nonfinite |= !(a <= 3.4e38f);
    amax = fmaxf(amax, a);
  }
  const uint32_t sbyte = nonfinite ? 0xFFu : block_scale_byte(amax, emax);
  const float mul = nonfinite ? 1.0f : pow2_neg((int)sbyte - 127);
  uint32_t q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    q[i] = nonfinite ? (FMT == 0 ? 0x7F7Fu : 0u) : cvt_pair<FMT>(__fmul_rn(v[2 * i], mul), __fmul_rn(v[2 * i + 1], mul));
  if constexpr (FMT == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = q[2 * i] | (q[2 * i + 1] << 16);
  } else if constexpr (FMT == 1 || FMT == 4) {
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const uint32_t g[4] = {q[8 * gi] | (q[8 * gi + 1] << 16), q[8 * gi + 2] | (q[8 * gi + 3] << 16),
                             q[8 * gi + 4] | (q[8 * gi + 5] << 16), q[8 * gi + 6] | (q[8 * gi + 7] << 16)};
      pack6x16(g, w + 4 * gi);
      w[4 * gi + 3] = 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = q[4 * i] | (q[4 * i + 1] << 8) | (q[4 * i + 2] << 16) | (q[4 * i + 3] << 24);
  }
  return sbyte;
}

// NVFP4 (fsa.h format 5): E2M1 codes with one E4M3 scale per 16 elements.  The
// scale is the E4M3 value nearest amax / 6 and the codes the E2M1 values nearest
// x / scale, both by a correctly rounded fp32 division and cvt.rn.satfinite: for
// bf16 inputs the fp32 quotient rounds to the same E4M3 / E2M1 code as the exact
// one (neither quotient is within 2^-24 of a rounding boundary unless it is one).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {     // exact: E4M3 fits f16
  float f;
  const uint16_t t = (uint16_t)((b & 0xFFu) | ((b & 0xFFu) << 8));
  asm("{\n .reg .b16 lo, hi;\n .reg .b32 h2;\n cvt.rn.f16x2.e4m3x2 h2, %1;\n"
      " mov.b32 {lo, hi}, h2;\n cvt.f32.f16 %0, lo;\n}" : "=f"(f) : "h"(t));
  return f;
}
// scale byte of a block with maximum magnitude amax (0x7F, the E4M3 NaN, for a
// non-finite block)
__device__ __forceinline__ uint32_t nvfp4_scale_byte(float amax, bool nonfinite) {
  return nonfinite ? 0x7Fu : (cvt_e4m3x2(__fdiv_rn(amax, 6.0f), 0.0f) & 0xFFu);
}
// codes of 8 consecutive elements (one 32-bit word, even element in the low nibble)
// under the block scale s (0 or NaN: zero codes)
__device__ __forceinline__ uint32_t nvfp4_codes8(const float* v, float s) {
  if (!(s > 0.0f)) return 0u;
  uint32_t w = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) w |= cvt_e2m1x2(__fdiv_rn(v[2 * e], s), __fdiv_rn(v[2 * e + 1], s)) << (8 * e);
  return w;
}

}  // namespace fsa
