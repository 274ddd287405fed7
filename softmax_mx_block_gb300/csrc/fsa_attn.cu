// fsa_attn.cu -- fused MX attention forward for sm_103a (and its BF16
// exact-softmax twin).
//
// What it computes (page titles and sections):
//  * "Fused-Softmax for efficient quantized attention", abstract: QK^T and PV
//    as MX block-scaled GEMMs, softmax reformulated so its work folds into them.
//  * "Moving softmax to matrix operations speeds up AI inference by over 2x",
//    summary / "Read it as" / "How it works" figure: the max subtraction and
//    exponentiation are one fused multiply-add on the score GEMM's output; the
//    row maximum is frozen speculatively with a fallback; a fast exponential;
//    "Exp + MX Quant" fused; probabilities summed on the matrix unit.
//  * "EFQ-Softmax: Exp-Free Quantization for Softmax", abstract: per 32-key
//    block an exponent-only scale from the local maximum and nonnegative E2M1
//    codes by one affine rule; the same operand feeds P~V and P~1; final
//    normalisation in high precision.
//
// Per query row and key tile of 128 (ascending), with s the raw fp32 score and
// c = fp32(scale * log2 e):
//   mx = tile max, x = fp32(mx*c); first tile: M = x; later: x > fp32(M + delta)
//   -> fallback: O_aug *= 2^(M - M'), M' = x (delta: margin of the fallback test).
//   per 32-key block: E = clamp(floor(fp32(fp32(smax*c) - M)) - emax, -127, 127),
//   r = fma(s, c, -fp32(M + E)); code = RN(exp2approx(r)) in the P format, or
//   EFQ: code = clamp(rne(2 r + beta), 0, 7); scale byte E + 127.
//   O_aug += P~ [V^ | 1]: column D of O_aug is the denominator l.
//   O = O_aug[:, :D] / l in fp32.
//
// CTA = one 128-row query tile of one (batch, head); 10 warps: warp 0 issues
// TMA loads, warp 1 issues the tcgen05 MMAs and owns tensor memory, warps 2..9
// are the softmax warps, two per tensor-memory lane quadrant, which take
// alternate key tiles (thread = one row, all 128 keys of the tile).  S is
// double buffered in tensor memory and released as soon as a softmax warp holds
// it in registers; P~ goes to buffers of its own, from which the PV MMA reads
// it; O_aug stays in tensor memory until the end.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "fsa_launch.h"
#include "fsa_mx.cuh"

namespace fsa {

constexpr float kNegInf = -__builtin_huge_valf();

// ---- packed fp32 pairs (f32x2 FMA-pipe ops on sm_100-family) ------------------
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fadd2_rm(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rm.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// max of 32 consecutive values (16 three-input max operations)
__device__ __forceinline__ float max32(const float* v) {
  float m0 = max3f(v[0], v[1], v[2]), m1 = max3f(v[3], v[4], v[5]), m2 = max3f(v[6], v[7], v[8]);
  float m3 = max3f(v[9], v[10], v[11]), m4 = max3f(v[12], v[13], v[14]), m5 = max3f(v[15], v[16], v[17]);
  float m6 = max3f(v[18], v[19], v[20]), m7 = max3f(v[21], v[22], v[23]), m8 = max3f(v[24], v[25], v[26]);
  float m9 = max3f(v[27], v[28], v[29]);
  m0 = max3f(m0, m1, m2);
  m3 = max3f(m3, m4, m5);
  m6 = max3f(m6, m7, m8);
  m9 = max3f(m9, v[30], v[31]);
  return fmaxf(max3f(m0, m3, m6), m9);
}

// Cubic through 2^f at f = 0, 1/3, 2/3, 1 (coefficients solved in fp64 from the
// four nodes and rounded to fp32), Horner with fused multiply-adds; 2^n by
// exponent addition after clamping r below at -64.  Two values at a time:
// floor(r) comes from adding 1.5*2^23 rounded toward -inf (exact for
// |r| < 2^22), f = r - floor(r) is exact, and 2^n is one integer multiply-add
// on the exponent field.
constexpr float kC3 = 0x1.43aa72p-4f, kC2 = 0x1.ccca58p-3f, kC1 = 0x1.64581cp-1f;
__device__ __forceinline__ void exp2_poly2(float& a, float& b) {
  const uint64_t r = pk2(fmaxf(a, -64.0f), fmaxf(b, -64.0f));
  const uint64_t j = fadd2_rm(r, pk2(12582912.0f, 12582912.0f));           // floor(r) + 1.5*2^23
  const uint64_t n = ffma2(j, pk2(1.0f, 1.0f), pk2(-12582912.0f, -12582912.0f));
  const uint64_t f = ffma2(n, pk2(-1.0f, -1.0f), r);                         // r - floor(r), exact
  uint64_t p = ffma2(pk2(kC3, kC3), f, pk2(kC2, kC2));
  p = ffma2(p, f, pk2(kC1, kC1));
  p = ffma2(p, f, pk2(1.0f, 1.0f));
  float p0, p1, j0, j1;
  upk2(p, p0, p1);
  upk2(j, j0, j1);
  // (bits(j) - bits(1.5*2^23)) << 23 == bits(j) << 23 (mod 2^32): the magic's low 9 bits are 0
  a = __int_as_float(__float_as_int(p0) + (__float_as_int(j0) << 23));
  b = __int_as_float(__float_as_int(p1) + (__float_as_int(j1) << 23));
}

// exp2 of 32 residuals in place.  EXPM 0: all by the cubic; 1: all by ex2.approx;
// 2: key positions 4k+3 by the cubic, the others by ex2.approx.
template <int EXPM>
__device__ __forceinline__ void exp2_block(float* v) {
  if constexpr (EXPM == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) exp2_poly2(v[i], v[i + 1]);
  } else if constexpr (EXPM == 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = ex2_approx(v[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      exp2_poly2(v[i + 3], v[i + 7]);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if ((e & 3) != 3) v[i + e] = ex2_approx(v[i + e]);
    }
  }
}

__device__ __forceinline__ uint32_t pack_b16x2(uint16_t lo, uint16_t hi) {
  uint32_t r;
  asm("mov.b32 %0, {%1, %2};" : "=r"(r) : "h"(lo), "h"(hi));
  return r;
}
__device__ __forceinline__ uint16_t cvt16_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t cvt16_e2m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t cvt16_e3m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// clamp(floor(t) - emax, -127, 127) in fp32, on the FMA pipe only (no conversions,
// no floorf): floor(t) is t + 1.5*2^23 rounded down, minus 1.5*2^23, exact for
// |t| < 2^22; a larger |t| only moves a result the clamp takes to -127 or 127 anyway
// (the sum stays on the same side), and NaN and -inf give -127, +inf 127.
// FOLD: subtract 1.5*2^23 + emax at once (the same exact integer subtraction, one
// add fewer); the exp paths keep the separate add, which measured faster there.
template <int EMAX, bool FOLD>
__device__ __forceinline__ float block_exp_f(float t) {
  static_assert(EMAX >= 0 && EMAX < 64, "exponent offset");
  const float fl = FOLD ? __fsub_rn(__fadd_rd(t, 12582912.0f), 12582912.0f + (float)EMAX)
                        : __fadd_rn(__fsub_rn(__fadd_rd(t, 12582912.0f), 12582912.0f), -(float)EMAX);
  return fminf(fmaxf(fl, -127.0f), 127.0f);
}
// scale byte E + 127 in the low byte of the bits of E + 127 + 2^23 (an integer below
// 2^24, exact); the caller gathers the low bytes of a tile's four blocks into one word
__device__ __forceinline__ uint32_t scale_word_f(float E) { return __float_as_uint(__fadd_rn(E, 8388735.0f)); }
// bytes 0 of a, b, c, d as one word (a in the low byte)
__device__ __forceinline__ uint32_t low_bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return prmt(prmt(a, b, 0x0040u), prmt(c, d, 0x0040u), 0x5410u);
}

// Exponent-only block scale: E = clamp(floor(fp32(fp32(smax*c) - M)) - emax, -127, 127).
// Returns E (as fp32) and writes -fp32(M + E).  A block with no visible key (smax = -inf)
// gets E = -127; its scores are -inf, so every code comes out 0.  A row with no
// visible key at all so far (M = -inf: causal rows before the first key) gets the
// shift 0, so that its residuals are -inf as well (not -inf + inf, whose NaN a
// format without a NaN code would saturate to a nonzero code).
template <int FPV>
__device__ __forceinline__ float block_exp(float bmax, float c, float M, float& nbE) {
  const float tmax = __fsub_rn(__fmul_rn(bmax, c), M);
  const float E = block_exp_f<Fmt<FPV>::emax, false>(tmax);
  nbE = M == kNegInf ? 0.0f : -__fadd_rn(M, E);
  return E;
}

__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// P codes of one 32-key block, in place: v[0..32) holds the raw scores (masked =
// -inf) on entry and is clobbered.  Writes 8 packed words (one byte per code) or 4
// (E2M1) to out[] and returns a word whose low byte is the scale byte E + 127.
template <int FPV, int EXPM>
__device__ __forceinline__ uint32_t pgen_block(float* v, float bmax, float c, float M, const KParams& p, uint32_t* out) {
  if constexpr (FPV == F_EFQ) {
    // EFQ: block exponent E = clamp(floor(fp32(tmax + phi)) - 2, -127, 127) from the
    // block maximum; then one fused multiply-add per score maps it to the code domain,
    // y = s * A + Bk with A = fp32(a c) and Bk = fp32(b - fp32(a fp32(M + E))), and
    // code = clamp(rne(y), 0, 7).  Computed as z = sat(y / 8) (the scaling by 1/8 is
    // exact, so z is fp32(y) / 8 clamped to [0, 1]); then z + 1.5*2^20 rounds 8z to
    // the nearest integer (ties to even) in the low bits of the sum.  A block with no
    // visible key has M + E = -inf, Bk = +inf and y NaN: sat gives 0.
    // EXPM 1: the host has checked that codes cannot exceed 7 (every residual is
    // below 3 - phi when the block exponent is not clamped from above, i.e. margin
    // delta <= 120, and a (3 - phi) + b < 7.49), so the nibbles need no fix; EXPM 0:
    // any constants, nibbles equal to 8 become 7.
    const float tmax = __fsub_rn(__fmul_rn(bmax, c), M);
    const float Ef = block_exp_f<2, true>(__fadd_rn(tmax, p.efq_phi));
    const float bE = __fadd_rn(M, Ef);
    // Bk / 8 = fp32(b/8 - fp32(a/8 * bE)): the same roundings as fp32(b - fp32(a bE)), scaled
    const float b8 = __fsub_rn(p.efq_b8, __fmul_rn(p.efq_a8, bE));
    const float a8 = p.efq_A8;
    const uint64_t mg = pk2(1572864.0f, 1572864.0f);                       // 1.5 * 2^20
    uint32_t t[32];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float k0, k1;
      upk2(fadd2(pk2(fma_sat(v[i], a8, b8), fma_sat(v[i + 1], a8, b8)), mg), k0, k1);
      t[i] = __float_as_uint(k0);
      t[i + 1] = __float_as_uint(k1);
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t* u = t + 8 * w;
      // the low byte of (u1 << 4) + u0 is k0 | k1 << 4 (the magic's bits stay above bit 21)
      const uint32_t a01 = (u[1] << 4) + u[0], a23 = (u[3] << 4) + u[2];
      const uint32_t a45 = (u[5] << 4) + u[4], a67 = (u[7] << 4) + u[6];
      const uint32_t wv = prmt(prmt(a01, a23, 0x0040u), prmt(a45, a67, 0x0040u), 0x5410u);
      // EXPM 0: codes are 0..8; turn each nibble equal to 8 into 7 (no nibble of 0..7
      // has bit 3)
      out[w] = EXPM == 1 ? wv : wv - ((wv >> 3) & 0x11111111u);
    }
    return scale_word_f(Ef);
  } else {
    float nb;
    const float Ef = block_exp<FPV>(bmax, c, M, nb);
    const uint64_t c2 = pk2(c, c), nb2 = pk2(nb, nb);
#pragma unroll
    for (int i = 0; i < 32; i += 2) upk2(ffma2(pk2(v[i], v[i + 1]), c2, nb2), v[i], v[i + 1]);
    exp2_block<EXPM>(v);
    if constexpr (FPV == F_E4M3) {
#pragma unroll
      for (int w = 0; w < 8; ++w)
        out[w] = pack_b16x2(cvt16_e4m3x2(v[4 * w], v[4 * w + 1]), cvt16_e4m3x2(v[4 * w + 2], v[4 * w + 3]));
    } else if constexpr (FPV == F_E2M3) {
      // tensor memory holds 6-bit A operands one per byte (low 6 bits)
#pragma unroll
      for (int w = 0; w < 8; ++w)
        out[w] = pack_b16x2(cvt16_e2m3x2(v[4 * w], v[4 * w + 1]), cvt16_e2m3x2(v[4 * w + 2], v[4 * w + 3]));
    } else if constexpr (FPV == F_E3M2) {
#pragma unroll
      for (int w = 0; w < 8; ++w)
        out[w] = pack_b16x2(cvt16_e3m2x2(v[4 * w], v[4 * w + 1]), cvt16_e3m2x2(v[4 * w + 2], v[4 * w + 3]));
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t b01 = cvt_e2m1x2(v[8 * w], v[8 * w + 1]), b23 = cvt_e2m1x2(v[8 * w + 2], v[8 * w + 3]);
        const uint32_t b45 = cvt_e2m1x2(v[8 * w + 4], v[8 * w + 5]), b67 = cvt_e2m1x2(v[8 * w + 6], v[8 * w + 7]);
        out[w] = prmt(prmt(b01, b23, 0x0040u), prmt(b45, b67, 0x0040u), 0x5410u);
      }
    }
    return scale_word_f(Ef);
  }
}

}  // namespace fsa

namespace fsa {

// Q quantised in the prologue: thread u of the 256 softmax threads takes row u % 128
// and half u / 128 of the bf16 tile `raw` (128 rows x 2D bytes), quantises its
// 32-element blocks exactly as the quantisation kernel does (quant_block32), and
// writes the codes into the MMA's K-major swizzled Q tile and the scale bytes into
// the tile's 128x4 scale atom (unused slots 0x7F).  Rows past Sq arrive as zeros.
template <int FQK, int D>
__device__ __forceinline__ void quantize_q_tile(const uint8_t* raw, uint8_t* sQ, uint8_t* sfq, int u) {
  using C = Cfg<FQK, FQK == F_E2M1 ? F_E2M1 : FQK, D>;
  constexpr int W = C::W_QK;
  constexpr int NB = D / 64;                       // blocks per thread
  constexpr int BB = FQK == F_E2M1 ? 16 : 32;      // code bytes per block
  const int r = u & 127, hf = u >> 7;
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    const int blk = hf * NB + i;
    const uint4* src = reinterpret_cast<const uint4*>(raw + r * (2 * D) + blk * 64);
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 x = src[c];
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[8 * c + 2 * e] = bf16_to_f32((uint16_t)(xs[e] & 0xFFFFu));
        v[8 * c + 2 * e + 1] = bf16_to_f32((uint16_t)(xs[e] >> 16));
      }
    }
    uint32_t w[8];
    const uint32_t sb = quant_block32<FQK>(v, w);
#pragma unroll
    for (int cc = 0; cc < BB / 16; ++cc) {
      const int o = blk * BB + 16 * cc;            // byte offset within the row
      const int ka = o / W, c = (o % W) / 16;
      const int sc = W == 128 ? (c ^ (r & 7)) : (W == 64 ? (c ^ ((r >> 1) & 3)) : (c ^ ((r >> 2) & 1)));
      *reinterpret_cast<uint4*>(sQ + ka * 128 * W + r * W + (sc << 4)) =
          make_uint4(w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
    }
    sfq[(r & 31) * 16 + (r >> 5) * 4 + blk] = (uint8_t)sb;
    if constexpr (D == 64) sfq[(r & 31) * 16 + (r >> 5) * 4 + blk + 2] = 0x7F;
  }
}

// DBG: the debug instance, which also writes each tile's raw scores, its frozen
// maximum and its P~ code and scale words to the dump buffers of KParams (tests).
// QF: Q is given as bf16 (tm_q maps it) and quantised by the softmax warps in the
// prologue, so it makes no round trip through HBM as MX codes.
template <int FQK, int FPV, int D, int EXPM, bool DBG = false, bool QF = false>
__global__ void __launch_bounds__(Cfg<FQK, FPV, D>::NTHREADS, 1)
fsa_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const KParams p, const DbgParams dbg) {
  using C = Cfg<FQK, FPV, D, false, QF>;
  constexpr int KIND_QK = Fmt<FQK>::kind, KIND_PV = Fmt<FPV>::kind;
  constexpr bool MX = C::MX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // the warp index (and below the tensor-memory base) through a lane-0 shuffle, which
  // the compiler knows to be warp-uniform: addresses derived from them stay uniform
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;

  // ---- work item
  // causal: one kv head (batch and kv head) per slow grid index, and on the fast axis
  // its query tiles heaviest first, the G = H/Hkv query heads of each tile together:
  // blocks are dispatched kv head by kv head, longest first within each, so the blocks
  // in flight share one kv head's K/V in L2 and the launch ends on short blocks.
  // Otherwise query tiles of one head run together and share its K/V in L2.
  const int G = p.H / p.Hkv;
  const int qt = p.causal ? (p.n_qtiles - 1 - (int)blockIdx.x / G) : (int)blockIdx.x;
  const int h = p.causal ? ((int)blockIdx.y % p.Hkv) * G + (int)blockIdx.x % G : (int)blockIdx.y;
  const int b = p.causal ? (int)blockIdx.y / p.Hkv : (int)blockIdx.z;
  const int kvh = h / (p.H / p.Hkv);
  const int q0 = qt * 128;
  const int nkt = (p.Sk + 127) / 128;
  int nT = nkt;
  if (p.causal) {
    const int lim = q0 + 127 + p.Sk - p.Sq;
    nT = lim < 0 ? 0 : min(nkt, lim / 128 + 1);
  }

  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = bars + 1 + C::NS;
  uint64_t* pv_done = bars + 1 + 2 * C::NS;     // PV(j) -> slot j % NS
  uint64_t* k_empty = bars + 1 + 3 * C::NS;    // S(j) done -> K slot j % NS
  uint64_t* s_full = bars + 1 + 4 * C::NS;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;               // P~(j) written -> barrier j % NPB
  uint64_t* drain = p_full + C::NPB;
  uint64_t* stall = drain + 1;
  uint64_t* qraw_full = drain + 2;              // QF: the bf16 Q tile landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 8);
  float* red = reinterpret_cast<float*>(sm + C::OFF_RED);

  if (threadIdx.x == 0) {
    mbar_init(q_full, QF ? 8 : 1);                // QF: one arrival per softmax warp
    if constexpr (QF) mbar_init(qraw_full, 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(k_full + i, 1); mbar_init(v_full + i, 1); mbar_init(pv_done + i, 1); mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      // one softmax warp per lane quadrant owns each tile
      mbar_init(s_full + i, 1); mbar_init(s_free + i, 4);
    }
    for (int i = 0; i < C::NPB; ++i) mbar_init(p_full + i, 4);
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    sts_vol(abort_flag, 0);
    fence_mbar_init();
    if (nT > 0) {
      // the first loads overlap the rest of the setup (tensor memory, constant rows)
      const int bhq = b * p.H + h, bhk = b * p.Hkv + kvh;
      if constexpr (QF) {
        mbar_expect_tx(qraw_full, 128 * D * 2);
        tma_load_3d(sm + C::OFF_QRAW, &tm_q, qraw_full, 0, q0, bhq);
      } else {
        mbar_expect_tx(q_full, C::TILE_QK + (MX ? C::SFQK : 0));
#pragma unroll
        for (int ka = 0; ka < C::NKA_QK; ++ka)
          tma_load_3d(sQ + ka * 128 * C::W_QK, &tm_q, q_full, ka * C::W_QK, q0, bhq);
        if (MX) bulk_load(sm + C::OFF_SFQ, p.sf_q + ((size_t)bhq * p.n_qtiles + qt) * C::SFQK, C::SFQK, q_full);
      }
      for (int j = 0; j < C::NS && j < nT; ++j) {
        mbar_expect_tx(k_full + j, C::TILE_QK + (MX ? C::SFQK : 0));
#pragma unroll
        for (int ka = 0; ka < C::NKA_QK; ++ka)
          tma_load_3d(sK + j * C::TILE_QK + ka * 128 * C::W_QK, &tm_k, k_full + j, ka * C::W_QK, j * 128, bhk);
        if (MX)
          bulk_load(sm + C::OFF_SFK + j * C::SFQK, p.sf_k + ((size_t)bhk * nkt + j) * C::SFQK, C::SFQK, k_full + j);
        mbar_expect_tx(v_full + j, C::TILE_V_TMA + (MX ? 512 : 0));
#pragma unroll
        for (int ka = 0; ka < C::NKA_V; ++ka)
          tma_load_3d(sV + j * C::TILE_V + ka * C::VATOM, &tm_v, v_full + j, j * C::RB_V + ka * C::W_V, 0, bhk);
        if (MX) bulk_load(sm + C::OFF_SFV + j * 512, p.sf_v + ((size_t)bhk * nkt + j) * 512, 512, v_full + j);
      }
    }
  }
  if (MX && warp >= 2) {
    // constant rows D..D+15 of every V stage (row D = ones, the rest zero) and the
    // scale atom that gives the ones row scale 2^0 in the upper tensor-memory columns
    const int t = threadIdx.x - 64;
    uint32_t one4;
    if constexpr (FPV == F_BF16) one4 = 0x3F803F80u;
    else if constexpr (FPV == F_E4M3) one4 = 0x38383838u;
    else if constexpr (FPV == F_E2M3 || FPV == F_E3M2) one4 = 0u;   // set per word below (packed 6-bit)
    else one4 = 0x22222222u;
    constexpr int ROWW = C::W_V / 4;                 // words per row per atom
    constexpr int PER_STAGE = C::NKA_V * 16 * ROWW;
    for (int i = t; i < C::NS * PER_STAGE; i += C::NTHREADS - 64) {
      const int st = i / PER_STAGE, rem = i % PER_STAGE;
      const int ka = rem / (16 * ROWW), r = (rem / ROWW) % 16, w = rem % ROWW;
      uint32_t val = 0u;
      if (r == 0) {
        if constexpr (FPV == F_E2M3) {
          const int wg = w & 3;                      // 16-byte group: bytes (08 82 20) x 4, then 4 zero bytes
          val = wg == 0 ? 0x08208208u : (wg == 1 ? 0x82082082u : (wg == 2 ? 0x20820820u : 0u));
        } else if constexpr (FPV == F_E3M2) {
          const int wg = w & 3;                      // 1.0 = code 0x0C: bytes (0C C3 30) x 4, then 4 zero bytes
          val = wg == 0 ? 0x0C30C30Cu : (wg == 1 ? 0xC30C30C3u : (wg == 2 ? 0x30C30C30u : 0u));
        } else {
          val = one4;
        }
      }
      uint32_t* dst = reinterpret_cast<uint32_t*>(sV + st * C::TILE_V + ka * C::VATOM + (D + r) * C::W_V);
      dst[w] = val;
    }
    if (MX) {
      uint32_t* one_atom = reinterpret_cast<uint32_t*>(sm + C::OFF_SFONE);
      for (int i = t; i < 128; i += C::NTHREADS - 64) one_atom[i] = 0x7F7F7F7Fu;
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  const AbortCtl ac{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // =============================================================== producer
    // Lane 0 loads Q and the K tiles, lane 1 the V tiles: a K tile waits only for
    // its own ring slot, never behind a V slot that a late PV still holds.
    if (lane < 2 && nT > 0) {
      const int bhk = b * p.Hkv + kvh;
      if (lane == 0) {
        // K(j) as soon as K slot j % NS is free (S(j - NS) done); Q and the first
        // NS tiles were requested during the setup
        int nk = min(C::NS, nT);
        for (int j = nk; j < nT; ++j) {
          const int st = j % C::NS;
          if (j >= C::NS && !mbar_wait(k_empty + st, ((j - C::NS) / C::NS) & 1, ac)) break;
          mbar_expect_tx(k_full + st, C::TILE_QK + (MX ? C::SFQK : 0));
#pragma unroll
          for (int ka = 0; ka < C::NKA_QK; ++ka)
            tma_load_3d(sK + st * C::TILE_QK + ka * 128 * C::W_QK, &tm_k, k_full + st, ka * C::W_QK, j * 128, bhk);
          if (MX)
            bulk_load(sm + C::OFF_SFK + st * C::SFQK, p.sf_k + ((size_t)bhk * nkt + j) * C::SFQK, C::SFQK,
                      k_full + st);
          ++nk;
        }
        mbar_drain(QF ? qraw_full : q_full, 0, ac);
        for (int st = 0; st < C::NS && st < nk; ++st)
          mbar_drain(k_full + st, ((nk - 1 - st) / C::NS) & 1, ac);
      } else {
        // V(j) as soon as V slot j % NS is free (PV(j - NS) done)
        int nv = min(C::NS, nT);
        for (int j = nv; j < nT; ++j) {
          const int st = j % C::NS;
          if (j >= C::NS && !mbar_wait(pv_done + st, ((j - C::NS) / C::NS) & 1, ac)) break;
          mbar_expect_tx(v_full + st, C::TILE_V_TMA + (MX ? 512 : 0));
#pragma unroll
          for (int ka = 0; ka < C::NKA_V; ++ka)
            tma_load_3d(sV + st * C::TILE_V + ka * C::VATOM, &tm_v, v_full + st, j * C::RB_V + ka * C::W_V, 0, bhk);
          if (MX) bulk_load(sm + C::OFF_SFV + st * 512, p.sf_v + ((size_t)bhk * nkt + j) * 512, 512, v_full + st);
          ++nv;
        }
        for (int st = 0; st < C::NS && st < nv; ++st)
          mbar_drain(v_full + st, ((nv - 1 - st) / C::NS) & 1, ac);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // =============================================================== MMA issuer
    // The warp runs converged; lane 0 polls the barriers and every tcgen05
    // instruction is issued by the elected lane (the same lane throughout, so its
    // commits cover all of them).  One warp issues both GEMMs: tcgen05 work from two
    // issuing warps of one CTA was measured to serialise badly.
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, ac));
    };
    if (nT > 0) {
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      constexpr uint32_t SWQ = swz_code(C::W_QK), SWV = swz_code(C::W_V);
      bool ok = true;
      if (p.inject_stall) ok = __all_sync(0xffffffffu, mbar_wait(stall, 0, ac));   // nobody arrives: must expire
      ok = ok && wait_all(q_full, 0);
      if (ok) {
        tc_fence_after();
        if constexpr (MX) {
#pragma unroll
          for (int a = 0; a < C::NATOM_QK; ++a)      // NVFP4: one atom per K = 64 step
            tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFQ + 4 * a,
                            smem_desc(smem_u32(sm + C::OFF_SFQ + 512 * a), 16, 128, 0));
          if constexpr (D == 128) {
            const uint64_t one = smem_desc(smem_u32(sm + C::OFF_SFONE), 16, 128, 0);
            tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFV + 4, one);
            tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFV + 12, one);
          }
        }
      }
      auto issue_pv = [&](int jj) {
        const int s = jj & 1, st = jj % C::NS;
        tc_fence_after();
        if constexpr (MX) {
          const uint64_t sfd = smem_desc(smem_u32(sm + C::OFF_SFV + st * 512), 16, 128, 0);
          tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFV + 8 * s, sfd);
        }
#pragma unroll
        for (int i = 0; i < C::PV_STEPS; ++i) {
          // P~ of step i sits in columns [8i, 8i+8) of its P buffer; the scale word of
          // each row (byte b = 32-key block b) is in column T_SFP + 4 (buffer) + lane quadrant
          const uint32_t a_tm = tbase + C::T_P + C::P_COLS * ((unsigned)jj % C::NPB) + 8 * i;
          const uint32_t sfa = tbase + C::T_SFP + 4 * ((unsigned)jj % C::NPB);
          const int ka = (i * 32) / C::W_V, off = (i * 32) % C::W_V;
          const uint64_t bd = smem_desc(sVa + st * C::TILE_V + ka * C::VATOM + off, 16, 8 * C::W_V, SWV);
          const uint32_t acc = (jj > 0 || i > 0) ? 1u : 0u;
          const uint32_t e = elect_u32();
          if constexpr (KIND_PV == 0) {
            mma_f16_ts_p(e, tbase + C::T_O, a_tm, bd, idesc_f16_bf16(C::N_PV), acc);
          } else if constexpr (KIND_PV == 1) {
            mma_mxf8f6f4_ts_p(e, tbase + C::T_O, a_tm, bd, idesc_bs(C::N_PV, Fmt<FPV>::code, i, i), sfa,
                              tbase + C::T_SFV + 8 * s, acc);
          } else {
            mma_mxf4_ts_p(e, tbase + C::T_O, a_tm, bd, idesc_bs(C::N_PV, 1, 2 * i, 2 * i), sfa,
                          tbase + C::T_SFV + 8 * s, acc);
          }
        }
        tc_commit_p(elect_u32(), pv_done + st);
      };
      auto issue_s = [&](int j) {
        const int s = j & 1, st = j % C::NS;
        tc_fence_after();
        if constexpr (MX) {
#pragma unroll
          for (int a = 0; a < C::NATOM_QK; ++a) {
            const uint64_t sfd = smem_desc(smem_u32(sm + C::OFF_SFK + st * C::SFQK + 512 * a), 16, 128, 0);
            tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFK + C::SFK_STEP * s + 4 * a, sfd);
          }
        }
#pragma unroll
        for (int i = 0; i < C::QK_STEPS; ++i) {
          const int ka = (i * 32) / C::W_QK, off = (i * 32) % C::W_QK;
          const uint64_t ad = smem_desc(sQa + ka * 128 * C::W_QK + off, 16, 8 * C::W_QK, SWQ);
          const uint64_t bd = smem_desc(sKa + st * C::TILE_QK + ka * 128 * C::W_QK + off, 16, 8 * C::W_QK, SWQ);
          const uint32_t acc = i > 0 ? 1u : 0u;
          const uint32_t e = elect_u32();
          if constexpr (KIND_QK == 0) {
            mma_f16_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_f16_bf16(128), acc);
          } else if constexpr (KIND_QK == 1) {
            mma_mxf8f6f4_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_bs(128, Fmt<FQK>::code, i, i),
                              tbase + C::T_SFQ, tbase + C::T_SFK + C::SFK_STEP * s, acc);
          } else if constexpr (KIND_QK == 2) {
            mma_mxf4_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_bs(128, 1, 2 * i, 2 * i),
                          tbase + C::T_SFQ, tbase + C::T_SFK + C::SFK_STEP * s, acc);
          } else {
            // NVFP4: step i reads the whole scale word of atom i (16 elements a byte)
            mma_nvf4_4x_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_nvfp4(128), tbase + C::T_SFQ + 4 * i,
                             tbase + C::T_SFK + C::SFK_STEP * s + 4 * i, acc);
          }
        }
        tc_commit_p(elect_u32(), s_full + s);
        tc_commit_p(elect_u32(), k_empty + st);
      };
      // Fixed order: QK^T(0), QK^T(1), then for each key tile j QK^T(j+2) -- once the
      // owners of tile j have loaded S(j), which frees its S buffer, and K(j+2) has
      // landed -- and PV(j), once P~(j) is written and V(j) has landed.  The owners
      // release S(j) early in tile j and write P~(j) at its end, so each wait is on
      // the event that comes next, and the warp sleeps in it until the phase
      // completes: PV(j) is issued as soon as its operands are there.
      auto qk_ready = [&](int jj) -> bool {
        return wait_all(k_full + jj % C::NS, (jj / C::NS) & 1) &&
               (jj < 2 || wait_all(s_free + (jj & 1), ((jj - 2) >> 1) & 1));
      };
      for (int jj = 0; ok && jj < 2 && jj < nT; ++jj) {
        ok = qk_ready(jj);
        if (ok) issue_s(jj);
      }
      for (int j = 0; ok && j < nT; ++j) {
        if (j + 2 < nT) {
          ok = qk_ready(j + 2);
          if (!ok) break;
          issue_s(j + 2);
        }
        // V(j) landed long before P~(j) is written: test it first, so that the warp
        // wakes from the P~ wait straight into the issue
        ok = wait_all(v_full + j % C::NS, (j / C::NS) & 1) && wait_all(p_full + (unsigned)j % C::NPB, ((unsigned)j / C::NPB) & 1);
        if (ok) issue_pv(j);
      }
      // all MMAs and copies issued by this warp complete before tensor memory is freed
      tc_commit_p(elect_u32(), drain);
      mbar_drain(drain, 0, ac);
    }
    __syncwarp();
  } else {
    // =============================================================== softmax / epilogue
    // The two warps of a tensor-memory lane quadrant take alternate key tiles: part pp
    // owns the tiles j with j % 2 == pp, all 128 keys of its 32 rows (thread = row),
    // and with them S buffer, P~ buffer and scale column pp.  The running maximum M
    // passes between the two once per tile (shared memory plus a named-barrier
    // handoff), so they work half a tile apart instead of in lockstep.
    constexpr int NBLK = 4;                         // 32-key blocks per tile
    const int pp = (warp - 2) >> 2;
    const int qd = warp & 3;                        // tensor-memory lane quadrant
    const int rl = 32 * qd + lane;                  // row within the tile
    const int row = q0 + rl;
    const bool row_valid = row < p.Sq;
    // debug dumps: this row's slot (negative: not dumped)
    long long dbg_row = -1;
    if constexpr (DBG) {
      if (row_valid) {
        const long long grow = ((long long)b * p.H + h) * p.Sq + row;
        dbg_row = dbg.row_slot ? (long long)dbg.row_slot[grow] : grow;
      }
    }
    const bool dbg_on = DBG && dbg_row >= 0;
    const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16);
    int lim = p.Sk - 1;
    if (p.causal) lim = min(lim, row + p.Sk - p.Sq);
    const float c = p.c;
    const int bar_in = 1 + qd + 4 * pp, bar_out = 1 + qd + 4 * (1 - pp);
    float* m_slot = red + rl;                       // M of this row after the latest tile
    float M = kNegInf;
    int nfb = 0, nvis = 0;
    bool ok = true;                                 // false once any wait failed: no more work
    // BF16: the denominator is summed here, per part, relative to the part's latest M
    float lsum = 0.0f, Ml = kNegInf;
    // every lane polls; the vote keeps the warp uniform.  The common case (phase
    // already complete) is one try_wait per lane and one vote, with no loop
    auto wait0 = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
      return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, ac));
    };
    if constexpr (QF) {
      // the bf16 Q tile -> MX codes and scale atom, then the MMA warp may read them
      if (nT > 0) {
        if (wait0(qraw_full, 0)) {
          quantize_q_tile<FQK, D>(sm + C::OFF_QRAW, sQ, sm + C::OFF_SFQ, (int)threadIdx.x - 64);
          fence_proxy_async_smem();
          __syncwarp();
          mbar_arrive_elect(q_full);
        } else {
          ok = false;
        }
      }
    }
    for (int j = pp; j < nT; j += 2) {
      const int s = pp;
      const bool got = ok && wait0(s_full + s, (j >> 1) & 1);
      if (!got) ok = false;
      float sv[128];
      float bm[NBLK];
#pragma unroll
      for (int b = 0; b < NBLK; ++b) bm[b] = kNegInf;
      if (got) {
        tc_fence_after();
        uint32_t raw[128];
        float bmr[NBLK];                              // block maxima, from the load itself
#pragma unroll
        for (int b = 0; b < NBLK; ++b) tmem_ld32_max(tl + C::T_S + 128 * s + 32 * b, raw + 32 * b, bmr[b]);
        tc_wait_ld();
        // S(j) is in registers: its buffer may take S(j+2)
        tc_fence_before();
        __syncwarp();
        mbar_arrive_elect(s_free + s);
#pragma unroll
        for (int i = 0; i < 128; ++i) sv[i] = __uint_as_float(raw[i]);
        // only diagonal / tail tiles mask keys; the branch is taken by the whole warp
        // (rows that need no mask compare and keep every key), which keeps the masking
        // off the path of the other tiles
        if (__any_sync(0xffffffffu, 128 * j + 127 > lim)) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (128 * j + i > lim) sv[i] = kNegInf;
#pragma unroll
          for (int b = 0; b < NBLK; ++b) bm[b] = max32(sv + 32 * b);
        } else {
#pragma unroll
          for (int b = 0; b < NBLK; ++b) bm[b] = bmr[b];
        }
        if constexpr (DBG) {
          if (dbg_on) {
            float4* ds = reinterpret_cast<float4*>(dbg.s + dbg_row * nkt * 128 + 128 * j);
#pragma unroll
            for (int i = 0; i < 32; ++i) ds[i] = make_float4(sv[4 * i], sv[4 * i + 1], sv[4 * i + 2], sv[4 * i + 3]);
          }
        }
      }
      // M after tile j-1 comes from the other part (NaN: it has stopped working)
      if (j > 0) {
        named_bar_sync(bar_in, 64);
        const float Mp = lds_f32(m_slot);
        if (isnan(Mp)) ok = false;
        else M = Mp;
      }
      // first visible tile: M = x; later: fallback when x > fp32(M + delta)
      const float hm = fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3]));
      if (128 * j <= lim) ++nvis;
      bool rescale = false;
      float Mn = M;
      if (ok && hm != kNegInf) {
        const float x = __fmul_rn(hm, c);
        if (M == kNegInf) {
          Mn = x;
        } else if (MX ? (x > __fadd_rn(M, p.delta)) : (__fsub_rn(x, M) > 8.0f)) {
          rescale = true;
          Mn = x;
        }
      }
      if (j + 1 < nT) {
        sts_f32(m_slot, ok ? Mn : __int_as_float(0x7FC00000));
        named_bar_arrive(bar_out, 64);
      }
      const float alpha = rescale ? ex2_approx(__fsub_rn(M, Mn)) : 1.0f;
      if (rescale) ++nfb;
      M = Mn;
      if constexpr (DBG) {
        if (ok && dbg_on) dbg.m[dbg_row * nkt + j] = M;
      }
      if constexpr (!MX) {
        if (Ml != kNegInf && M != Ml) lsum *= ex2_approx(__fsub_rn(Ml, M));
        Ml = M;
      }
      if (ok) {
        // ---- P~ of the tile in two halves of two 32-key blocks.  The first half is
        // generated before waiting for the PVs that the rescale and the buffer reuse
        // depend on, which gives them that much longer to finish.
        constexpr int HW = C::P_COLS / 2;             // words (columns) per half
        const uint32_t tp = tl + C::T_P + C::P_COLS * ((unsigned)j % C::NPB);
        uint32_t sw = 0;                            // the blocks' scale bytes, block b in byte b
        // EFQ: the blocks' scale words, gathered by byte permutes (one instruction fewer
        // per block; the exp paths keep the shifts, which measured faster there)
        uint32_t swb[NBLK] = {};
        uint64_t acc = pk2(0.0f, 0.0f);               // BF16: sum of the rounded p
        const float nM = M == kNegInf ? 0.0f : -M;    // BF16, no visible key yet: every s is -inf, p = 0
        auto gen_half = [&](int hf, uint32_t* pw) {
          if constexpr (MX) {
            constexpr int WB = C::P_COLS / NBLK;       // words per block: 8, or 4 for E2M1
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              const uint32_t w = pgen_block<FPV, EXPM>(sv + 64 * hf + 32 * b, bm[2 * hf + b], c, M, p, pw + WB * b);
              if constexpr (FPV == F_EFQ) swb[2 * hf + b] = w;
              else sw |= (w & 0xFFu) << (8 * (2 * hf + b));
            }
          } else {
            const uint64_t c2 = pk2(c, c), nM2 = pk2(nM, nM);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float a, bb;
              upk2(ffma2(pk2(sv[64 * hf + 2 * i], sv[64 * hf + 2 * i + 1]), c2, nM2), a, bb);
              pw[i] = cvt_bf16x2(ex2_approx(a), ex2_approx(bb));
              // the denominator sums the rounded p that the PV MMA multiplies
              acc = fadd2(acc, pk2(__uint_as_float(pw[i] << 16), __uint_as_float(pw[i] & 0xFFFF0000u)));
            }
          }
        };
        auto dbg_words = [&](int hf, const uint32_t* pw) {
          if constexpr (DBG) {
            if (dbg_on) {
#pragma unroll
              for (int w = 0; w < HW; ++w) dbg.p[(dbg_row * nkt + j) * 32 + HW * hf + w] = pw[w];
            }
          }
        };
        uint32_t pw[HW];
        if constexpr (MX) {
          gen_half(0, pw);                           // (BF16: too many registers to hold across)
          dbg_words(0, pw);
        }
        // fallback: O_aug row *= 2^(M_old - M) once PV(j-1) has landed.  tcgen05.ld/st
        // are warp-collective, so the whole warp rescales when any of its rows falls
        // back; the other rows multiply by exactly 1.
        if (__any_sync(0xffffffffu, rescale)) {
          // PV(j-NPB) first: with two PV barriers (BF16) PV(j-1) shares its barrier with
          // PV(j-3), and its parity only identifies PV(j-1) once PV(j-3) has completed
          const bool prev = j < C::NPB || wait0(pv_done + (j - C::NPB) % C::NS, ((j - C::NPB) / C::NS) & 1);
          if (prev && wait0(pv_done + (j - 1) % C::NS, ((j - 1) / C::NS) & 1)) {
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < C::N_PV; c0 += 8) {
              uint32_t o[8];
              TmemLd<8>::run(tl + C::T_O + c0, o);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__fmul_rn(__uint_as_float(o[i]), alpha));
              TmemSt<8>::run(tl + C::T_O + c0, o);
            }
            tc_wait_st();
          } else {
            ok = false;
          }
        }
        // P~ buffer j % NPB and its scale column were last read by PV(j - NPB): with two
        // buffers wait for it; with more it completed before S(j) was signalled
        if constexpr (C::NPB < 3) {
          if (ok && j >= C::NPB && !wait0(pv_done + (j - C::NPB) % C::NS, ((j - C::NPB) / C::NS) & 1)) ok = false;
        }
        if (ok) {
          tc_fence_after();
          if constexpr (!MX) gen_half(0, pw);
          tmem_st_cols<HW>(tp, pw);
          gen_half(1, pw);
          dbg_words(1, pw);
          tmem_st_cols<HW>(tp + HW, pw);
          // A scales of the PV MMA: lane quadrant q reads column base + q
          if constexpr (FPV == F_EFQ) sw = low_bytes4(swb[0], swb[1], swb[2], swb[3]);
          if constexpr (MX) TmemSt<1>::run(tl + C::T_SFP + 4 * ((unsigned)j % C::NPB) + qd, &sw);
          if constexpr (DBG) {
            if (dbg_on) dbg.sf[dbg_row * nkt + j] = sw;
          }
          if constexpr (!MX) {
            float a0, a1;
            upk2(acc, a0, a1);
            lsum += a0 + a1;
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (ok) mbar_arrive_elect(p_full + (unsigned)j % C::NPB);
      }
    }
    // ---- epilogue: O = O_aug[:, :D] / l, D/2 columns per part
    constexpr int DP = D / 2;
    float lb = 0.0f;                                 // BF16: l of the row from both parts
    if constexpr (!MX) {
      float* xl = red + 256 + 4 * rl;                // [row] {l, M} of each part
      xl[2 * pp] = lsum;
      xl[2 * pp + 1] = Ml;
      named_bar_sync(9 + qd, 64);
      const float l0 = xl[0], m0 = xl[1], l1 = xl[2], m1 = xl[3];
      const float mf = fmaxf(m0, m1);
      lb = (m0 != kNegInf ? l0 * ex2_approx(__fsub_rn(m0, mf)) : 0.0f) +
           (m1 != kNegInf ? l1 * ex2_approx(__fsub_rn(m1, mf)) : 0.0f);
      named_bar_sync(9 + qd, 64);                    // both have read before the slots are reused
    }
    // O rows go out through shared memory and TMA: each warp writes its 32 rows x DP
    // columns as 32x32 fp32 boxes (128B swizzle) into the K/V ring, which no copy or
    // MMA uses any more, and one lane stores them (rows past Sq are clipped).
    constexpr int NBOX = DP / 32;                    // boxes per warp
    // PV(nT-2) before PV(nT-1), for the same parity reason as the rescale wait
    const bool done = ok && nT > 0 && (nT < 2 || wait0(pv_done + (nT - 2) % C::NS, ((nT - 2) / C::NS) & 1)) &&
                      wait0(pv_done + (nT - 1) % C::NS, ((nT - 1) / C::NS) & 1);
    if (done || nT == 0) {
      uint32_t o[DP];
      float l = 0.f;
      if (done) {
        tc_fence_after();
        uint32_t lraw = 0;
        if constexpr (MX) TmemLd<1>::run(tl + C::T_O + D, &lraw);
        tmem_ld_cols<DP>(tl + C::T_O + DP * pp, o);
        tc_wait_ld();
        l = MX ? __uint_as_float(lraw) : lb;
      }
      // fp32 normalisation: one correctly rounded reciprocal of l per row, then products
      // (within 1.5 ulp of the quotient).  A row with no visible key has l = 0 (or
      // NaN: its residuals are -inf + inf) and gets zeros.
      const bool lpos = l > 0.f;
      const float rinv = lpos ? __frcp_rn(l) : 0.f;
      fence_proxy_async_smem();                      // the ring was last written by TMA loads
      if (p.out_bf16) {
        // bf16 output: the same fp32 quotients rounded to nearest even, one box of 32
        // rows x DP bf16 per warp (128B swizzle for 128-byte rows, else 64B)
        uint8_t* box = sm + C::OFF_OSTAGE + (qd * 2 + pp) * 4096;
        auto qv = [&](uint32_t x) { return lpos ? __fmul_rn(__uint_as_float(x), rinv) : 0.f; };
#pragma unroll
        for (int ch = 0; ch < DP / 8; ++ch) {
          const uint32_t* src = o + 8 * ch;
          uint4 wv;
          wv.x = cvt_bf16x2(qv(src[0]), qv(src[1]));
          wv.y = cvt_bf16x2(qv(src[2]), qv(src[3]));
          wv.z = cvt_bf16x2(qv(src[4]), qv(src[5]));
          wv.w = cvt_bf16x2(qv(src[6]), qv(src[7]));
          const int off = DP == 64 ? lane * 128 + ((ch ^ (lane & 7)) << 4) : lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4);
          *reinterpret_cast<uint4*>(box + off) = wv;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_o, box, DP * pp, q0 + 32 * qd, b * p.H + h);
          bulk_commit_group();
          bulk_wait_all();
        }
        __syncwarp();
      } else {
#pragma unroll
      for (int t = 0; t < NBOX; ++t) {
        uint8_t* box = sm + C::OFF_OSTAGE + (qd * (D / 32) + (DP * pp) / 32 + t) * 4096;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float4 v;
          const uint32_t* src = o + 32 * t + 4 * ch;
          v.x = lpos ? __fmul_rn(__uint_as_float(src[0]), rinv) : 0.f;
          v.y = lpos ? __fmul_rn(__uint_as_float(src[1]), rinv) : 0.f;
          v.z = lpos ? __fmul_rn(__uint_as_float(src[2]), rinv) : 0.f;
          v.w = lpos ? __fmul_rn(__uint_as_float(src[3]), rinv) : 0.f;
          // 128B swizzle: 16-byte chunk ch of row `lane` sits at chunk ch ^ (lane % 8)
          *reinterpret_cast<float4*>(box + lane * 128 + ((ch ^ (lane & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();                      // generic writes -> TMA reads
      __syncwarp();
      if (lane == 0) {
        const int bh = b * p.H + h;
#pragma unroll
        for (int t = 0; t < NBOX; ++t)
          tma_store_3d(&tm_o, sm + C::OFF_OSTAGE + (qd * (D / 32) + (DP * pp) / 32 + t) * 4096,
                       DP * pp + 32 * t, q0 + 32 * qd, bh);
        bulk_commit_group();
        bulk_wait_all();                             // before the CTA (and its shared memory) ends
      }
      __syncwarp();
      }
    }
    // ---- statistics: each part counted the tiles it owns
    int* nfb_other = reinterpret_cast<int*>(red) + 128 + rl;
    if (pp == 1) *nfb_other = nfb;
    named_bar_sync(9 + qd, 64);
    if (pp == 0 && row_valid && p.row_fallbacks)
      p.row_fallbacks[((size_t)b * p.H + h) * p.Sq + row] = nfb + *nfb_other;
    unsigned long long f = row_valid ? (unsigned long long)nfb : 0ull;
    unsigned long long v = row_valid ? (unsigned long long)nvis : 0ull;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      f += __shfl_xor_sync(0xffffffffu, f, o2);
      v += __shfl_xor_sync(0xffffffffu, v, o2);
    }
    if (lane == 0 && p.stat_fallbacks) {
      atomicAdd(p.stat_fallbacks, f);
      atomicAdd(p.stat_row_tiles, v);
    }
  }
  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace fsa

#include "fsa_attn_persistent.cuh"

namespace fsa {

// ----------------------------------------------------------------------------- host launch
template <int FQK, int FPV, int D, int EXPM, bool DBG = false, bool QF = false>
static cudaError_t launch_one(const AttnLaunch& a) {
  using C = Cfg<FQK, FPV, D, false, QF>;
  // at least 116 KB so that one CTA (and its 512 tensor-memory columns) owns an SM
  constexpr int smem = (C::SMEM > 116 * 1024 ? C::SMEM : 116 * 1024);
  auto kern = fsa_attn_kernel<FQK, FPV, D, EXPM, DBG, QF>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid = a.p.causal ? dim3((a.p.H / a.p.Hkv) * a.p.n_qtiles, a.p.Hkv * a.p.B, 1)
                               : dim3(a.p.n_qtiles, a.p.H, a.p.B);
  kern<<<grid, C::NTHREADS, smem, a.stream>>>(a.tq, a.tk, a.tv, a.to, a.p, a.dbg);
  return cudaGetLastError();
}

// Persistent schedule: one CTA per SM (no more CTAs than query tiles), enough CTAs
// that none takes more than MAX_ITEMS query tiles.
template <int FQK, int FPV, int D, int EXPM>
static cudaError_t launch_persistent(const AttnLaunch& a) {
  using C = Cfg<FQK, FPV, D, true>;
  constexpr int smem = (C::SMEM > 116 * 1024 ? C::SMEM : 116 * 1024);
  auto kern = fsa_attn_persistent_kernel<FQK, FPV, D, EXPM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  int grid = a.p.n_items < n_sm ? a.p.n_items : n_sm;
  const int need = (a.p.n_items + C::MAX_ITEMS - 1) / C::MAX_ITEMS;
  if (grid < need) grid = need;
  if (grid == 0) return cudaSuccess;
  kern<<<grid, C::NTHREADS, smem, a.stream>>>(a.tq, a.tk, a.tv, a.to, a.p);
  return cudaGetLastError();
}

// The debug instance exists for every MX format pair with the cubic or the hardware
// exp2, under the per-query-tile schedule.
template <int FQK, int FPV>
constexpr bool kHasDebug = FQK != F_BF16;

template <int FQK, int FPV, int D, int EXPM>
static cudaError_t launch_sched(const AttnLaunch& a) {
  if (a.debug) {
    if constexpr (kHasDebug<FQK, FPV> && EXPM < 2) return launch_one<FQK, FPV, D, EXPM, true>(a);
    return cudaErrorNotSupported;
  }
  // Q quantised in the prologue: the library's default exp2 path (and EFQ), one CTA
  // per query tile
  if (a.q_fused) {
    if constexpr ((EXPM == 1 || FPV == F_EFQ) && FQK != F_BF16 && FQK != F_NVFP4)
      return launch_one<FQK, FPV, D, EXPM, false, true>(a);
    return cudaErrorNotSupported;
  }
  // NVFP4 Q/K: one CTA per query tile only
  if constexpr (FQK == F_NVFP4) return a.persistent ? cudaErrorNotSupported : launch_one<FQK, FPV, D, EXPM>(a);
  else return a.persistent ? launch_persistent<FQK, FPV, D, EXPM>(a) : launch_one<FQK, FPV, D, EXPM>(a);
}

// The exp-mode slot: 0/1/2 the exp2 path of the exp-then-round formats; for EFQ 1
// when the codes need no fix (see pgen_block), else 0; BF16 has one path.
template <int FQK, int FPV>
cudaError_t launch_attn_impl(const AttnLaunch& a) {
  if constexpr (FPV == F_BF16) {
    return a.D == 64 ? launch_sched<FQK, FPV, 64, 1>(a) : launch_sched<FQK, FPV, 128, 1>(a);
  } else if constexpr (FPV == F_EFQ) {
    if (a.D == 64) return a.exp_mode == 1 ? launch_sched<FQK, FPV, 64, 1>(a) : launch_sched<FQK, FPV, 64, 0>(a);
    return a.exp_mode == 1 ? launch_sched<FQK, FPV, 128, 1>(a) : launch_sched<FQK, FPV, 128, 0>(a);
  } else {
    if (a.D == 64) {
      if (a.exp_mode == 0) return launch_sched<FQK, FPV, 64, 0>(a);
      if (a.exp_mode == 1) return launch_sched<FQK, FPV, 64, 1>(a);
      return launch_sched<FQK, FPV, 64, 2>(a);
    }
    if (a.exp_mode == 0) return launch_sched<FQK, FPV, 128, 0>(a);
    if (a.exp_mode == 1) return launch_sched<FQK, FPV, 128, 1>(a);
    return launch_sched<FQK, FPV, 128, 2>(a);
  }
}

}  // namespace fsa

#if defined(FSA_INST_QK) && defined(FSA_INST_PV)
template cudaError_t fsa::launch_attn_impl<FSA_INST_QK, FSA_INST_PV>(const fsa::AttnLaunch&);
#endif
