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
// TMA loads, warp 1 (one thread) issues tcgen05 MMAs and owns tensor memory,
// warps 2..9 are two softmax warpgroups that split each key tile into halves
// of 64 keys (thread = one row, one half).  S is double buffered in tensor
// memory; P~ overwrites the consumed half of S and is read by the PV MMA
// straight from tensor memory; O_aug stays in tensor memory until the end.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "fsa_launch.h"

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
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Exponent-only block scale: E = clamp(floor(fp32(fp32(smax*c) - M)) - emax, -127, 127).
// Returns E and writes -fp32(M + E).  A block with no visible key (smax = -inf)
// gets E = -127; its scores are -inf, so every code comes out 0.
template <int FPV>
__device__ __forceinline__ int block_exp(float bmax, float c, float M, float& nbE) {
  const float tmax = __fsub_rn(__fmul_rn(bmax, c), M);
  int E = (int)fmaxf(floorf(tmax), -256.0f) - Fmt<FPV>::emax;
  E = E < -127 ? -127 : (E > 127 ? 127 : E);
  nbE = -__fadd_rn(M, (float)E);
  return E;
}

// P codes of one 64-key half tile (raw scores sv[0..63] as two 32-key blocks,
// masked = -inf) as packed words in out[] (16 words for one byte per code, 8 for
// E2M1).  Returns the two scale bytes (block 0 in the low byte).
template <int FPV, int EXPM>
__device__ __forceinline__ uint32_t pgen_half(const float* sv, float bm0, float bm1, float c, float M, int beta,
                                              uint32_t* out) {
  float nb0, nb1;
  const int E0 = block_exp<FPV>(bm0, c, M, nb0);
  const int E1 = block_exp<FPV>(bm1, c, M, nb1);
  const uint64_t c2 = pk2(c, c), n0 = pk2(nb0, nb0), n1 = pk2(nb1, nb1);
  float r[64];
#pragma unroll
  for (int i = 0; i < 64; i += 2) upk2(ffma2(pk2(sv[i], sv[i + 1]), c2, i < 32 ? n0 : n1), r[i], r[i + 1]);
  if constexpr (FPV == F_EFQ) {
    // k = clamp(rne(2 r + beta), 0, 7): fma onto the integer grid of 1.5*2^23, whose
    // low bits then hold k; nibble pairs combine by shift-add, bytes merge by permute
    const float magic = 12582912.0f;
    const uint64_t two2 = pk2(2.0f, 2.0f), kb2 = pk2(magic + (float)beta, magic + (float)beta);
    uint32_t y[64];
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      float y0, y1;
      upk2(ffma2(two2, pk2(r[i], r[i + 1]), kb2), y0, y1);
      y[i] = __float_as_uint(fminf(fmaxf(y0, magic), magic + 7.0f));
      y[i + 1] = __float_as_uint(fminf(fmaxf(y1, magic), magic + 7.0f));
    }
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t* t = y + 8 * w;
      // low byte of (t1 << 4) + t0 is k0 | k1 << 4 (the magic's bits stay above bit 21)
      const uint32_t a01 = (t[1] << 4) + t[0], a23 = (t[3] << 4) + t[2];
      const uint32_t a45 = (t[5] << 4) + t[4], a67 = (t[7] << 4) + t[6];
      out[w] = prmt(prmt(a01, a23, 0x0040u), prmt(a45, a67, 0x0040u), 0x5410u);
    }
  } else {
    exp2_block<EXPM>(r);
    exp2_block<EXPM>(r + 32);
    if constexpr (FPV == F_E4M3) {
#pragma unroll
      for (int w = 0; w < 16; ++w)
        out[w] = pack_b16x2(cvt16_e4m3x2(r[4 * w], r[4 * w + 1]), cvt16_e4m3x2(r[4 * w + 2], r[4 * w + 3]));
    } else if constexpr (FPV == F_E2M3) {
      // tensor memory holds 6-bit A operands one per byte (low 6 bits)
#pragma unroll
      for (int w = 0; w < 16; ++w)
        out[w] = pack_b16x2(cvt16_e2m3x2(r[4 * w], r[4 * w + 1]), cvt16_e2m3x2(r[4 * w + 2], r[4 * w + 3]));
    } else {
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const uint32_t b01 = cvt_e2m1x2(r[8 * w], r[8 * w + 1]), b23 = cvt_e2m1x2(r[8 * w + 2], r[8 * w + 3]);
        const uint32_t b45 = cvt_e2m1x2(r[8 * w + 4], r[8 * w + 5]), b67 = cvt_e2m1x2(r[8 * w + 6], r[8 * w + 7]);
        out[w] = prmt(prmt(b01, b23, 0x0040u), prmt(b45, b67, 0x0040u), 0x5410u);
      }
    }
  }
  return (uint32_t)(E0 + 127) | ((uint32_t)(E1 + 127) << 8);
}

// bar.red.or over `nthreads` threads of named barrier `id`: true if any predicate is set.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n barrier.red.or.pred q, %2, %3, p;\n"
               " selp.b32 %0, 1, 0, q;\n}" : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}

}  // namespace fsa

namespace fsa {

template <int FQK, int FPV, int D, int EXPM>
__global__ void __launch_bounds__(320, 1)
fsa_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const KParams p) {
  using C = Cfg<FQK, FPV, D>;
  constexpr int KIND_QK = Fmt<FQK>::kind, KIND_PV = Fmt<FPV>::kind;
  constexpr bool MX = C::MX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: heavy causal tiles first
  const int qt = p.causal ? (p.n_qtiles - 1 - (int)blockIdx.x) : (int)blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
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
  uint64_t* k_empty = bars + 1 + C::NS;
  uint64_t* v_full = bars + 1 + 2 * C::NS;
  uint64_t* v_empty = bars + 1 + 3 * C::NS;
  uint64_t* s_full = bars + 1 + 4 * C::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = s_full + 4;
  uint64_t* drain = s_full + 6;
  uint64_t* stall = s_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 8);
  float* red = reinterpret_cast<float*>(sm + C::OFF_RED);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1);
      mbar_init(v_full + i, 1); mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) { mbar_init(s_full + i, 1); mbar_init(p_full + i, 8); mbar_init(pv_done + i, 1); }
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp >= 2) {
    // constant rows D..D+15 of every V stage (row D = ones, the rest zero) and the
    // scale atom that gives the ones row scale 2^0 in the upper tensor-memory columns
    const int t = threadIdx.x - 64;
    uint32_t one4;
    if constexpr (FPV == F_BF16) one4 = 0x3F803F80u;
    else if constexpr (FPV == F_E4M3) one4 = 0x38383838u;
    else if constexpr (FPV == F_E2M3) one4 = 0u;   // set per word below (packed 6-bit)
    else one4 = 0x22222222u;
    constexpr int ROWW = C::W_V / 4;                 // words per row per atom
    constexpr int PER_STAGE = C::NKA_V * 16 * ROWW;
    for (int i = t; i < C::NS * PER_STAGE; i += 256) {
      const int st = i / PER_STAGE, rem = i % PER_STAGE;
      const int ka = rem / (16 * ROWW), r = (rem / ROWW) % 16, w = rem % ROWW;
      uint32_t val = 0u;
      if (r == 0) {
        if constexpr (FPV == F_E2M3) {
          const int wg = w & 3;                      // 16-byte group: bytes (08 82 20) x 4, then 4 zero bytes
          val = wg == 0 ? 0x08208208u : (wg == 1 ? 0x82082082u : (wg == 2 ? 0x20820820u : 0u));
        } else {
          val = one4;
        }
      }
      uint32_t* dst = reinterpret_cast<uint32_t*>(sV + st * C::TILE_V + ka * C::VATOM + (D + r) * C::W_V);
      dst[w] = val;
    }
    if (MX) {
      uint32_t* one_atom = reinterpret_cast<uint32_t*>(sm + C::OFF_SFONE);
      for (int i = t; i < 128; i += 256) one_atom[i] = 0x7F7F7F7Fu;
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const AbortCtl ac{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // =============================================================== producer
    if (lane == 0 && nT > 0) {
      int issued_k[C::NS] = {}, issued_v[C::NS] = {};
      const int bhq = b * p.H + h, bhk = b * p.Hkv + kvh;
      mbar_expect_tx(q_full, C::TILE_QK + (MX ? 512 : 0));
#pragma unroll
      for (int ka = 0; ka < C::NKA_QK; ++ka)
        tma_load_3d(sQ + ka * 128 * C::W_QK, &tm_q, q_full, ka * C::W_QK, q0, bhq);
      if (MX) bulk_load(sm + C::OFF_SFQ, p.sf_q + ((size_t)bhq * p.n_qtiles + qt) * 512, 512, q_full);
      for (int j = 0; j < nT; ++j) {
        const int st = j % C::NS;
        const uint32_t ph = (j / C::NS) & 1;
        if (!mbar_wait(k_empty + st, ph ^ 1, ac)) break;
        mbar_expect_tx(k_full + st, C::TILE_QK + (MX ? 512 : 0));
#pragma unroll
        for (int ka = 0; ka < C::NKA_QK; ++ka)
          tma_load_3d(sK + st * C::TILE_QK + ka * 128 * C::W_QK, &tm_k, k_full + st, ka * C::W_QK, j * 128, bhk);
        if (MX) bulk_load(sm + C::OFF_SFK + st * 512, p.sf_k + ((size_t)bhk * nkt + j) * 512, 512, k_full + st);
        ++issued_k[st];
        if (!mbar_wait(v_empty + st, ph ^ 1, ac)) break;
        mbar_expect_tx(v_full + st, C::TILE_V_TMA + (MX ? 512 : 0));
#pragma unroll
        for (int ka = 0; ka < C::NKA_V; ++ka)
          tma_load_3d(sV + st * C::TILE_V + ka * C::VATOM, &tm_v, v_full + st, j * C::RB_V + ka * C::W_V, 0, bhk);
        if (MX) bulk_load(sm + C::OFF_SFV + st * 512, p.sf_v + ((size_t)bhk * nkt + j) * 512, 512, v_full + st);
        ++issued_v[st];
      }
      // every copy this thread started has landed before the CTA tears down
      mbar_wait_drain(q_full, 0, p.timeout_ns);
      for (int st = 0; st < C::NS; ++st) {
        if (issued_k[st]) mbar_wait_drain(k_full + st, (issued_k[st] - 1) & 1, p.timeout_ns);
        if (issued_v[st]) mbar_wait_drain(v_full + st, (issued_v[st] - 1) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // =============================================================== MMA issuer
    if (lane == 0 && nT > 0) {
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      constexpr uint32_t SWQ = swz_code(C::W_QK), SWV = swz_code(C::W_V);
      bool ok = true;
      if (p.inject_stall) ok = mbar_wait(stall, 0, ac);        // nobody arrives: the wait must expire
      ok = ok && mbar_wait(q_full, 0, ac);
      if (ok) {
        tc_fence_after();
        if constexpr (MX) {
          tc_cp_sf_atom(tbase + C::T_SFQ, smem_desc(smem_u32(sm + C::OFF_SFQ), 16, 128, 0));
          if constexpr (D == 128) {
            tc_cp_sf_atom(tbase + C::T_SFV + 4, smem_desc(smem_u32(sm + C::OFF_SFONE), 16, 128, 0));
            tc_cp_sf_atom(tbase + C::T_SFV + 12, smem_desc(smem_u32(sm + C::OFF_SFONE), 16, 128, 0));
          }
        }
      }
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj & 1, st = jj % C::NS;
        const uint32_t ph = (jj / C::NS) & 1;
        if (!mbar_wait(p_full + s, (jj >> 1) & 1, ac)) return false;
        if (!mbar_wait(v_full + st, ph, ac)) return false;
        tc_fence_after();
        if constexpr (MX)
          tc_cp_sf_atom(tbase + C::T_SFV + 8 * s, smem_desc(smem_u32(sm + C::OFF_SFV + st * 512), 16, 128, 0));
#pragma unroll
        for (int i = 0; i < C::PV_STEPS; ++i) {
          const int hh = i / C::STEPS_PER_HALF, j2 = i % C::STEPS_PER_HALF;
          const uint32_t a_tm = tbase + C::T_S + 128 * s + 64 * hh + 8 * j2;
          const int ka = (i * 32) / C::W_V, off = (i * 32) % C::W_V;
          const uint64_t bd = smem_desc(sVa + st * C::TILE_V + ka * C::VATOM + off, 16, 8 * C::W_V, SWV);
          const uint32_t acc = (jj > 0 || i > 0) ? 1u : 0u;
          if constexpr (KIND_PV == 0) {
            mma_f16_ts(tbase + C::T_O, a_tm, bd, idesc_f16_bf16(C::N_PV), acc);
          } else if constexpr (KIND_PV == 1) {
            mma_mxf8f6f4_ts(tbase + C::T_O, a_tm, bd, idesc_bs(C::N_PV, Fmt<FPV>::code, j2, i),
                            tbase + C::T_SFP + 8 * s + 4 * hh, tbase + C::T_SFV + 8 * s, acc);
          } else {
            mma_mxf4_ts(tbase + C::T_O, a_tm, bd, idesc_bs(C::N_PV, 1, 0, 2 * i),
                        tbase + C::T_SFP + 8 * s + 4 * hh, tbase + C::T_SFV + 8 * s, acc);
          }
        }
        tc_commit(pv_done + s);
        tc_commit(v_empty + st);
        return true;
      };
      for (int j = 0; ok && j < nT; ++j) {
        const int s = j & 1, st = j % C::NS;
        const uint32_t ph = (j / C::NS) & 1;
        if (!mbar_wait(k_full + st, ph, ac)) { ok = false; break; }
        tc_fence_after();
        if constexpr (MX)
          tc_cp_sf_atom(tbase + C::T_SFK + 4 * s, smem_desc(smem_u32(sm + C::OFF_SFK + st * 512), 16, 128, 0));
#pragma unroll
        for (int i = 0; i < C::QK_STEPS; ++i) {
          const int ka = (i * 32) / C::W_QK, off = (i * 32) % C::W_QK;
          const uint64_t ad = smem_desc(sQa + ka * 128 * C::W_QK + off, 16, 8 * C::W_QK, SWQ);
          const uint64_t bd = smem_desc(sKa + st * C::TILE_QK + ka * 128 * C::W_QK + off, 16, 8 * C::W_QK, SWQ);
          const uint32_t acc = i > 0 ? 1u : 0u;
          if constexpr (KIND_QK == 0) {
            mma_f16_ss(tbase + C::T_S + 128 * s, ad, bd, idesc_f16_bf16(128), acc);
          } else if constexpr (KIND_QK == 1) {
            mma_mxf8f6f4_ss(tbase + C::T_S + 128 * s, ad, bd, idesc_bs(128, Fmt<FQK>::code, i, i),
                            tbase + C::T_SFQ, tbase + C::T_SFK + 4 * s, acc);
          } else {
            mma_mxf4_ss(tbase + C::T_S + 128 * s, ad, bd, idesc_bs(128, 1, 2 * i, 2 * i),
                        tbase + C::T_SFQ, tbase + C::T_SFK + 4 * s, acc);
          }
        }
        tc_commit(s_full + s);
        tc_commit(k_empty + st);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nT - 1);
      // all MMAs and copies issued by this thread complete before tensor memory is freed
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // =============================================================== softmax / epilogue
    const int hh = (warp - 2) >> 2;                 // key half of every tile
    const int qd = warp & 3;                        // tensor-memory lane quadrant
    const int rl = 32 * qd + lane;                  // row within the tile
    const int row = q0 + rl;
    const bool row_valid = row < p.Sq;
    const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16);
    int lim = p.Sk - 1;
    if (p.causal) lim = min(lim, row + p.Sk - p.Sq);
    const float c = p.c;
    float M = kNegInf;
    int nfb = 0, nvis = 0;
    bool ok = true;
    for (int j = 0; j < nT; ++j) {
      const int s = j & 1;
      // a failed wait (here or in the previous fallback) is exchanged with the partner
      // warp below, so both warps of a row pair leave the loop at the same iteration
      const bool got = __all_sync(0xffffffffu, ok && mbar_wait(s_full + s, (j >> 1) & 1, ac));
      float sv[64];
      float bm0 = kNegInf, bm1 = kNegInf;
      if (got) {
        tc_fence_after();
        uint32_t raw[64];
        tmem_ld_cols<64>(tl + C::T_S + 128 * s + 64 * hh, raw);
        tc_wait_ld();
        const int kbase = 128 * j + 64 * hh;
#pragma unroll
        for (int i = 0; i < 64; ++i) sv[i] = __uint_as_float(raw[i]);
        if (kbase + 63 > lim) {                     // only diagonal / tail tiles mask keys
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (kbase + i > lim) sv[i] = kNegInf;
        }
        bm0 = max32(sv);
        bm1 = max32(sv + 32);
      }
      // The row's two halves agree on the tile maximum only when some row of the warp
      // pair needs it: its first visible tile, a fallback (x > M + delta), or a failed
      // wait.  The test per half is exact: rounding is monotone, so
      // fp32(max(a,b)*c) > T  <=>  fp32(a*c) > T or fp32(b*c) > T.
      const float hm = fmaxf(bm0, bm1);
      const bool vis = 128 * j <= lim;               // first key of the tile visible to this row
      const bool need = !got || (vis && (M == kNegInf ||
                                         (MX ? (__fmul_rn(hm, c) > __fadd_rn(M, p.delta))
                                             : (__fsub_rn(__fmul_rn(hm, c), M) > 8.0f))));
      bool rescale = false;
      float Mn = M;
      if (vis) ++nvis;
      if (named_bar_or(1 + qd, 64, need)) {
        red[(s * 2 + hh) * 128 + rl] = got ? hm : __int_as_float(0x7FC00000);
        named_bar_sync(1 + qd, 64);
        const float other = red[(s * 2 + (1 - hh)) * 128 + rl];
        if (!got || isnan(other)) { ok = false; break; }
        const float mx = fmaxf(hm, other);
        const float x = __fmul_rn(mx, c);
        if (mx != kNegInf) {
          if (M == kNegInf) {
            M = x;
          } else if (MX ? (x > __fadd_rn(M, p.delta)) : (__fsub_rn(x, M) > 8.0f)) {
            rescale = true;
            Mn = x;
          }
        }
      }
      // fallback: O_aug row *= 2^(M - M') once the previous PV has landed.  tcgen05.ld/st
      // are warp-collective, so the whole warp rescales when any of its rows falls
      // back; the other rows multiply by exactly 1.
      if (__any_sync(0xffffffffu, rescale)) {
        const float alpha = rescale ? ex2_approx(__fsub_rn(M, Mn)) : 1.0f;
        const bool pv_ok = __all_sync(0xffffffffu, mbar_wait(pv_done + ((j - 1) & 1), ((j - 1) >> 1) & 1, ac));
        if (!pv_ok) ok = false;
        tc_fence_after();
        constexpr int HALF = C::N_PV / 2;             // 72 or 40 columns, in chunks of 8
#pragma unroll
        for (int c0 = 0; c0 < HALF; c0 += 8) {
          uint32_t o[8];
          TmemLd<8>::run(tl + C::T_O + hh * HALF + c0, o);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__fmul_rn(__uint_as_float(o[i]), alpha));
          TmemSt<8>::run(tl + C::T_O + hh * HALF + c0, o);
        }
        tc_wait_st();
        if (rescale) {
          M = Mn;
          ++nfb;
        }
      }
      // ---- P~ for this half: codes into the consumed S columns, scales into SFP
      if constexpr (MX) {
        uint32_t pw[16];
        const uint32_t sw = pgen_half<FPV, EXPM>(sv, bm0, bm1, c, M, p.efq_beta, pw);
        tmem_st_cols<C::P_COLS_HALF>(tl + C::T_S + 128 * s + 64 * hh, pw);
        TmemSt<1>::run(tl + C::T_SFP + 8 * s + 4 * hh + qd, &sw);
      } else {
        uint32_t pw[32];
        const float nM = M == kNegInf ? 0.0f : -M;   // no visible key yet: every s is -inf, p = 0
        const uint64_t c2 = pk2(c, c), nM2 = pk2(nM, nM);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float a, bb;
          upk2(ffma2(pk2(sv[2 * i], sv[2 * i + 1]), c2, nM2), a, bb);
          pw[i] = cvt_bf16x2(ex2_approx(a), ex2_approx(bb));
        }
        tmem_st_cols<32>(tl + C::T_S + 128 * s + 64 * hh, pw);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + s);
    }
    // ---- epilogue: O = O_aug[:, :D] / l
    float* orow = p.out + (((size_t)b * p.H + h) * p.Sq + (row_valid ? row : 0)) * D + hh * (D / 2);
    const bool done = ok && nT > 0 &&
                      __all_sync(0xffffffffu, mbar_wait(pv_done + ((nT - 1) & 1), ((nT - 1) >> 1) & 1, ac));
    if (done) {
      tc_fence_after();
      uint32_t lraw;
      TmemLd<1>::run(tl + C::T_O + D, &lraw);
      uint32_t o[D / 2];
      tmem_ld_cols<D / 2>(tl + C::T_O + hh * (D / 2), o);
      tc_wait_ld();
      const float l = __uint_as_float(lraw);
      if (row_valid) {
#pragma unroll
        for (int i = 0; i < D / 2; i += 4) {
          float4 v;
          v.x = l > 0.f ? __fdiv_rn(__uint_as_float(o[i]), l) : 0.f;
          v.y = l > 0.f ? __fdiv_rn(__uint_as_float(o[i + 1]), l) : 0.f;
          v.z = l > 0.f ? __fdiv_rn(__uint_as_float(o[i + 2]), l) : 0.f;
          v.w = l > 0.f ? __fdiv_rn(__uint_as_float(o[i + 3]), l) : 0.f;
          *reinterpret_cast<float4*>(orow + i) = v;
        }
      }
    } else if (nT == 0 && row_valid) {
#pragma unroll
      for (int i = 0; i < D / 2; i += 4) *reinterpret_cast<float4*>(orow + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (hh == 0) {
      if (row_valid && p.row_fallbacks) p.row_fallbacks[((size_t)b * p.H + h) * p.Sq + row] = nfb;
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
  }
  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ----------------------------------------------------------------------------- host launch
template <int FQK, int FPV, int D, int EXPM>
static cudaError_t launch_one(const AttnLaunch& a) {
  using C = Cfg<FQK, FPV, D>;
  // at least 116 KB so that one CTA (and its 512 tensor-memory columns) owns an SM
  constexpr int smem = (C::SMEM > 116 * 1024 ? C::SMEM : 116 * 1024);
  auto kern = fsa_attn_kernel<FQK, FPV, D, EXPM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.p.n_qtiles, a.p.H, a.p.B);
  kern<<<grid, C::NTHREADS, smem, a.stream>>>(a.tq, a.tk, a.tv, a.p);
  return cudaGetLastError();
}

template <int FQK, int FPV>
cudaError_t launch_attn_impl(const AttnLaunch& a) {
  constexpr bool efq_or_bf16 = FPV == F_EFQ || FPV == F_BF16;
  if (a.D == 64) {
    if constexpr (efq_or_bf16) return launch_one<FQK, FPV, 64, 1>(a);
    else {
      if (a.exp_mode == 0) return launch_one<FQK, FPV, 64, 0>(a);
      if (a.exp_mode == 1) return launch_one<FQK, FPV, 64, 1>(a);
      return launch_one<FQK, FPV, 64, 2>(a);
    }
  }
  if constexpr (efq_or_bf16) return launch_one<FQK, FPV, 128, 1>(a);
  else {
    if (a.exp_mode == 0) return launch_one<FQK, FPV, 128, 0>(a);
    if (a.exp_mode == 1) return launch_one<FQK, FPV, 128, 1>(a);
    return launch_one<FQK, FPV, 128, 2>(a);
  }
}

}  // namespace fsa

#if defined(FSA_INST_QK) && defined(FSA_INST_PV)
template cudaError_t fsa::launch_attn_impl<FSA_INST_QK, FSA_INST_PV>(const fsa::AttnLaunch&);
#endif
