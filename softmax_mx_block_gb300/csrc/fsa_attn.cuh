// fsa_attn.cuh -- compile-time configuration of the fused attention kernel:
// operand storage formats, shared-memory and tensor-memory layouts.
#pragma once
#include <cstdint>
#include "fsa_ptx.cuh"

namespace fsa {

// Operand formats (0..4 as fsa.h numbers them; F_NVFP4 is fsa.h's 5).  F_EFQ stores
// E2M1 like F_E2M1; it only changes how the softmax warps produce P.  F_NVFP4 is a
// QK^T operand format only: E2M1 codes, one E4M3 scale per 16 elements.
enum : int { F_E4M3 = 0, F_E2M3 = 1, F_E2M1 = 2, F_EFQ = 3, F_E3M2 = 4, F_BF16 = 5, F_NVFP4 = 6 };

template <int F> struct Fmt;
// kind: 0 = kind::f16, 1 = kind::mxf8f6f4 (scale_vec 1X, K = 32), 2 = kind::mxf4 (2X, K = 64),
// 3 = kind::mxf4nvf4 (4X, K = 64, UE4M3 scales)
// code: the element type field of the block-scaled instruction descriptor
// bits2: storage bits per element * 2 (E2M1 packs two per byte)
template <> struct Fmt<F_BF16> { static constexpr int kind = 0, bits2 = 32, code = 0, emax = 0; };
template <> struct Fmt<F_E4M3> { static constexpr int kind = 1, bits2 = 16, code = 0, emax = 8; };
template <> struct Fmt<F_E2M3> { static constexpr int kind = 1, bits2 = 16, code = 3, emax = 2; };  // 16 codes / 16 bytes
template <> struct Fmt<F_E3M2> { static constexpr int kind = 1, bits2 = 16, code = 4, emax = 4; };  // 16 codes / 16 bytes
template <> struct Fmt<F_E2M1> { static constexpr int kind = 2, bits2 = 8, code = 1, emax = 2; };
template <> struct Fmt<F_EFQ>  { static constexpr int kind = 2, bits2 = 8, code = 1, emax = 2; };
template <> struct Fmt<F_NVFP4> { static constexpr int kind = 3, bits2 = 8, code = 1, emax = 0; };

__host__ __device__ constexpr int swz_code(int width) { return width == 128 ? 2 : (width == 64 ? 4 : 6); }

// PERSIST: the persistent schedule (one CTA per SM walking a list of query tiles),
// which adds a second Q buffer, an output staging area and the list.
// QF: Q arrives as bf16 and is quantised in the kernel's prologue, which adds a
// staging area for the bf16 tile and its barrier (one CTA per query tile only).
template <int FQK, int FPV, int D_, bool PERSIST = false, bool QF = false>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int BM = 128, BN = 128;
  static constexpr bool MX = FQK != F_BF16;
  static_assert((FQK == F_BF16) == (FPV == F_BF16), "BF16 kernel uses BF16 for both GEMMs");
  static_assert(FQK != F_EFQ, "EFQ is a P format");
  static_assert(FPV != F_NVFP4, "NVFP4 is a QK^T operand format");
  // NVFP4 Q/K: one 512-byte scale atom per K = 64 step (D/64 of them per tile)
  static constexpr bool NV = FQK == F_NVFP4;
  static_assert(!(NV && (PERSIST || QF)), "NVFP4 runs one CTA per query tile with Q quantised beforehand");
  static constexpr int NATOM_QK = NV ? D_ / 64 : 1;
  static constexpr int SFQK = 512 * NATOM_QK;                       // scale bytes of a Q or K tile
  // ---- QK^T operands (Q, K rows of D elements)
  static constexpr int RB_QK = D * Fmt<FQK>::bits2 / 16;            // bytes per row
  static constexpr int W_QK = RB_QK < 128 ? RB_QK : 128;            // swizzle atom width
  static constexpr int NKA_QK = RB_QK / W_QK;                       // atoms along K
  static constexpr int QK_STEPS = RB_QK / 32;                       // 32 bytes of K per MMA
  static constexpr int TILE_QK = BM * RB_QK;                        // bytes of a 128-row tile
  // ---- PV operands (V^T rows of 128 keys; the MX kernels add 16 rows, a ones row
  // and zero rows, whose product column accumulates the denominator l)
  static constexpr int N_PV = MX ? D + 16 : D;
  static constexpr int RB_V = BN * Fmt<FPV>::bits2 / 16;            // bytes per V^T row per key tile
  static constexpr int W_V = RB_V < 128 ? RB_V : 128;
  static constexpr int NKA_V = RB_V / W_V;
  static constexpr int PV_STEPS = RB_V / 32;
  static constexpr int VATOM = N_PV * W_V;                          // bytes of one K-atom of the V tile
  static constexpr int TILE_V = NKA_V * VATOM;
  static constexpr int TILE_V_TMA = NKA_V * D * W_V;                // bytes TMA writes per tile
  // ---- softmax: two warps per tensor-memory lane quadrant, taking alternate key
  // tiles (thread = one row, all 128 keys of the tile)
  static constexpr int NQ = 2;
  static constexpr int NSW = 4 * NQ;                                // softmax warps
  // ---- P~ in tensor memory, its own buffers (so S is free once loaded)
  static constexpr int P_COLS = 128 * Fmt<FPV>::bits2 / 16 / 4;     // 32 (8-bit), 16 (E2M1), 64 (BF16)
  // P~ buffers (and P~ scale columns and P~-arrival barriers): four for 16-column E2M1
  // P~ in the per-tile kernel, where the scale columns fit.  With three or more, the
  // PV that last read buffer j % NPB, PV(j - NPB), has completed by the time S(j) is
  // there: the MMA warp issues QK^T(j) after PV(j - 3), and the commit that signals
  // S(j) covers every MMA the warp issued before it.  So the softmax warps need no
  // wait for the buffer; with two they wait for PV(j - 2).
  // (NVFP4 Q/K: three, with the P~ scale columns after the buffers, since its scale
  // atoms take the columns in front of them)
  static constexpr int NPB = (MX && !PERSIST && P_COLS == 16) ? (NV ? 3 : 4) : 2;
  static_assert(P_COLS == 8 * PV_STEPS, "one PV step per 8 columns");
  // ---- pipeline
  static constexpr int NS = MX ? 4 : 2;                             // K/V stages
  static constexpr int SF_BYTES = 512;
  // ---- shared memory offsets (1024-aligned tiles)
  static constexpr int NQB = PERSIST ? 2 : 1;                       // Q buffers
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQB * TILE_QK;
  static constexpr int OFF_V = OFF_K + NS * TILE_QK;
  static constexpr int OFF_SF = (OFF_V + NS * TILE_V + 1023) / 1024 * 1024;
  static constexpr int OFF_SFQ = OFF_SF;
  static constexpr int OFF_SFK = OFF_SFQ + NQB * SFQK;
  static constexpr int OFF_SFV = OFF_SFK + NS * SFQK;
  static constexpr int OFF_SFONE = OFF_SFV + NS * SF_BYTES;
  static constexpr int OFF_RED = OFF_SFONE + SF_BYTES;              // M handoff, fallback counts, BF16 {l, M} x 2
  static constexpr int OFF_BAR = OFF_RED + (256 + 4 * 128) * 4;
  // q full (+ q empty x2 when persistent), k/v full, pv done, k empty x NS, s full/free,
  // p full x2, (o free,) drain, stall
  static_assert(!(PERSIST && QF), "Q quantised in the prologue: one CTA per query tile");
  static constexpr int NBAR = PERSIST ? 4 + 4 * NS + 3 * 2 + 3 : 1 + 4 * NS + 2 * 2 + NPB + 2 + (QF ? 1 : 0);
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;               // tmem slot, abort flag
  // output staging: one CTA per query tile stages O (128 rows x D fp32, 32x32 boxes)
  // in the K/V ring, free by then; the persistent schedule has two 32-row x 16-column
  // fp32 boxes (64B swizzle) per softmax warp, used in turn (BF16: one)
  static constexpr int OFF_OSTAGE = PERSIST ? (OFF_MISC + 64 + 1023) / 1024 * 1024 : OFF_K;
  static_assert(PERSIST || OFF_K + 128 * D * 4 <= OFF_SF, "O staging fits the K/V ring");
  // persistent: the CTA's query tiles in processing order (at most MAX_ITEMS)
  static constexpr int MAX_ITEMS = 256;
  static constexpr int OSTAGE_WARP = MX ? 4096 : 2048;                // BF16: one box (shared memory)
  static constexpr int OFF_ITEMS = OFF_OSTAGE + NSW * OSTAGE_WARP;
  // QF: the bf16 Q tile, 128 rows x 2D bytes, unswizzled
  static constexpr int OFF_QRAW = (OFF_MISC + 64 + 1023) / 1024 * 1024;
  static constexpr int SMEM = PERSIST ? OFF_ITEMS + MAX_ITEMS * 16 + 1024
                                      : (QF ? OFF_QRAW + 128 * D * 2 : OFF_MISC + 64) + 1024;   // + alignment slack
  static_assert(SMEM <= 227 * 1024, "shared memory");
  // ---- tensor memory columns
  static constexpr uint32_t T_S = 0;          // S0 [0,128), S1 [128,256)
  static constexpr uint32_t T_O = 256;        // [256, 256 + N_PV)
  // a scale atom occupies 4 columns (lane quadrant q reads column + q); NVFP4 Q and K
  // have two atoms per tile at D = 128
  static constexpr uint32_t T_SFQ = 400;
  static constexpr uint32_t SFK_STEP = 4 * NATOM_QK;                // columns per K parity
  static constexpr uint32_t T_SFK = T_SFQ + 4 * NATOM_QK;          // + SFK_STEP * parity
  static constexpr uint32_t T_SFV = T_SFK + 2 * SFK_STEP;          // + 8 * parity (4 from the V atom, 4 constant)
  static constexpr uint32_t T_P = MX ? 448 : T_O + D;   // + P_COLS * buffer (BF16: no scales)
  // P~ scales: + 4 * (P~ buffer) + lane quadrant; after the P~ buffers for NVFP4 Q/K
  static constexpr bool SFP_AFTER = NV && NPB == 3;
  static constexpr uint32_t T_SFP = SFP_AFTER ? T_P + NPB * P_COLS : T_SFV + 16;
  static constexpr uint32_t T_SFQ1 = 436;     // persistent: scale atom of the second Q buffer
  static_assert(T_O + N_PV <= (MX ? T_SFQ : T_P), "tmem");
  static_assert(!MX || T_SFQ1 + 4 <= T_P, "tmem");
  static_assert(!MX || T_SFP + 4 * NPB <= (PERSIST ? T_SFQ1 : (SFP_AFTER ? 512u : T_P)), "tmem");
  static_assert(!MX || SFP_AFTER || T_SFV + 16 <= T_P, "tmem");
  static_assert(T_P + NPB * P_COLS <= (SFP_AFTER ? T_SFP : 512u), "tmem");
  // ---- threads
  static constexpr int NTHREADS = 64 + 32 * NSW;   // warp 0 TMA, warp 1 MMA, then the softmax warps
};

struct KParams {          // kept within 128 bytes: larger parameter blocks measured more spills
  int B, H, Hkv, Sq, Sk, n_qtiles, causal;
  int n_items;            // query tiles over all (batch, head): B * H * n_qtiles
  float c;                // fp32(scale * log2 e)
  float delta;
  // EFQ rule (see pgen_block): A8 = fp32(a c) / 8, a8 = a / 8, b8 = b / 8 (all exact
  // scalings by 1/8), phi the block scale's reference point
  float efq_A8, efq_a8, efq_b8, efq_phi;
  const uint8_t* sf_q;    // [B*H][ceil(Sq/128)][512]
  const uint8_t* sf_k;    // [B*Hkv][ceil(Sk/128)][512]
  const uint8_t* sf_v;    // [B*Hkv][Sp/128][512]
  uint64_t timeout_ns;
  int32_t* row_fallbacks; // optional [B][H][Sq]
  unsigned long long* stat_fallbacks;
  unsigned long long* stat_row_tiles;
  int* status;
  int inject_stall;
  int out_bf16;           // 1: O is written as bf16 (round to nearest even), else fp32
};
static_assert(sizeof(KParams) <= 128, "kernel parameter block");

// Dump pointers of the debug instance (fsa_debug_dump): raw scores [slot][nkt*128],
// M [slot][nkt], P~ words [slot][nkt][32], P~ scale word [slot][nkt]; null otherwise.
struct DbgParams {
  float* s;
  float* m;
  uint32_t* p;
  uint32_t* sf;
  const int32_t* row_slot;   // dump slot of each query row (null: the row itself; < 0: none)
};

}  // namespace fsa
