// fsa_attn_persistent.cuh -- the persistent schedule of the fused MX attention
// forward (and its BF16 twin): one CTA per SM walks a list of query tiles (snake
// order over the grid, heaviest first when causal), so a CTA's setup, first loads,
// pipeline fill and drain are paid once per SM instead of once per query tile.
//
// Per key tile the work is the one of fsa_attn_kernel (fsa_attn.cu): the same TMA
// producer, MMA issuer and softmax warps, the same arithmetic in the same order,
// so the two schedules give bit-identical outputs.  What changes: key tiles are
// counted over the CTA's query tiles (g), so ring slots, S and P~ buffers and
// barrier phases run on across them; Q is double-buffered; a query tile's first PV
// (which overwrites O_aug) waits on o_free, which both softmax parts arrive on once
// they hold the previous tile's O_aug rows; output rows go out through two 32x16 boxes
// per warp by TMA stores.
#pragma once

namespace fsa {

// One part's half of a finished query tile's output rows (thread = row): O_aug
// columns [DP*pp, DP*pp + DP) and l from tensor memory, 16 columns at a time (few
// registers next to the key-tile loop); each chunk is normalised, written to the
// warp's two 32x16 staging boxes in turn (64B swizzle) and stored by TMA (rows past
// Sq are clipped).  After the last tensor-memory load, o_free: O_aug may be overwritten.
// A query tile without key tiles gets zeros.
template <int D, bool MX>
__device__ __forceinline__ void write_rows(uint32_t t_o, int pp, int qd, int lane, float lb, bool done, bool has_keys,
                                           uint8_t* stage, const CUtensorMap* tm_o, int q0, int bhq, uint64_t* o_free,
                                           bool bf16) {
  constexpr int DP = D / 2;
  if (!done && has_keys) {                           // aborted: release O_aug, write nothing
    tc_fence_before();
    __syncwarp();
    mbar_arrive_elect(o_free);
    return;
  }
  float l = 0.f;
  if (done) {
    tc_fence_after();
    if constexpr (MX) {
      uint32_t lraw;
      TmemLd<1>::run(t_o + D, &lraw);
      tc_wait_ld();
      l = __uint_as_float(lraw);
    } else {
      l = lb;
    }
  }
  // fp32 normalisation: one correctly rounded reciprocal of l per row, then products
  // (within 1.5 ulp of the quotient).  A row with no visible key has l = 0 (or NaN:
  // its residuals are -inf + inf) and gets zeros.
  const bool lpos = l > 0.f;
  const float rinv = lpos ? __frcp_rn(l) : 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < DP; c0 += 16) {
    uint32_t o[16];
    if (done) {
      tmem_ld_cols<16>(t_o + DP * pp + c0, o);
      tc_wait_ld();
      if (c0 + 16 == DP) {
        tc_fence_before();
        __syncwarp();
        mbar_arrive_elect(o_free);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = 0u;
    }
    // MX: two boxes in turn, and the store that last read this chunk's box is the one
    // before the latest, so the latest may still be reading the other box (BF16: one)
    uint8_t* box = stage + (MX ? ((c0 / 16) & 1) * 2048 : 0);
    if (lane == 0) {
      if constexpr (MX) bulk_wait_read_1();
      else bulk_wait_read();
    }
    __syncwarp();
    if (bf16) {
      // bf16: the same fp32 quotients rounded to nearest even, 32 bytes per row (32B
      // swizzle: 16-byte chunk ch of row `lane` sits at chunk ch ^ ((lane / 4) % 2))
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = lpos ? __fmul_rn(__uint_as_float(o[8 * ch + 2 * e]), rinv) : 0.f;
          const float b = lpos ? __fmul_rn(__uint_as_float(o[8 * ch + 2 * e + 1]), rinv) : 0.f;
          w[e] = cvt_bf16x2(a, b);
        }
        *reinterpret_cast<uint4*>(box + lane * 32 + ((ch ^ ((lane >> 2) & 1)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const float4 v = lpos ? make_float4(__fmul_rn(__uint_as_float(o[4 * ch]), rinv),
                                            __fmul_rn(__uint_as_float(o[4 * ch + 1]), rinv),
                                            __fmul_rn(__uint_as_float(o[4 * ch + 2]), rinv),
                                            __fmul_rn(__uint_as_float(o[4 * ch + 3]), rinv))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        // 64B swizzle: 16-byte chunk ch of row `lane` sits at chunk ch ^ ((lane / 2) % 4)
        *reinterpret_cast<float4*>(box + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4)) = v;
      }
    }
    fence_proxy_async_smem();                        // generic writes -> TMA reads
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tm_o, box, DP * pp + c0, q0 + 32 * qd, bhq);
      bulk_commit_group();
    }
  }
}

// One query tile of one (batch, head): its first row and its number of key tiles.
struct Item {
  int q0, bhq, bhk, nT;
};
// Query tiles in processing order: causal, heaviest first with (batch, head) fastest;
// otherwise the query tiles of one head together, so that the CTAs of a round share
// its K/V in L2.
__device__ __forceinline__ Item item_of(const KParams& p, int k) {
  const int BH = p.B * p.H;
  int qt, bh;
  if (p.causal) {
    qt = p.n_qtiles - 1 - k / BH;
    bh = k % BH;
  } else {
    bh = k / p.n_qtiles;
    qt = k % p.n_qtiles;
  }
  const int h = bh % p.H, b = bh / p.H;
  Item it;
  it.q0 = qt * 128;
  it.bhq = bh;
  it.bhk = b * p.Hkv + h / (p.H / p.Hkv);
  const int nkt = (p.Sk + 127) / 128;
  it.nT = nkt;
  if (p.causal) {
    const int lim = it.q0 + 127 + p.Sk - p.Sq;
    it.nT = lim < 0 ? 0 : min(nkt, lim / 128 + 1);
  }
  return it;
}
// The query tile this CTA takes in round r (snake order over the grid, which keeps the
// heaviest-first order balanced), or -1 past the last.
__device__ __forceinline__ int item_at(int r, int n_items) {
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const int k = r * G + ((r & 1) ? G - 1 - c : c);
  return k < n_items ? k : -1;
}

// The key tiles of one query tile that one softmax part owns (see the kernel's
// softmax section).
struct TileState {
  float lsum, Ml;   // BF16: the part's denominator and the maximum it is relative to
  int nfb, nvis;    // fallbacks and visible tiles of this row
  bool ok;
};
template <int FQK, int FPV, int D, int EXPM>
__device__ __forceinline__ TileState softmax_tiles(uint32_t tl, uint64_t* s_full, uint64_t* pv_done, float* m_slot,
                                                AbortCtl ac, const KParams& p, int pp, int qd,
                                                int lim, int nT, int g0, bool ok) {
  using C = Cfg<FQK, FPV, D, true>;
  constexpr bool MX = C::MX;
  constexpr int NBLK = 4;                         // 32-key blocks per tile
  const float c = p.c;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;
  const int bar_in = 1 + qd + 4 * pp, bar_out = 1 + qd + 4 * (1 - pp);
  auto wait0 = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, ac));
  };
  float M = kNegInf;
  int nfb = 0, nvis = 0;
  float lsum = 0.0f, Ml = kNegInf;
    for (int j = pp ^ (g0 & 1); j < nT; j += 2) {
      const int g = g0 + j;
      const int s = pp;
      const bool got = ok && wait0(s_full + s, (g >> 1) & 1);
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
      if constexpr (!MX) {
        if (Ml != kNegInf && M != Ml) lsum *= ex2_approx(__fsub_rn(Ml, M));
        Ml = M;
      }
      if (ok) {
        // ---- P~ of the tile in two halves of two 32-key blocks.  The first half is
        // generated before waiting for the PVs that the rescale and the buffer reuse
        // depend on, which gives them that much longer to finish.
        constexpr int HW = C::P_COLS / 2;             // words (columns) per half
        const uint32_t tp = tl + C::T_P + C::P_COLS * (g % C::NPB);
        uint32_t swb[NBLK] = {};                    // scale bytes of the blocks (low bytes)
        uint64_t acc = pk2(0.0f, 0.0f);               // BF16: sum of the rounded p
        const float nM = M == kNegInf ? 0.0f : -M;    // BF16, no visible key yet: every s is -inf, p = 0
        auto gen_half = [&](int hf, uint32_t* pw) {
          if constexpr (MX) {
            constexpr int WB = C::P_COLS / NBLK;       // words per block: 8, or 4 for E2M1
#pragma unroll
            for (int b = 0; b < 2; ++b)
              swb[2 * hf + b] = pgen_block<FPV, EXPM>(sv + 64 * hf + 32 * b, bm[2 * hf + b], c, M, p, pw + WB * b);
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
        uint32_t pw[HW];
        if constexpr (MX) gen_half(0, pw);           // (BF16: too many registers to hold across)
        // fallback: O_aug row *= 2^(M_old - M) once PV(j-1) has landed.  tcgen05.ld/st
        // are warp-collective, so the whole warp rescales when any of its rows falls
        // back; the other rows multiply by exactly 1.
        if (__any_sync(0xffffffffu, rescale)) {
          // PV(j-2) first: with two PV barriers (BF16) PV(j-1) shares its barrier with
          // PV(j-3), and its parity only identifies PV(j-1) once PV(j-3) has completed
          const bool prev = g < C::NPB || wait0(pv_done + (g - C::NPB) % C::NS, ((g - C::NPB) / C::NS) & 1);
          if (prev && wait0(pv_done + (g - 1) % C::NS, ((g - 1) / C::NS) & 1)) {
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
        // P~ buffer g % NPB and scale column s were last read by PV(g - NPB)
        if (ok && g >= C::NPB && !wait0(pv_done + (g - C::NPB) % C::NS, ((g - C::NPB) / C::NS) & 1)) ok = false;
        if (ok) {
          tc_fence_after();
          if constexpr (!MX) gen_half(0, pw);
          tmem_st_cols<HW>(tp, pw);
          gen_half(1, pw);
          tmem_st_cols<HW>(tp + HW, pw);
          // A scales of the PV MMA: lane quadrant q reads column base + q
          const uint32_t sw = low_bytes4(swb[0], swb[1], swb[2], swb[3]);
          if constexpr (MX) TmemSt<1>::run(tl + C::T_SFP + 4 * s + qd, &sw);
          if constexpr (!MX) {
            float a0, a1;
            upk2(acc, a0, a1);
            lsum += a0 + a1;
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (ok) mbar_arrive_elect(p_full + s);
      }
    }
  TileState st;
  st.lsum = lsum;
  st.Ml = Ml;
  st.nfb = nfb;
  st.nvis = nvis;
  st.ok = ok;
  return st;
}

template <int FQK, int FPV, int D, int EXPM>
__global__ void __launch_bounds__(Cfg<FQK, FPV, D, true>::NTHREADS, 1)
fsa_attn_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const KParams p) {
  using C = Cfg<FQK, FPV, D, true>;
  constexpr int KIND_QK = Fmt<FQK>::kind, KIND_PV = Fmt<FPV>::kind;
  constexpr bool MX = C::MX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
  const int n_items = p.n_items;
  const int nkt = (p.Sk + 127) / 128;

  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* q_full = bars;                      // Q buffer b landed (per query tile with keys)
  uint64_t* q_empty = bars + 2;                 // QK^T of the tile that used Q buffer b done
  uint64_t* k_full = bars + 4;
  uint64_t* v_full = k_full + C::NS;
  uint64_t* pv_done = v_full + C::NS;           // PV(g) -> slot g % NS (g: the CTA's key-tile count)
  uint64_t* k_empty = pv_done + C::NS;          // S(g) done -> K slot g % NS
  uint64_t* s_full = k_empty + C::NS;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;
  uint64_t* o_free = s_full + 6;                // O_aug of the previous query tile read out
  uint64_t* drain = s_full + 7;
  uint64_t* stall = s_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 8);
  float* red = reinterpret_cast<float*>(sm + C::OFF_RED);

  // the first query tile's Q and first ring of K/V tiles are requested while the rest
  // of the CTA sets up; E counts the key tiles requested that way
  const Item it0 = item_of(p, item_at(0, n_items));
  const int E = min(C::NS, it0.nT);
  auto load_q = [&](const Item& it, int qb) {
    mbar_expect_tx(q_full + qb, C::TILE_QK + (MX ? 512 : 0));
#pragma unroll
    for (int ka = 0; ka < C::NKA_QK; ++ka)
      tma_load_3d(sQ + qb * C::TILE_QK + ka * 128 * C::W_QK, &tm_q, q_full + qb, ka * C::W_QK, it.q0, it.bhq);
    if (MX)
      bulk_load(sm + C::OFF_SFQ + qb * 512, p.sf_q + ((size_t)it.bhq * p.n_qtiles + it.q0 / 128) * 512, 512,
                q_full + qb);
  };
  auto load_k = [&](const Item& it, int j, int st) {
    mbar_expect_tx(k_full + st, C::TILE_QK + (MX ? 512 : 0));
#pragma unroll
    for (int ka = 0; ka < C::NKA_QK; ++ka)
      tma_load_3d(sK + st * C::TILE_QK + ka * 128 * C::W_QK, &tm_k, k_full + st, ka * C::W_QK, j * 128, it.bhk);
    if (MX) bulk_load(sm + C::OFF_SFK + st * 512, p.sf_k + ((size_t)it.bhk * nkt + j) * 512, 512, k_full + st);
  };
  auto load_v = [&](const Item& it, int j, int st) {
    mbar_expect_tx(v_full + st, C::TILE_V_TMA + (MX ? 512 : 0));
#pragma unroll
    for (int ka = 0; ka < C::NKA_V; ++ka)
      tma_load_3d(sV + st * C::TILE_V + ka * C::VATOM, &tm_v, v_full + st, j * C::RB_V + ka * C::W_V, 0, it.bhk);
    if (MX) bulk_load(sm + C::OFF_SFV + st * 512, p.sf_v + ((size_t)it.bhk * nkt + j) * 512, 512, v_full + st);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1); mbar_init(q_empty + i, 1);
    }
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(k_full + i, 1); mbar_init(v_full + i, 1); mbar_init(pv_done + i, 1); mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      // one softmax warp per lane quadrant owns each key tile
      mbar_init(s_full + i, 1); mbar_init(s_free + i, 4); mbar_init(p_full + i, 4);
    }
    mbar_init(o_free, C::NSW);
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    sts_vol(abort_flag, 0);
    fence_mbar_init();
    if (it0.nT > 0) {
      load_q(it0, 0);
      for (int j = 0; j < E; ++j) {
        load_k(it0, j, j);
        load_v(it0, j, j);
      }
    }
  }
  // the CTA's query tiles, one per thread (the host keeps them within MAX_ITEMS)
  Item* items = reinterpret_cast<Item*>(sm + C::OFF_ITEMS);
  for (int r = threadIdx.x; r < C::MAX_ITEMS; r += C::NTHREADS) {
    const int k = item_at(r, n_items);
    if (k < 0) break;
    items[r] = item_of(p, k);
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
    // Lane 0 loads Q (one buffer per query tile with keys, two buffers) and the K
    // tiles, lane 1 the V tiles; both walk the CTA's query tiles in order, counting
    // key tiles g across them, so a ring slot is g % NS whatever tile it belongs to.
    if (lane < 2) {
      bool run = true;
      int g = 0, nq = 0;
      for (int r = 0; run; ++r) {
        if (item_at(r, n_items) < 0) break;
        const Item it = items[r];
        if (it.nT == 0) continue;
        if (lane == 0) {
          const int qb = nq & 1;
          if (nq > 0 || it0.nT == 0) {               // (the first one went out during the setup)
            if (nq >= 2 && !mbar_wait(q_empty + qb, ((nq - 2) >> 1) & 1, ac)) break;
            load_q(it, qb);
          }
          ++nq;
        }
        for (int j = 0; j < it.nT; ++j, ++g) {
          if (g < E) continue;
          const int st = g % C::NS;
          if (lane == 0) {
            // K slot st is free once S(g - NS) is done
            if (g >= C::NS && !mbar_wait(k_empty + st, ((g - C::NS) / C::NS) & 1, ac)) { run = false; break; }
            load_k(it, j, st);
          } else {
            // V slot st is free once PV(g - NS) is done
            if (g >= C::NS && !mbar_wait(pv_done + st, ((g - C::NS) / C::NS) & 1, ac)) { run = false; break; }
            load_v(it, j, st);
          }
        }
      }
      // every copy this thread started has landed before the CTA tears down
      // (g counts the key tiles requested, those of the setup included)
      if (lane == 0) {
        for (int qb = 0; qb < 2 && qb < nq; ++qb)
          mbar_drain(q_full + qb, ((nq - 1 - qb) >> 1) & 1, ac);
        for (int st = 0; st < C::NS && st < g; ++st)
          mbar_drain(k_full + st, ((g - 1 - st) / C::NS) & 1, ac);
      } else {
        for (int st = 0; st < C::NS && st < g; ++st)
          mbar_drain(v_full + st, ((g - 1 - st) / C::NS) & 1, ac);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // =============================================================== MMA issuer
    // The warp runs converged; every lane polls and the votes agree, and each tcgen05
    // instruction is issued by the elected lane (the same lane throughout, so its
    // commits cover all of them).  One warp issues both GEMMs: tcgen05 work from two
    // issuing warps of one CTA was measured to serialise badly.
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, ac));
    };
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
    constexpr uint32_t SWQ = swz_code(C::W_QK), SWV = swz_code(C::W_V);
    bool ok = true;
    if (p.inject_stall) ok = __all_sync(0xffffffffu, mbar_wait(stall, 0, ac));   // nobody arrives: must expire
    if (ok) {
      tc_fence_after();
      if constexpr (MX && D == 128) {
        const uint64_t one = smem_desc(smem_u32(sm + C::OFF_SFONE), 16, 128, 0);
        tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFV + 4, one);
        tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFV + 12, one);
      }
    }
    // PV of key tile g; `first`: the query tile's first, which overwrites O_aug
    auto issue_pv = [&](int g, bool first) {
      const int s = g & 1, st = g % C::NS;
      tc_fence_after();
      if constexpr (MX) {
        const uint64_t sfd = smem_desc(smem_u32(sm + C::OFF_SFV + st * 512), 16, 128, 0);
        tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFV + 8 * s, sfd);
      }
#pragma unroll
      for (int i = 0; i < C::PV_STEPS; ++i) {
        // P~ of step i sits in columns [8i, 8i+8) of its P buffer; the scale word of
        // each row (byte b = 32-key block b) is in column T_SFP + 4 s + lane quadrant
        const uint32_t a_tm = tbase + C::T_P + C::P_COLS * (g % C::NPB) + 8 * i;
        const uint32_t sfa = tbase + C::T_SFP + 4 * s;
        const int ka = (i * 32) / C::W_V, off = (i * 32) % C::W_V;
        const uint64_t bd = smem_desc(sVa + st * C::TILE_V + ka * C::VATOM + off, 16, 8 * C::W_V, SWV);
        const uint32_t acc = (!first || i > 0) ? 1u : 0u;
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
    // QK^T of key tile g against Q buffer qb; `first`: the query tile's first (its Q
    // scales go to tensor memory), `last`: its last (Q buffer qb is then free)
    auto issue_s = [&](int g, int qb, bool first, bool last) {
      const int s = g & 1, st = g % C::NS;
      const uint32_t t_sfq = qb ? C::T_SFQ1 : C::T_SFQ;
      tc_fence_after();
      if constexpr (MX) {
        const uint64_t sfd = smem_desc(smem_u32(sm + C::OFF_SFK + st * 512), 16, 128, 0);
        tc_cp_sf_atom_p(elect_u32(), tbase + C::T_SFK + 4 * s, sfd);
      }
#pragma unroll
      for (int i = 0; i < C::QK_STEPS; ++i) {
        const int ka = (i * 32) / C::W_QK, off = (i * 32) % C::W_QK;
        const uint64_t ad = smem_desc(sQa + qb * C::TILE_QK + ka * 128 * C::W_QK + off, 16, 8 * C::W_QK, SWQ);
        const uint64_t bd = smem_desc(sKa + st * C::TILE_QK + ka * 128 * C::W_QK + off, 16, 8 * C::W_QK, SWQ);
        const uint32_t acc = i > 0 ? 1u : 0u;
        const uint32_t e = elect_u32();
        if constexpr (KIND_QK == 0) {
          mma_f16_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_f16_bf16(128), acc);
        } else if constexpr (KIND_QK == 1) {
          mma_mxf8f6f4_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_bs(128, Fmt<FQK>::code, i, i),
                            tbase + t_sfq, tbase + C::T_SFK + 4 * s, acc);
        } else {
          mma_mxf4_ss_p(e, tbase + C::T_S + 128 * s, ad, bd, idesc_bs(128, 1, 2 * i, 2 * i),
                        tbase + t_sfq, tbase + C::T_SFK + 4 * s, acc);
        }
      }
      tc_commit_p(elect_u32(), s_full + s);
      tc_commit_p(elect_u32(), k_empty + st);
    };
    // The next query tile with keys at or after round r (false: none left).
    // Query tile by query tile (those with key tiles): Q landed, its scale atom to
    // tensor memory, then the key tiles through a non-blocking scheduler, and after
    // them a commit that frees the Q buffer.  Key tiles are counted over the CTA (g),
    // so ring slots and buffer phases run on across query tiles.  Each round every
    // lane tests the barriers of the next QK^T (K landed, S buffer loaded by its
    // owners) and of the next PV (P~ written, V landed), and whichever GEMM is ready
    // is issued; a query tile's first PV also waits until the previous tile's O_aug
    // has been read out.
    int g = 0, qi = 0;
    for (int r = 0; ok && item_at(r, n_items) >= 0; ++r) {
      const int nT = items[r].nT;
      if (nT == 0) continue;
      const int qb = qi & 1;
      if (!wait_all(q_full + qb, (qi >> 1) & 1)) break;
      if constexpr (MX) {
        tc_fence_after();
        tc_cp_sf_atom_p(elect_u32(), tbase + (qb ? C::T_SFQ1 : C::T_SFQ),
                        smem_desc(smem_u32(sm + C::OFF_SFQ + qb * 512), 16, 128, 0));
      }
      int jS = 0, jP = 0;
      uint32_t idle = 0;
      uint64_t t0 = 0;
      while (ok && jP < nT) {
        const int gS = g + jS, gP = g + jP;
        const bool tk = jS < nT && mbar_test(k_full + gS % C::NS, (gS / C::NS) & 1);
        const bool tf = gS < 2 || mbar_test(s_free + (gS & 1), ((gS - 2) >> 1) & 1);
        const bool tp = jP < jS && mbar_test(p_full + (gP & 1), (gP >> 1) & 1);
        const bool tv = mbar_test(v_full + gP % C::NS, (gP / C::NS) & 1);
        const bool rs = __all_sync(0xffffffffu, tk && tf), rp = __all_sync(0xffffffffu, tp && tv);
        if (rs) issue_s(gS, qb, false, false), ++jS;
        if (rp) {
          if (jP == 0 && qi > 0 && !wait_all(o_free, (qi - 1) & 1)) {
            ok = false;
            break;
          }
          issue_pv(gP, jP == 0);
          ++jP;
        }
        if (rs || rp) {
          idle = 0;
          continue;
        }
        // nothing ready: park in a suspending try_wait on what most likely completes
        // next, so the warp takes no issue slots from the softmax warps of its
        // scheduler.  The owners of a key tile release its S when they load it, early
        // in the tile, and write P~ at its end; the other part's tiles are half a tile
        // behind.  So the release of S(gS-2) comes before P~(gP) unless PV lags QK^T by
        // four tiles or more.
        if (jS < nT && jS - jP <= 3) {
          if (!tk) mbar_try_wait(k_full + gS % C::NS, (gS / C::NS) & 1);
          else if (gS >= 2) mbar_try_wait(s_free + (gS & 1), ((gS - 2) >> 1) & 1);
        } else if (jP < jS) {
          if (!tp) mbar_try_wait(p_full + (gP & 1), (gP >> 1) & 1);
          else mbar_try_wait(v_full + gP % C::NS, (gP / C::NS) & 1);
        }
        __syncwarp();
        // bounded wait, abort check
        if (++idle == 1) t0 = globaltimer_ns();
        if ((idle & 7u) == 0) {
          bool stop = lds_vol(ac.flag) != 0;
          if (!stop && globaltimer_ns() - t0 > ac.limit_ns) {
            sts_vol(ac.flag, 1);
            if (ac.status) atomicExch(ac.status, -4);   // FSA_ERR_TIMEOUT
            stop = true;
          }
          if (__any_sync(0xffffffffu, stop)) ok = false;
        }
      }
      // the Q buffer is free once this query tile's MMAs have completed
      tc_commit_p(elect_u32(), q_empty + qb);
      g += nT;
      ++qi;
    }
    // all MMAs and copies issued by this warp complete before tensor memory is freed
    tc_commit_p(elect_u32(), drain);
    mbar_drain(drain, 0, ac);
    __syncwarp();
  } else {
    // =============================================================== softmax / epilogue
    // The two warps of a tensor-memory lane quadrant take alternate key tiles: part pp
    // owns the tiles g (counted over the CTA's query tiles) with g % 2 == pp, all 128
    // keys of its 32 rows (thread = row), and with them S buffer, P~ buffer and scale
    // column pp.  The running maximum M passes between the two once per key tile
    // (shared memory plus a named-barrier handoff).  After its last key tile of a
    // query tile each part writes its half of the output rows and goes on to the next
    // query tile.
    constexpr int NBLK = 4;                         // 32-key blocks per tile
    const int pp = (warp - 2) >> 2;
    const int qd = warp & 3;                        // tensor-memory lane quadrant
    const int rl = 32 * qd + lane;                  // row within the tile
    const uint32_t tl = tbase + ((uint32_t)(32 * qd) << 16);
    const float c = p.c;
    const int bar_in = 1 + qd + 4 * pp, bar_out = 1 + qd + 4 * (1 - pp);
    float* m_slot = red + rl;                       // M of this row after the latest tile
    bool ok = true;                                 // false once any wait failed: no more work
    // every lane polls; the vote keeps the warp uniform
    auto wait0 = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
      return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, ac));
    };
    int g0 = 0;                                     // key tiles of the earlier query tiles
    for (int r = 0;; ++r) {
    if (item_at(r, n_items) < 0) break;
    int lim = p.Sk - 1;
    if (p.causal) lim = min(lim, items[r].q0 + rl + p.Sk - p.Sq);
    const TileState ts = softmax_tiles<FQK, FPV, D, EXPM>(tl, s_full, pv_done, m_slot, ac, p, pp, qd,
                                                          lim, items[r].nT, g0, ok);
    const Item it = items[r];                       // re-read: not held across the key-tile loop
    const int nT = it.nT;
    const int row = it.q0 + rl;
    const bool row_valid = row < p.Sq;
    ok = ts.ok;
    const int nfb = ts.nfb, nvis = ts.nvis;
    const float lsum = ts.lsum, Ml = ts.Ml;
    // ---- this query tile's output: O = O_aug[:, :D] / l, D/2 columns per part
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
    // PV(gl-1) before PV(gl): with two PV barriers (BF16) the parity of PV(gl) only
    // identifies it once PV(gl-2) has completed
    const int gl = g0 + nT - 1;
    const bool done = ok && nT > 0 && (gl < 1 || wait0(pv_done + (gl - 1) % C::NS, ((gl - 1) / C::NS) & 1)) &&
                      wait0(pv_done + gl % C::NS, (gl / C::NS) & 1);
    write_rows<D, MX>(tl + C::T_O, pp, qd, lane, lb, done, nT > 0, sm + C::OFF_OSTAGE + (warp - 2) * C::OSTAGE_WARP, &tm_o,
                      it.q0, it.bhq, o_free, p.out_bf16 != 0);
    // ---- statistics: each part counted the key tiles it owns
    int* nfb_other = reinterpret_cast<int*>(red) + 128 + rl;
    if (pp == 1) *nfb_other = nfb;
    named_bar_sync(9 + qd, 64);
    if (pp == 0 && row_valid && p.row_fallbacks)
      p.row_fallbacks[(size_t)it.bhq * p.Sq + row] = nfb + *nfb_other;
    named_bar_sync(9 + qd, 64);                      // read before the next query tile's write
    {
      int f = row_valid ? nfb : 0, v = row_valid ? nvis : 0;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) {
        f += __shfl_xor_sync(0xffffffffu, f, o2);
        v += __shfl_xor_sync(0xffffffffu, v, o2);
      }
      if (lane == 0 && p.stat_fallbacks) {
        if (f) atomicAdd(p.stat_fallbacks, (unsigned long long)f);
        atomicAdd(p.stat_row_tiles, (unsigned long long)v);
      }
    }
    g0 += nT;
    }
    if (lane == 0) bulk_wait_all();                  // the output stores are done before the CTA ends
  }
  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace fsa
