// fsa_quant.cu -- bf16 -> MX (OCP microscaling) quantisation kernels and the
// bf16 V transpose used by the BF16 baseline.
//
// MX operands: the Fused-Softmax brief (abstract) runs QK^T and PV as MXFP8 /
// MXFP6 / MXFP4 GEMMs.  Blocks of 32 elements share one E8M0 scale 2^E with
// E = clamp(floor(log2 amax) - emax, -127, 127); element codes are x * 2^-E
// rounded to nearest even with saturation (cvt.rn.satfinite).  Layouts are the
// ones fsa.h documents: Q/K blocked along D, V stored transposed and blocked
// along keys, scales in 128x4 atoms that tcgen05.cp copies into tensor memory.
#include <cstdint>
#include <cuda_runtime.h>
#include "fsa_launch.h"
#include "fsa_mx.cuh"

namespace fsa {

// --------------------------------------------------------------------------
// Rows layout (Q, K): one CTA per (128-row tile, b*h), 256 threads.  Chunk =
// 8 consecutive elements of a row, 4 chunks = one 32-element block; thread t
// takes chunks t, t + 256, ... of the tile, all loads issued before any
// arithmetic.  The tile's 512-byte scale atom is assembled in shared memory
// (unused slots 0x7F) and written whole.
// x: [BH][S][D] bf16, codes: [BH*S][row bytes], scales: [BH][ceil(S/128)][512].
// tile_id = b*h * ceil(S/128) + tile; atom: 512 bytes of shared memory.
template <int FMT, int D>
__device__ __forceinline__ void quant_rows_tile(const uint16_t* __restrict__ x, int S, uint8_t* __restrict__ codes,
                                                uint8_t* __restrict__ scales, int64_t tile_id, uint8_t* atom) {
  constexpr int emax = mx_emax(FMT);
  constexpr int CPR = D / 8;                       // chunks per row
  constexpr int NCH = 128 * CPR / 256;             // chunks per thread
  constexpr int RB = FMT == 2 ? D / 2 : D;         // code bytes per row
  const int t = threadIdx.x;
  const int ntiles = (S + 127) / 128;
  const int64_t bh = tile_id / ntiles;             // one grid axis: no limit on B*H
  const int s0 = (int)(tile_id % ntiles) * 128;
  const int nrows = min(128, S - s0);
  const uint16_t* src = x + ((int64_t)bh * S + s0) * D;
  uint8_t* dst = codes + ((int64_t)bh * S + s0) * RB;
  if (t < 128) reinterpret_cast<uint32_t*>(atom)[t] = 0x7F7F7F7Fu;
  uint4 raw[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int ch = t + 256 * i;
    raw[i] = ch / CPR < nrows ? *reinterpret_cast<const uint4*>(src + 8 * ch) : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();                                 // atom initialised before the scale bytes land
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int ch = t + 256 * i, r = ch / CPR, c = ch % CPR;
    const bool active = r < nrows;
    const uint32_t wr[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    float v[8];
    float amax = 0.f;
    bool nonfinite = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = bf16_to_f32((uint16_t)(wr[e] & 0xFFFF));
      v[2 * e + 1] = bf16_to_f32((uint16_t)(wr[e] >> 16));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float a = fabsf(v[e]);
      nonfinite |= !(a <= 3.4e38f);
      amax = fmaxf(amax, a);
    }
    // 4-lane group reduction (groups are lane-aligned: CPR and 256 are multiples of 4)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int nf = nonfinite;
    nf |= __shfl_xor_sync(0xffffffffu, nf, 1);
    nf |= __shfl_xor_sync(0xffffffffu, nf, 2);
    const uint32_t sbyte = nf ? 0xFFu : block_scale_byte(amax, emax);
    const float mul = nf ? 1.0f : pow2_neg((int)sbyte - 127);
    uint32_t q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (nf) q[e] = FMT == 0 ? 0x7F7Fu : 0u;
      else q[e] = cvt_pair<FMT>(__fmul_rn(v[2 * e], mul), __fmul_rn(v[2 * e + 1], mul));
    }
    if constexpr (mx_six_bit(FMT)) {
      // 16-element groups: the even chunk packs its and its neighbour's codes
      uint32_t w[4] = {q[0] | (q[1] << 16), q[2] | (q[3] << 16), 0u, 0u};
      w[2] = __shfl_down_sync(0xffffffffu, w[0], 1);
      w[3] = __shfl_down_sync(0xffffffffu, w[1], 1);
      if (active && (c & 1) == 0) {
        uint32_t o[3];
        pack6x16(w, o);
        *reinterpret_cast<uint4*>(dst + r * RB + 8 * c) = make_uint4(o[0], o[1], o[2], 0u);
      }
    } else if (active) {
      if constexpr (FMT == 0)
        *reinterpret_cast<uint2*>(dst + r * RB + 8 * c) = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
      else
        *reinterpret_cast<uint32_t*>(dst + r * RB + 4 * c) = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
    }
    if (active && (c & 3) == 0) atom[(r & 31) * 16 + (r >> 5) * 4 + (c >> 2)] = (uint8_t)sbyte;
  }
  __syncthreads();
  if (t < 32) reinterpret_cast<uint4*>(scales + tile_id * 512)[t] = reinterpret_cast<const uint4*>(atom)[t];
}

// NVFP4 rows (Q, K): as quant_rows_tile with 16-element blocks (two lanes, two
// chunks) and D/64 scale atoms per tile: block b of row r goes to byte
// (b/4)*512 + (r%32)*16 + (r/32)*4 + b%4 (rows past S keep 0x38, 1.0).
template <int D>
__device__ __forceinline__ void quant_rows_tile_nv(const uint16_t* __restrict__ x, int S, uint8_t* __restrict__ codes,
                                                   uint8_t* __restrict__ scales, int64_t tile_id, uint8_t* atom,
                                                   const uint4* staged = nullptr) {
  constexpr int CPR = D / 8;                       // chunks per row
  constexpr int NCH = 128 * CPR / 256;             // chunks per thread
  constexpr int RB = D / 2;                        // code bytes per row
  constexpr int NATOM = D / 64;
  const int t = threadIdx.x;
  const int ntiles = (S + 127) / 128;
  const int64_t bh = tile_id / ntiles;
  const int s0 = (int)(tile_id % ntiles) * 128;
  const int nrows = min(128, S - s0);
  const uint16_t* src = x + ((int64_t)bh * S + s0) * D;
  uint8_t* dst = codes + ((int64_t)bh * S + s0) * RB;
  if (t < 128 * NATOM) reinterpret_cast<uint32_t*>(atom)[t] = 0x38383838u;
  uint4 raw[NCH];
  if (staged == nullptr) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ch = t + 256 * i;
      raw[i] = ch / CPR < nrows ? *reinterpret_cast<const uint4*>(src + 8 * ch) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncthreads();                                 // atoms initialised before the scale bytes land
  if (staged != nullptr) {
#pragma unroll
    for (int i = 0; i < NCH; ++i) raw[i] = staged[t + 256 * i];
  }
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int ch = t + 256 * i, r = ch / CPR, c = ch % CPR;
    const uint32_t wr[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    float v[8];
    float amax = 0.f;
    bool nonfinite = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = bf16_to_f32((uint16_t)(wr[e] & 0xFFFF));
      v[2 * e + 1] = bf16_to_f32((uint16_t)(wr[e] >> 16));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float a = fabsf(v[e]);
      nonfinite |= !(a <= 3.4e38f);
      amax = fmaxf(amax, a);
    }
    // 2-lane group reduction (a block is chunks 2m, 2m + 1 of one row: CPR is even)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const int nf = nonfinite | __shfl_xor_sync(0xffffffffu, (int)nonfinite, 1);
    const uint32_t sbyte = nvfp4_scale_byte(amax, nf != 0);
    const uint32_t w = nf ? 0u : nvfp4_codes8(v, e4m3_to_f32(sbyte));
    if (r < nrows) {
      *reinterpret_cast<uint32_t*>(dst + r * RB + 4 * c) = w;
      if ((c & 1) == 0) {
        const int b = c >> 1;
        atom[(b >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (b & 3)] = (uint8_t)sbyte;
      }
    }
  }
  __syncthreads();
  if (t < 32 * NATOM)
    reinterpret_cast<uint4*>(scales + tile_id * 512 * NATOM)[t] = reinterpret_cast<const uint4*>(atom)[t];
}

template <int FMT, int D>
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(const uint16_t* __restrict__ x, int S,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  __shared__ __align__(16) uint8_t atom[1024];
  if constexpr (FMT == 5) quant_rows_tile_nv<D>(x, S, codes, scales, blockIdx.x, atom);
  else quant_rows_tile<FMT, D>(x, S, codes, scales, blockIdx.x, atom);
}

// --------------------------------------------------------------------------
// Transposed layout (V): one CTA per (128-key tile, b*h), 256 threads.  The
// tile is loaded into shared memory (all loads issued first); then each thread
// quantises two adjacent columns d, d+1 over one 32-key block, and the scale
// atom (rows d >= D and blocks past the sequence: 0x7F) is written whole.
// x: [BH][S][D] bf16; codes: [BH][D][Sp] elements; scales: [BH][Sp/128][512].
// tile_id = b*h * (Sp/128) + tile; tile: 128 x D bf16 of shared memory; atom: 512 bytes.
template <int FMT, int D>
__device__ __forceinline__ void quant_cols_tile(const uint16_t* __restrict__ x, int S, int Sp,
                                                uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                int64_t tile_id, uint32_t* tile, uint8_t* atom) {
  constexpr int NV = 128 * D / 8 / 256;            // 16-byte vectors per thread
  constexpr int DW = D / 2;                        // 32-bit words per tile row
  const int t = threadIdx.x;
  const int ntiles = Sp / 128;
  const int64_t bh = tile_id / ntiles;
  const int s0 = (int)(tile_id % ntiles) * 128;
  const int nrows = min(128, S - s0);
  const uint16_t* src = x + ((int64_t)bh * S + s0) * D;
  uint4 raw[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vi = t + 256 * i;
    raw[i] = (vi * 8) / D < nrows ? *reinterpret_cast<const uint4*>(src + 8 * vi) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) reinterpret_cast<uint4*>(tile)[t + 256 * i] = raw[i];
  if (t < 128) reinterpret_cast<uint32_t*>(atom)[t] = 0x7F7F7F7Fu;
  __syncthreads();
  if (t < DW * 4) {
    const int d2 = t % DW, kb = t / DW;
    const int d = 2 * d2, k0 = 32 * kb;
    uint32_t w0[8], w1[8];
    uint32_t sb0 = 0x7Fu, sb1 = 0x7Fu;
    if (s0 + k0 < S) {                             // else: block wholly past the sequence end, zero codes
      float v0[32], v1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t pr = tile[(k0 + i) * DW + d2];
        v0[i] = bf16_to_f32((uint16_t)(pr & 0xFFFF));
        v1[i] = bf16_to_f32((uint16_t)(pr >> 16));
      }
      sb0 = quant_block32<FMT>(v0, w0);
      sb1 = quant_block32<FMT>(v1, w1);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w0[i] = w1[i] = 0u;
    }
    const int64_t e0 = ((bh * D + d) * (int64_t)Sp) + s0 + k0;   // element index of column d's block
    if constexpr (FMT == 2) {
      uint4* p0 = reinterpret_cast<uint4*>(codes + e0 / 2);
      uint4* p1 = reinterpret_cast<uint4*>(codes + (e0 + Sp) / 2);
      p0[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
      p1[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    } else {
      uint4* p0 = reinterpret_cast<uint4*>(codes + e0);
      uint4* p1 = reinterpret_cast<uint4*>(codes + e0 + Sp);
      p0[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
      p0[1] = make_uint4(w0[4], w0[5], w0[6], w0[7]);
      p1[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
      p1[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
    }
    atom[(d & 31) * 16 + (d >> 5) * 4 + kb] = (uint8_t)sb0;
    atom[((d + 1) & 31) * 16 + ((d + 1) >> 5) * 4 + kb] = (uint8_t)sb1;
  }
  __syncthreads();
  if (t < 32) reinterpret_cast<uint4*>(scales + tile_id * 512)[t] = reinterpret_cast<const uint4*>(atom)[t];
}

template <int FMT, int D>
__global__ void __launch_bounds__(256) mx_quant_cols_kernel(const uint16_t* __restrict__ x, int S, int Sp,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  __shared__ __align__(16) uint32_t tile[128 * D / 2];
  __shared__ __align__(16) uint8_t atom[512];
  quant_cols_tile<FMT, D>(x, S, Sp, codes, scales, blockIdx.x, tile, atom);
}

// --------------------------------------------------------------------------
// Q, K and V of one attention call in one launch: CTAs [0, nq) take the tiles
// of Q, [nq, nq + nk) those of K (rows layout), the rest those of V
// (transposed layout).  The same codes and scales as three separate launches,
// without two kernel boundaries between them.
struct QkvArgs {
  const uint16_t* x[3];
  uint8_t* codes[3];
  uint8_t* scales[3];
  int Sq, Sk, Spv;
  int64_t nq, nk;
};

// Four CTAs per SM (registers capped at 64; a few bytes spill): more tiles' loads in
// flight measured 13% faster at 128K keys than three CTAs per SM.
template <int FQK, int FV, int D>
__global__ void __launch_bounds__(256, 4) mx_quant_qkv_kernel(const QkvArgs a) {
  __shared__ __align__(16) uint32_t tile[128 * D / 2];
  __shared__ __align__(16) uint8_t atom[FQK == 5 ? 512 * (D / 64) : 512];
  const int64_t b = blockIdx.x;                    // block-uniform branch
  auto rows = [&](const uint16_t* x, int S, uint8_t* codes, uint8_t* scales, int64_t tid) {
    if constexpr (FQK == 5) quant_rows_tile_nv<D>(x, S, codes, scales, tid, atom);   // NVFP4 Q and K
    else quant_rows_tile<FQK, D>(x, S, codes, scales, tid, atom);
  };
  if (b < a.nq) rows(a.x[0], a.Sq, a.codes[0], a.scales[0], b);
  else if (b < a.nq + a.nk) rows(a.x[1], a.Sk, a.codes[1], a.scales[1], b - a.nq);
  else quant_cols_tile<FV, D>(a.x[2], a.Sk, a.Spv, a.codes[2], a.scales[2], b - a.nq - a.nk, tile, atom);
}

// V [BH][S][D] bf16 -> V^T [BH][D][Sp] bf16 (zero padded), one CTA per 128-key tile.
__global__ void __launch_bounds__(256) transpose_v_kernel(const uint16_t* __restrict__ x, int S, int D, int Sp,
                                                          uint16_t* __restrict__ vt) {
  extern __shared__ __align__(16) uint16_t tile[];        // [128][D]
  const int t = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int s0 = t * 128;
  const uint16_t* src = x + (bh * S) * (int64_t)D;
  const int nvec = 128 * D / 8;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
    const int s = (i * 8) / D, d = (i * 8) % D;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (s0 + s < S) val = *reinterpret_cast<const uint4*>(src + (int64_t)(s0 + s) * D + d);
    *reinterpret_cast<uint4*>(tile + s * D + d) = val;
  }
  __syncthreads();
  const int nout = D * 16;                      // each thread: 8 consecutive keys of one d
  for (int i = threadIdx.x; i < nout; i += blockDim.x) {
    const int d = i / 16, k8 = (i % 16) * 8;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = (uint32_t)tile[(k8 + 2 * j) * D + d] | ((uint32_t)tile[(k8 + 2 * j + 1) * D + d] << 16);
    *reinterpret_cast<uint4*>(vt + (bh * D + d) * (int64_t)Sp + s0 + k8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------------ launchers
template <int FMT>
static cudaError_t quant_rows_d(const uint16_t* x, int BH, int S, int D, uint8_t* c, uint8_t* s, cudaStream_t st) {
  const int64_t n = ((int64_t)S + 127) / 128 * BH;                   // (b*h, tile), tile fastest
  if (n > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const unsigned grid = (unsigned)n;
  if (D == 128) mx_quant_rows_kernel<FMT, 128><<<grid, 256, 0, st>>>(x, S, c, s);
  else mx_quant_rows_kernel<FMT, 64><<<grid, 256, 0, st>>>(x, S, c, s);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t quant_cols_d(const uint16_t* x, int BH, int S, int D, uint8_t* c, uint8_t* s, cudaStream_t st) {
  const int Sp = (S + 127) / 128 * 128;
  const int64_t n = (int64_t)Sp / 128 * BH;
  if (n > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const unsigned grid = (unsigned)n;
  if (D == 128) mx_quant_cols_kernel<FMT, 128><<<grid, 256, 0, st>>>(x, S, Sp, c, s);
  else mx_quant_cols_kernel<FMT, 64><<<grid, 256, 0, st>>>(x, S, Sp, c, s);
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_rows(const void* x, int BH, int S, int D, int fmt, void* codes, void* scales,
                                 cudaStream_t st) {
  auto* xs = static_cast<const uint16_t*>(x);
  auto* c = static_cast<uint8_t*>(codes);
  auto* s = static_cast<uint8_t*>(scales);
  switch (fmt) {
    case 0: return quant_rows_d<0>(xs, BH, S, D, c, s, st);
    case 1: return quant_rows_d<1>(xs, BH, S, D, c, s, st);
    case 4: return quant_rows_d<4>(xs, BH, S, D, c, s, st);
    case 5: return quant_rows_d<5>(xs, BH, S, D, c, s, st);
    default: return quant_rows_d<2>(xs, BH, S, D, c, s, st);
  }
}

cudaError_t launch_mx_quant_cols(const void* x, int BH, int S, int D, int fmt, void* codes, void* scales,
                                 cudaStream_t st) {
  auto* xs = static_cast<const uint16_t*>(x);
  auto* c = static_cast<uint8_t*>(codes);
  auto* s = static_cast<uint8_t*>(scales);
  switch (fmt) {
    case 0: return quant_cols_d<0>(xs, BH, S, D, c, s, st);
    case 1: return quant_cols_d<1>(xs, BH, S, D, c, s, st);
    case 4: return quant_cols_d<4>(xs, BH, S, D, c, s, st);
    default: return quant_cols_d<2>(xs, BH, S, D, c, s, st);
  }
}

template <int FQK, int FV>
static cudaError_t quant_qkv_d(const QkvArgs& a, int64_t n, int D, cudaStream_t st) {
  if (D == 128) mx_quant_qkv_kernel<FQK, FV, 128><<<(unsigned)n, 256, 0, st>>>(a);
  else mx_quant_qkv_kernel<FQK, FV, 64><<<(unsigned)n, 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int FQK>
static cudaError_t quant_qkv_fv(const QkvArgs& a, int64_t n, int D, int fv, cudaStream_t st) {
  switch (fv) {
    case 0: return quant_qkv_d<FQK, 0>(a, n, D, st);
    case 1: return quant_qkv_d<FQK, 1>(a, n, D, st);
    case 4: return quant_qkv_d<FQK, 4>(a, n, D, st);
    default: return quant_qkv_d<FQK, 2>(a, n, D, st);
  }
}

cudaError_t launch_mx_quant_qkv(const void* q, const void* k, const void* v, int BHq, int BHk, int Sq, int Sk, int D,
                                int fqk, int fv, void* cq, void* sq, void* ck, void* sk, void* cv, void* sv,
                                cudaStream_t st) {
  QkvArgs a;
  a.x[0] = static_cast<const uint16_t*>(q);
  a.x[1] = static_cast<const uint16_t*>(k);
  a.x[2] = static_cast<const uint16_t*>(v);
  a.codes[0] = static_cast<uint8_t*>(cq); a.scales[0] = static_cast<uint8_t*>(sq);
  a.codes[1] = static_cast<uint8_t*>(ck); a.scales[1] = static_cast<uint8_t*>(sk);
  a.codes[2] = static_cast<uint8_t*>(cv); a.scales[2] = static_cast<uint8_t*>(sv);
  a.Sq = Sq;
  a.Sk = Sk;
  a.Spv = (Sk + 127) / 128 * 128;
  a.nq = ((int64_t)Sq + 127) / 128 * BHq;
  a.nk = ((int64_t)Sk + 127) / 128 * BHk;
  const int64_t n = a.nq + a.nk + (int64_t)a.Spv / 128 * BHk;
  if (n > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  switch (fqk) {
    case 0: return quant_qkv_fv<0>(a, n, D, fv, st);
    case 1: return quant_qkv_fv<1>(a, n, D, fv, st);
    case 4: return quant_qkv_fv<4>(a, n, D, fv, st);
    case 5: return quant_qkv_fv<5>(a, n, D, fv, st);
    default: return quant_qkv_fv<2>(a, n, D, fv, st);
  }
}

cudaError_t launch_transpose_v(const void* v, void* vt, int BH, int S, int D, cudaStream_t st) {
  const int Sp = (S + 127) / 128 * 128;
  dim3 grid(Sp / 128, BH);
  transpose_v_kernel<<<grid, 256, (size_t)128 * D * 2, st>>>(static_cast<const uint16_t*>(v), S, D, Sp,
                                                             static_cast<uint16_t*>(vt));
  return cudaGetLastError();
}

}  // namespace fsa
