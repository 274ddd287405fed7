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

namespace fsa {

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
  else return cvt_e2m1x2(lo, hi);
}

// --------------------------------------------------------------------------
// Rows layout (Q, K): one thread per 8 consecutive elements; 4 lanes = 1 block.
// x: [R][D] bf16 (R = B*H*S), codes: [R][row_bytes], scales: 128x4 atoms.
template <int FMT>
__global__ void __launch_bounds__(256) mx_quant_rows_kernel(const uint16_t* __restrict__ x, int64_t R, int S, int D,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  constexpr int emax = FMT == 0 ? 8 : 2;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;    // chunk id
  const int chunks_per_row = D / 8;
  const int64_t row = g / chunks_per_row;
  const bool active = row < R;
  const int c = (int)(g - row * chunks_per_row);
  float v[8];
  float amax = 0.f;
  bool nonfinite = false;
  if (active) {
    const uint4 raw = *reinterpret_cast<const uint4*>(x + row * D + 8 * c);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_to_f32((uint16_t)(w[i] & 0xFFFF));
      v[2 * i + 1] = bf16_to_f32((uint16_t)(w[i] >> 16));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float a = fabsf(v[i]);
      nonfinite |= !(a <= 3.4e38f);
      amax = fmaxf(amax, a);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  // 4-lane group reduction (groups are lane-aligned: D/8 chunks per row is a multiple of 4)
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  int nf = nonfinite;
  nf |= __shfl_xor_sync(0xffffffffu, nf, 1);
  nf |= __shfl_xor_sync(0xffffffffu, nf, 2);
  const uint32_t sbyte = nf ? 0xFFu : block_scale_byte(amax, emax);
  const float mul = nf ? 1.0f : pow2_neg((int)sbyte - 127);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (nf) q[i] = FMT == 0 ? 0x7F7Fu : 0u;
    else q[i] = cvt_pair<FMT>(__fmul_rn(v[2 * i], mul), __fmul_rn(v[2 * i + 1], mul));
  }
  if (FMT == 1) {
    // 16-element groups: the even chunk packs its and its neighbour's codes
    uint32_t w[4] = {q[0] | (q[1] << 16), q[2] | (q[3] << 16), 0u, 0u};
    w[2] = __shfl_down_sync(0xffffffffu, w[0], 1);
    w[3] = __shfl_down_sync(0xffffffffu, w[1], 1);
    if (active && (c & 1) == 0) {
      uint32_t o[3];
      pack6x16(w, o);
      *reinterpret_cast<uint4*>(codes + row * D + 8 * c) = make_uint4(o[0], o[1], o[2], 0u);
    }
  } else if (active) {
    if (FMT == 0) {
      *reinterpret_cast<uint2*>(codes + row * D + 8 * c) = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
    } else {
      *reinterpret_cast<uint32_t*>(codes + row * (D / 2) + 4 * c) =
          q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
    }
  }
  if (active && (c & 3) == 0) {
    const int64_t bh = row / S;
    const int s = (int)(row - bh * S);
    const int kb = c >> 2;
    const int64_t atom = bh * ((S + 127) / 128) + s / 128;
    const int rr = s & 127;
    scales[atom * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + kb] = (uint8_t)sbyte;
  }
}

// --------------------------------------------------------------------------
// Transposed layout (V): one CTA per (128-key tile, b*h); the tile is staged
// in shared memory, each thread quantises (d, key block) columns.
// x: [BH][S][D] bf16; codes: [BH][D][Sp] elements; scales: [BH][Sp/128] atoms.
template <int FMT>
__global__ void __launch_bounds__(256) mx_quant_cols_kernel(const uint16_t* __restrict__ x, int S, int D, int Sp,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  constexpr int emax = FMT == 0 ? 8 : 2;
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
  const int npairs = D * 4;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int d = p % D, kb = p / D;
    const int k0 = 32 * kb;
    const int64_t code_elem = ((bh * D + d) * (int64_t)Sp) + s0 + k0;
    uint32_t sbyte;
    uint32_t q[16];
    if (s0 + k0 >= S) {                         // block wholly past the sequence end
      sbyte = 0x7Fu;
#pragma unroll
      for (int i = 0; i < 16; ++i) q[i] = 0u;
    } else {
      float v[32];
      float amax = 0.f;
      bool nonfinite = false;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = bf16_to_f32(tile[(k0 + i) * D + d]);
        const float a = fabsf(v[i]);
        nonfinite |= !(a <= 3.4e38f);
        amax = fmaxf(amax, a);
      }
      sbyte = nonfinite ? 0xFFu : block_scale_byte(amax, emax);
      const float mul = nonfinite ? 1.0f : pow2_neg((int)sbyte - 127);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        q[i] = nonfinite ? (FMT == 0 ? 0x7F7Fu : 0u) : cvt_pair<FMT>(__fmul_rn(v[2 * i], mul), __fmul_rn(v[2 * i + 1], mul));
    }
    if (FMT == 0) {
      uint4* dst = reinterpret_cast<uint4*>(codes + code_elem);
      dst[0] = make_uint4(q[0] | (q[1] << 16), q[2] | (q[3] << 16), q[4] | (q[5] << 16), q[6] | (q[7] << 16));
      dst[1] = make_uint4(q[8] | (q[9] << 16), q[10] | (q[11] << 16), q[12] | (q[13] << 16), q[14] | (q[15] << 16));
    } else if (FMT == 1) {
      uint4* dst = reinterpret_cast<uint4*>(codes + code_elem);
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const uint32_t w[4] = {q[8 * gi] | (q[8 * gi + 1] << 16), q[8 * gi + 2] | (q[8 * gi + 3] << 16),
                               q[8 * gi + 4] | (q[8 * gi + 5] << 16), q[8 * gi + 6] | (q[8 * gi + 7] << 16)};
        uint32_t o[3];
        pack6x16(w, o);
        dst[gi] = make_uint4(o[0], o[1], o[2], 0u);
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(codes + code_elem / 2);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = q[4 * i] | (q[4 * i + 1] << 8) | (q[4 * i + 2] << 16) | (q[4 * i + 3] << 24);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (d < 128) scales[(bh * (Sp / 128) + t) * 512 + (d & 31) * 16 + (d >> 5) * 4 + kb] = (uint8_t)sbyte;
  }
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
cudaError_t launch_mx_quant_rows(const void* x, int64_t R, int S, int D, int fmt, void* codes, void* scales,
                                 cudaStream_t st) {
  const int64_t chunks = R * (D / 8);
  const int threads = 256;
  const int64_t blocks = (chunks + threads - 1) / threads;
  auto* xs = static_cast<const uint16_t*>(x);
  auto* c = static_cast<uint8_t*>(codes);
  auto* s = static_cast<uint8_t*>(scales);
  switch (fmt) {
    case 0: mx_quant_rows_kernel<0><<<(unsigned)blocks, threads, 0, st>>>(xs, R, S, D, c, s); break;
    case 1: mx_quant_rows_kernel<1><<<(unsigned)blocks, threads, 0, st>>>(xs, R, S, D, c, s); break;
    default: mx_quant_rows_kernel<2><<<(unsigned)blocks, threads, 0, st>>>(xs, R, S, D, c, s); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_mx_quant_cols(const void* x, int BH, int S, int D, int fmt, void* codes, void* scales,
                                 cudaStream_t st) {
  const int Sp = (S + 127) / 128 * 128;
  dim3 grid(Sp / 128, BH);
  const size_t smem = (size_t)128 * D * 2;
  auto* xs = static_cast<const uint16_t*>(x);
  auto* c = static_cast<uint8_t*>(codes);
  auto* s = static_cast<uint8_t*>(scales);
  switch (fmt) {
    case 0: mx_quant_cols_kernel<0><<<grid, 256, smem, st>>>(xs, S, D, Sp, c, s); break;
    case 1: mx_quant_cols_kernel<1><<<grid, 256, smem, st>>>(xs, S, D, Sp, c, s); break;
    default: mx_quant_cols_kernel<2><<<grid, 256, smem, st>>>(xs, S, D, Sp, c, s); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_transpose_v(const void* v, void* vt, int BH, int S, int D, cudaStream_t st) {
  const int Sp = (S + 127) / 128 * 128;
  dim3 grid(Sp / 128, BH);
  transpose_v_kernel<<<grid, 256, (size_t)128 * D * 2, st>>>(static_cast<const uint16_t*>(v), S, D, Sp,
                                                             static_cast<uint16_t*>(vt));
  return cudaGetLastError();
}

}  // namespace fsa
