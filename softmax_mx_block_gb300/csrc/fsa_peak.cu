// fsa_peak.cu -- dense tensor-core throughput probe: the roofline denominator of
// the attention kernels, measured with the MMA shapes they issue.
//
// The Fused-Softmax brief (abstract) quotes MXFP8 / MXFP6 / MXFP4 attention
// throughputs against the block-scaled matrix cores; this probe measures what
// those cores deliver on this GPU.  One CTA per SM keeps operand tiles resident in
// shared memory and scale factors in tensor memory and issues `iters` MMAs of
// M = 128 and N = 128 (the attention kernel's score MMA; three accumulators in
// rotation) or N = 256 (one accumulator) from one elected thread, SS form, K-major
// swizzled tiles.  At N = 128 an MXFP4 MMA reads 8 KB of shared memory per 2 MFLOP,
// which is near the shared-memory bandwidth; N = 256 halves the A traffic per FLOP:
//   kind 0  kind::f16, bf16 x bf16,                         K = 16 per MMA
//   kind 1  kind::mxf8f6f4 block_scale scale_vec::1X, E4M3, K = 32 per MMA
//   kind 2  kind::mxf4 block_scale scale_vec::2X, E2M1,     K = 64 per MMA
//   kind 3  kind::mxf4nvf4 block_scale scale_vec::2X, E2M1 with E8M0 scales (the
//           same MXFP4 operands through the NVFP4-capable kind), K = 64 per MMA
// The operand bytes are a fixed finite pattern (values do not change the
// instruction rate); scales are 2^0.  The final commit is awaited with a bounded
// wait; on expiry the status word gets FSA_ERR_TIMEOUT.
#include <cstdint>
#include <cuda_runtime.h>
#include "fsa_launch.h"

namespace fsa {

namespace {

constexpr int kPeakThreads = 128;
constexpr int kTileBytes = 128 * 256;       // A: 128 rows of up to 256 bytes (bf16, K = 128)
constexpr int kOffA = 0, kOffB = kTileBytes, kOffSF = kOffB + 2 * kTileBytes, kOffBar = kOffSF + 1024;
// more shared memory than two CTAs could share, so that each CTA (and its 512
// tensor-memory columns) has an SM to itself
constexpr int kPeakSmem = 120 * 1024;   // B: up to 256 rows of 256 bytes
static_assert(kOffBar + 64 + 1024 <= kPeakSmem, "shared memory");

template <int KIND, int N>
__global__ void __launch_bounds__(kPeakThreads, 1) fsa_mma_peak_kernel(long long iters, int* status,
                                                                       uint64_t timeout_ns) {
  // bytes per operand row (K = 128 elements) and the swizzle atom of the tiles
  constexpr int RB = KIND == 0 ? 256 : (KIND == 1 ? 128 : 64);   // kinds 2, 3: packed E2M1
  constexpr int W = RB < 128 ? RB : 128;
  constexpr int STEPS = RB / 32;            // 32 bytes of K per MMA
  constexpr uint32_t SWZ = W == 128 ? 2u : 4u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBar + 8);
  uint64_t* done = reinterpret_cast<uint64_t*>(sm + kOffBar);
  const int warp = threadIdx.x >> 5;
  // finite operand bytes (every byte <= 0x3F: no E4M3 NaN, bf16 magnitudes < 2) and
  // scale atoms of 2^0
  for (int i = threadIdx.x; i < 3 * kTileBytes / 4; i += kPeakThreads) {
    uint32_t h = (uint32_t)i * 0x9E3779B1u;
    h ^= h >> 15;
    reinterpret_cast<uint32_t*>(sm)[i] = h & 0x3F3F3F3Fu;
  }
  for (int i = threadIdx.x; i < 256; i += kPeakThreads) reinterpret_cast<uint32_t*>(sm + kOffSF)[i] = 0x7F7F7F7Fu;
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = __shfl_sync(0xffffffffu, *tmem_slot, 0);
  if (warp == 0) {
    const uint32_t sA = smem_u32(sm + kOffA), sB = smem_u32(sm + kOffB);
    constexpr uint32_t T_SFA = 400, T_SFB = 404;
    if constexpr (KIND != 0) {
      tc_cp_sf_atom_p(elect_u32(), tbase + T_SFA, smem_desc(smem_u32(sm + kOffSF), 16, 128, 0));
      tc_cp_sf_atom_p(elect_u32(), tbase + T_SFB, smem_desc(smem_u32(sm + kOffSF + 512), 16, 128, 0));
    }
    // N = 128: accumulators at columns 0, 128, 256; N = 256: one at column 0 (the scale
    // columns 400..411 stay clear of both)
    constexpr int NACC = N == 128 ? 3 : 1;
    int acc_buf = 0;
    for (long long it = 0; it < iters; ++it) {
      const uint32_t d = tbase + 128u * (uint32_t)acc_buf;
#pragma unroll
      for (int i = 0; i < STEPS; ++i) {
        const int ka = (i * 32) / W, off = (i * 32) % W;
        const uint64_t ad = smem_desc(sA + ka * 128 * W + off, 16, 8 * W, SWZ);
        const uint64_t bd = smem_desc(sB + ka * N * W + off, 16, 8 * W, SWZ);
        const uint32_t acc = (it >= NACC || i > 0) ? 1u : 0u;
        const uint32_t e = elect_u32();
        if constexpr (KIND == 0) {
          mma_f16_ss_p(e, d, ad, bd, idesc_f16_bf16(N), acc);
        } else if constexpr (KIND == 1) {
          mma_mxf8f6f4_ss_p(e, d, ad, bd, idesc_bs(N, 0, i, i), tbase + T_SFA, tbase + T_SFB, acc);
        } else if constexpr (KIND == 2) {
          mma_mxf4_ss_p(e, d, ad, bd, idesc_bs(N, 1, 2 * i, 2 * i), tbase + T_SFA, tbase + T_SFB, acc);
        } else {
          mma_mxf4nvf4_ss_p(e, d, ad, bd, idesc_bs(N, 1, 2 * i, 2 * i), tbase + T_SFA, tbase + T_SFB, acc);
        }
      }
      acc_buf = acc_buf == NACC - 1 ? 0 : acc_buf + 1;
    }
    tc_commit_p(elect_u32(), done);
    // every MMA of this warp has completed before tensor memory is freed
    if (!__all_sync(0xffffffffu, mbar_wait_drain(done, 0, timeout_ns)) && threadIdx.x == 0 && status)
      atomicExch(status, -4);   // FSA_ERR_TIMEOUT
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace

double mma_peak_flops_per_iter(int kind, int n) {
  // 2 * M * N * K per iteration (its MMAs cover K = 128 elements)
  return 2.0 * 128.0 * (double)n * 128.0;
}

cudaError_t launch_mma_peak(int kind, int n, int n_ctas, long long iters, int* status, uint64_t timeout_ns,
                            cudaStream_t st) {
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem);
    if (e != cudaSuccess) return e;
    kern<<<n_ctas, kPeakThreads, kPeakSmem, st>>>(iters, status, timeout_ns);
    return cudaGetLastError();
  };
  if (n == 256) {
    if (kind == 0) return run(fsa_mma_peak_kernel<0, 256>);
    if (kind == 1) return run(fsa_mma_peak_kernel<1, 256>);
    if (kind == 2) return run(fsa_mma_peak_kernel<2, 256>);
    return run(fsa_mma_peak_kernel<3, 256>);
  }
  if (kind == 0) return run(fsa_mma_peak_kernel<0, 128>);
  if (kind == 1) return run(fsa_mma_peak_kernel<1, 128>);
  if (kind == 2) return run(fsa_mma_peak_kernel<2, 128>);
  return run(fsa_mma_peak_kernel<3, 128>);
}

}  // namespace fsa
