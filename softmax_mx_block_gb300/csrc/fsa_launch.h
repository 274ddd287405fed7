// fsa_launch.h -- host-side launch descriptors shared by the API and the kernel TUs.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "fsa_attn.cuh"

namespace fsa {

struct AttnLaunch {
  CUtensorMap tq, tk, tv, to;   // Q, K, V^T codes; fp32 output (32x32 boxes, or 16x32 when persistent)
  KParams p;
  DbgParams dbg;         // the debug instance's dump pointers (null otherwise)
  int D;
  int exp_mode;          // 0 poly, 1 MUFU, 2 split (ignored for EFQ and BF16)
  int persistent;        // 1: the persistent schedule (tq..to built for it), 0: one CTA per query tile
  int debug;             // 1: the debug instance (per-tile dumps into dbg)
  int q_fused;           // 1: tq maps bf16 Q, quantised in the kernel's prologue
  cudaStream_t stream;
};

// One explicit instantiation per (QK format, PV format) lives in its own
// translation unit (compiled in parallel); D and exp_mode dispatch inside.
template <int FQK, int FPV>
cudaError_t launch_attn_impl(const AttnLaunch& a);

cudaError_t launch_mx_quant_rows(const void* x, int BH, int S, int D, int fmt, void* codes, void* scales,
                                 cudaStream_t st);
cudaError_t launch_mx_quant_cols(const void* x, int BH, int S, int D, int fmt, void* codes, void* scales,
                                 cudaStream_t st);
cudaError_t launch_mx_quant_qkv(const void* q, const void* k, const void* v, int BHq, int BHk, int Sq, int Sk, int D,
                                int fqk, int fv, void* cq, void* sq, void* ck, void* sk, void* cv, void* sv,
                                cudaStream_t st);
cudaError_t launch_transpose_v(const void* v, void* vt, int BH, int S, int D, cudaStream_t st);

// Tensor-core throughput probe (fsa_peak.cu): kind 0 bf16, 1 MXFP8 E4M3, 2 MXFP4 E2M1.
double mma_peak_flops_per_iter(int kind, int n);
cudaError_t launch_mma_peak(int kind, int n, int n_ctas, long long iters, int* status, uint64_t timeout_ns,
                            cudaStream_t st);

}  // namespace fsa
