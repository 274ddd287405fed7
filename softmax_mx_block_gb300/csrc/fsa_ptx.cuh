// fsa_ptx.cuh -- inline-PTX building blocks for sm_103a: mbarriers with bounded
// waits, TMA tile and bulk copies, and the tcgen05 tensor-core / tensor-memory
// instructions.  Layout facts used here (shared-memory matrix descriptors,
// instruction descriptors, scale-factor placement in tensor memory) follow the
// PTX ISA for tcgen05 and were checked on the device with small in-bounds MMAs.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fsa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               " selp.b32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Non-blocking test of phase `parity` (never suspends the thread).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               " selp.b32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// As above, but the thread may sleep up to `hint_ns` inside the instruction (it
// resumes as soon as the phase completes), so a waiting warp issues few polls.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
               " selp.b32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// Shared-memory scalars through explicit .shared accesses (a generic pointer to a
// volatile would become a system-scope load or store).  Ordering against other
// threads comes from the named barriers and mbarriers around them.
__device__ __forceinline__ int lds_vol(const int* p) {
  int v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void sts_vol(int* p, int v) {
  asm volatile("st.volatile.shared.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ float lds_f32(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(float* p, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(smem_u32(p)), "f"(v) : "memory");
}

// Shared abort state of one CTA: once any wait gives up, every later wait of
// the CTA returns false at once so that all roles drain and reach teardown.
struct AbortCtl {
  int* flag;               // shared memory (lds_vol / sts_vol)
  int* status;             // global status word (may be null)
  uint64_t limit_ns;
};

// Wait for phase `parity` of `bar`; false if the limit passed or the CTA aborted.
// SLEEP lets the thread doze inside each poll (few issue slots taken from the
// warps it shares a scheduler with); the latency-critical waits poll without it.
template <bool SLEEP = true>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const AbortCtl& ac) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (SLEEP ? mbar_try_wait_sleep(bar, parity, 20000u) : mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 0) {
      if (lds_vol(ac.flag)) return false;
      if (globaltimer_ns() - t0 > ac.limit_ns) {
        sts_vol(ac.flag, 1);
        if (ac.status) atomicExch(ac.status, -4);   // FSA_ERR_TIMEOUT
        return false;
      }
    }
  }
}

// Wait that ignores the CTA abort flag (teardown: drain work still in flight).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Teardown wait for work this CTA still has in flight (copies, MMAs).  On expiry the
// CTA is marked aborted and the status word gets FSA_ERR_TIMEOUT, so the caller
// learns that the teardown was not clean (the output is then undefined).
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, const AbortCtl& ac) {
  if (mbar_wait_drain(bar, parity, ac.limit_ns)) return true;
  sts_vol(ac.flag, 1);
  if (ac.status) atomicExch(ac.status, -4);   // FSA_ERR_TIMEOUT
  return false;
}

// One lane of a converged warp (the lowest active one) gets true.  The tcgen05
// issuing warp runs converged and elects its issuing lane per instruction.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.b32 %0, 1, 0, p;\n}" : "=r"(e));
  return e != 0;
}

// 1 in the elected lane of a converged warp, else 0 (a value for the predicated
// forms below, so no branch diverges the warp)
__device__ __forceinline__ uint32_t elect_u32() {
  uint32_t e;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.b32 %0, 1, 0, p;\n}" : "=r"(e));
  return e;
}
// mbarrier arrive by the elected lane only (whole warp converged)
__device__ __forceinline__ void mbar_arrive_elect(uint64_t* bar) {
  asm volatile("{\n .reg .pred e;\n .reg .b64 st;\n elect.sync _|e, 0xffffffff;\n"
               " @e mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------- TMA / bulk
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z) : "memory");
}
// Tiled store shared -> global (bulk async group); x must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* smem_src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(tmap), "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every bulk store of this thread's groups has been performed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Wait until every bulk store of this thread's groups has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the most recent bulk group have finished reading their shared memory
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Untiled bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrive on named barrier `id` without waiting (the producer side of a handoff).
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(slot_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Copy a 512-byte 128x4 scale atom (32 lines of 16 bytes) from shared memory
// into 4 tensor-memory columns, replicated in all four lane quadrants:
// lane 32q+r, column c receives line r bytes 4c..4c+3.
__device__ __forceinline__ void tc_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, BF16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem)^T, BF16.
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// Block-scaled, 8/6/4-bit elements (one scale per 32 K per MMA, K = 32).
__device__ __forceinline__ void mma_mxf8f6f4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
               "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_mxf8f6f4_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
               "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
}
// Block-scaled packed E2M1 (two scales per MMA, K = 64).
__device__ __forceinline__ void mma_mxf4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
               "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_mxf4_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
               "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc) : "memory");
}

// Predicated forms: issued only where e != 0 (the warp stays converged).
__device__ __forceinline__ void tc_commit_p(uint32_t e, uint64_t* bar) {
  asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %1, 0;\n"
               "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}"
               ::"r"(smem_u32(bar)), "r"(e) : "memory");
}
__device__ __forceinline__ void tc_cp_sf_atom_p(uint32_t e, uint32_t taddr, uint64_t sdesc) {
  asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n"
               "@q tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n}" ::"r"(taddr), "l"(sdesc), "r"(e) : "memory");
}
__device__ __forceinline__ void mma_f16_ss_p(uint32_t e, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(e) : "memory");
}
__device__ __forceinline__ void mma_f16_ts_p(uint32_t e, uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(e) : "memory");
}
__device__ __forceinline__ void mma_mxf8f6f4_ss_p(uint32_t e, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                  uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %6, 0;\n setp.ne.b32 q, %7, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(e) : "memory");
}
__device__ __forceinline__ void mma_mxf8f6f4_ts_p(uint32_t e, uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                  uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %6, 0;\n setp.ne.b32 q, %7, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(e) : "memory");
}
__device__ __forceinline__ void mma_mxf4_ss_p(uint32_t e, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %6, 0;\n setp.ne.b32 q, %7, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(e) : "memory");
}
// kind::mxf4nvf4 with scale_vec::2X and E8M0 scales: the same MXFP4 operands (E2M1,
// one scale per 32 elements) through the NVFP4-capable instruction kind.
__device__ __forceinline__ void mma_mxf4nvf4_ss_p(uint32_t e, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                  uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %6, 0;\n setp.ne.b32 q, %7, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(e) : "memory");
}
__device__ __forceinline__ void mma_mxf4_ts_p(uint32_t e, uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %6, 0;\n setp.ne.b32 q, %7, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(e) : "memory");
}

// kind::mxf4nvf4 with scale_vec::4X: E2M1 operands, one scale byte per 16 elements
// (four per row per K = 64 step, the whole 32-bit scale word; with UE4M3 scales for
// NVFP4, descriptor bit 23 clear).
__device__ __forceinline__ void mma_nvf4_4x_ss_p(uint32_t e, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                 uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n .reg .pred p, q;\n setp.ne.b32 p, %6, 0;\n setp.ne.b32 q, %7, 0;\n"
               "@q tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc), "r"(e) : "memory");
}

// Shared-memory matrix descriptor: start address, stride between 8-row core
// groups (sbo), leading offset (lbo, unused for K-major swizzled tiles),
// descriptor version 1 (bit 46), swizzle code in bits 61-63
// (0 none, 2 = 128B, 4 = 64B, 6 = 32B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

// Instruction descriptors (M = 128, fp32 accumulator).
__host__ __device__ constexpr uint32_t idesc_f16_bf16(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
// Block-scaled: a/b element codes (mxf8f6f4: E4M3 0, E2M3 3, E2M1 5; mxf4: E2M1 1),
// E8M0 scales (bit 23), scale byte selectors sfa_id (bits 29-30), sfb_id (bits 4-5).
__host__ __device__ constexpr uint32_t idesc_bs(int N, uint32_t ab_fmt, uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(128 >> 4) << 24) | (sfa_id << 29);
}
// NVFP4 (kind::mxf4nvf4, scale_vec::4X): E2M1 a/b (1), UE4M3 scales (bit 23 clear),
// the whole scale word of each row per instruction (selectors 0).
__host__ __device__ constexpr uint32_t idesc_nvfp4(int N) { return idesc_bs(N, 1, 0, 0) & ~(1u << 23); }

// tcgen05.ld / st, 32 lanes x 32 bits, N consecutive columns per thread.
template <int N> struct TmemLd;
#define FSA_TMEM_LD(N, REGS, ...)                                                            \
  template <> struct TmemLd<N> {                                                             \
    __device__ __forceinline__ static void run(uint32_t taddr, uint32_t* r) {                \
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x" #N ".b32 {" REGS "}, [%" #N "];"       \
                   : __VA_ARGS__ : "r"(taddr) : "memory");                                   \
    }                                                                                        \
  };
FSA_TMEM_LD(1, "%0", "=r"(r[0]))
FSA_TMEM_LD(4, "%0,%1,%2,%3", "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]))
FSA_TMEM_LD(8, "%0,%1,%2,%3,%4,%5,%6,%7", "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
            "=r"(r[5]), "=r"(r[6]), "=r"(r[7]))
FSA_TMEM_LD(16, "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15", "=r"(r[0]), "=r"(r[1]), "=r"(r[2]),
            "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]),
            "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]))
#undef FSA_TMEM_LD

template <int N> struct TmemSt;
#define FSA_TMEM_ST(N, REGS, ...)                                                            \
  template <> struct TmemSt<N> {                                                             \
    __device__ __forceinline__ static void run(uint32_t taddr, const uint32_t* r) {          \
      asm volatile("tcgen05.st.sync.aligned.32x32b.x" #N ".b32 [%0], {" REGS "};"            \
                   ::"r"(taddr), __VA_ARGS__ : "memory");                                    \
    }                                                                                        \
  };
FSA_TMEM_ST(1, "%1", "r"(r[0]))
FSA_TMEM_ST(4, "%1,%2,%3,%4", "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]))
FSA_TMEM_ST(8, "%1,%2,%3,%4,%5,%6,%7,%8", "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
            "r"(r[6]), "r"(r[7]))
FSA_TMEM_ST(16, "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16", "r"(r[0]), "r"(r[1]), "r"(r[2]),
            "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
            "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]))
#undef FSA_TMEM_ST

// 32 consecutive columns of the thread's lane, and their maximum (tcgen05.ld.red:
// the reduction runs over the columns each thread loads).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t* r, float& m) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
      : "r"(taddr) : "memory");
}

// NCOLS consecutive columns (8, or a multiple of 16).
template <int NCOLS>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (NCOLS >= 16) {
#pragma unroll
    for (int c = 0; c < NCOLS; c += 16) TmemLd<16>::run(taddr + c, r + c);
  } else {
    TmemLd<NCOLS>::run(taddr, r);
  }
}
template <int NCOLS>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  if constexpr (NCOLS >= 16) {
#pragma unroll
    for (int c = 0; c < NCOLS; c += 16) TmemSt<16>::run(taddr + c, r + c);
  } else {
    TmemSt<NCOLS>::run(taddr, r);
  }
}

// ------------------------------------------------------------- conversions
// Two fp32 -> packed codes; `lo` lands in the low byte / nibble.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e2m3x2(float lo, float hi) {   // each code in a byte, low 6 bits
  uint16_t r;
  asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e3m2x2(float lo, float hi) {   // each code in a byte, low 6 bits
  uint16_t r;
  asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {   // one byte, lo in the low nibble
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack 16 six-bit codes (one per byte in w[0..3], little-endian) into 12 bytes
// (least significant bit first) in out[0..2]; the 16-byte group's last word is 0.
__device__ __forceinline__ void pack6x16(const uint32_t* w, uint32_t* out) {
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t u = (w[i] & 0x003F003Fu) | ((w[i] & 0x3F003F00u) >> 2);   // 12-bit pairs at bits 0, 16
    p[i] = (u & 0xFFFu) | ((u >> 4) & 0xFFF000u);                        // 24 bits
  }
  out[0] = p[0] | (p[1] << 24);
  out[1] = (p[1] >> 8) | (p[2] << 16);
  out[2] = (p[2] >> 16) | (p[3] << 8);
}

}  // namespace fsa
