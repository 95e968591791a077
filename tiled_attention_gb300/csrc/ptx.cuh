// ptx.cuh — thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers (with time-bounded waits), TMA bulk tensor copies, and tcgen05 (TMEM allocation,
// MMA with TMEM accumulators, TMEM loads/stores). Nothing here allocates or frees memory.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only; the library does not link libcuda)

namespace ta {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Device status word shared by all kernels of the library (first error wins).
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Every pipeline wait goes through this: it gives up after `timeout_ns` of %globaltimer time
// or 2^26 polls, whichever comes first, or as soon as another role of the CTA has given up
// (shared abort flag). On giving up it records ATTN_ERR_TIMEOUT (-4) and returns false; the
// caller then leaves its loop so the CTA can still free its TMEM and exit.
struct WaitCtl {
  uint64_t timeout_ns;
  int* status;
  volatile int* abort_flag;  // shared memory; nullptr for drain waits that must not abort early
};

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t polls = 0; polls < (1u << 26); ++polls) {
    if (mbar_try_wait(bar, parity)) return true;
    if (w.abort_flag && *w.abort_flag) return false;
    if (global_timer_ns() - t0 > w.timeout_ns) break;
  }
  if (w.abort_flag) *w.abort_flag = 1;
  report_status(w.status, -4);
  return false;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Contiguous bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled bulk store shared -> global through a tensor map, tracked by bulk groups. Rows past
// the tensor's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Returns once every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Orders this thread's ordinary shared-memory writes before later TMA reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
// TMEM allocation is warp-collective; the allocated base address is written to *slot (smem).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The tcgen05 issue helpers below are called by a whole converged warp: the warp computes the
// (warp-uniform) operands together and one lane, chosen by elect.sync, issues the instruction.
// elect.sync picks the same lane every time for a full mask, so the commit that tracks a
// thread's MMAs runs on the lane that issued them.

// D[tmem] (+)= A[smem desc] * B[smem desc]; kind::f16 (bf16 inputs here), fp32 accumulate.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]; kind::f8f6f4 (E4M3 inputs here), fp32 accumulate.
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc].
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Eight SS MMAs of one accumulator chain from one elected lane: K = 8 steps of 16 columns of
// two K-major operands stored as 64-column 128-byte-swizzle panels kP16 x 16 bytes apart (a step
// is 32 bytes inside a panel row); the first step overwrites D.
template <uint32_t kP16>
__device__ __forceinline__ void mma_ss_chain8(uint32_t d_tmem, uint64_t a, uint64_t b,
                                              uint32_t idesc) {
  asm volatile(
      "{\n .reg .pred e, t, f;\n"
      " .reg .b64 a1, b1, a2, b2, a3, b3, a4, b4, a5, b5, a6, b6, a7, b7;\n"
      " setp.ne.b32 t, 1, 0;\n setp.ne.b32 f, 0, 0;\n"
      " add.s64 a1, %1, 2;\n add.s64 b1, %2, 2;\n add.s64 a2, %1, 4;\n add.s64 b2, %2, 4;\n"
      " add.s64 a3, %1, 6;\n add.s64 b3, %2, 6;\n add.s64 a4, %1, %4;\n add.s64 b4, %2, %4;\n"
      " add.s64 a5, a4, 2;\n add.s64 b5, b4, 2;\n add.s64 a6, a4, 4;\n add.s64 b6, b4, 4;\n"
      " add.s64 a7, a4, 6;\n add.s64 b7, b4, 6;\n"
      " elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, t;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "l"(static_cast<uint64_t>(kP16))
      : "memory");
}

// Eight TS MMAs of one accumulator chain from one elected lane: A from TMEM (8 columns per
// 16-key step), B an MN-major operand whose 16-key steps are 2048 bytes apart; the first step
// accumulates iff acc0 != 0.
__device__ __forceinline__ void mma_ts_chain8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                              uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n .reg .pred e, t, p;\n .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n"
      " .reg .b32 a1, a2, a3, a4, a5, a6, a7;\n"
      " setp.ne.b32 t, 1, 0;\n setp.ne.b32 p, %4, 0;\n"
      " add.s32 a1, %1, 8;\n add.s32 a2, %1, 16;\n add.s32 a3, %1, 24;\n add.s32 a4, %1, 32;\n"
      " add.s32 a5, %1, 40;\n add.s32 a6, %1, 48;\n add.s32 a7, %1, 56;\n"
      " add.s64 b1, %2, 128;\n add.s64 b2, %2, 256;\n add.s64 b3, %2, 384;\n"
      " add.s64 b4, %2, 512;\n add.s64 b5, %2, 640;\n add.s64 b6, %2, 768;\n"
      " add.s64 b7, %2, 896;\n"
      " elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, t;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc0)
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation the elected lane issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#include "tmem_io.inc"

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle (the layout a TMA load
// with CU_TENSOR_MAP_SWIZZLE_128B writes): start address, leading / stride byte offsets
// (16-byte units), descriptor version 1, layout type 2 (SWIZZLE_128B). The tile base must be
// 1024-byte aligned; advancing the start address inside a 128-byte row steps along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo_bytes,
                                               uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D: D format bits [4,6) = 1,
// A format [7,10) = 1, B format [10,13) = 1, A / B major-ness bits 15 / 16 (1 = MN-major),
// N >> 3 in [17,23), M >> 4 in [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with E4M3 A/B (format code 0) and fp32 D, both
// operands K-major; the other fields as in idesc_bf16.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Per-warpgroup register reallocation; every warp of the warpgroup must execute it. The sum
// over warpgroups must stay within the registers the block was launched with.
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace ta
