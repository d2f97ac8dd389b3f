// dsv_device.cuh — device-side building blocks for the sm_103a kernels.
//
// Inline PTX for mbarrier, TMA (cp.async.bulk.tensor), the 5th-generation
// tensor cores (tcgen05.mma with TMEM accumulators) and bounded waits that
// record an error instead of hanging.  Written from the public PTX ISA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsv.h"

namespace dsv {

// ---------------------------------------------------------------------------
// Device error word (one per device, owned by the API translation unit) and
// the per-launch control block passed by value to every kernel.
// ---------------------------------------------------------------------------
struct DeviceErr {
  unsigned int code;
  unsigned int info;
};
struct Ctl {
  DeviceErr* err;                    // device address of the error word
  unsigned long long wait_limit_ns;  // time limit of every bounded wait
};

// First error wins; `info` says which wait or which index.
__device__ __forceinline__ void set_error(const Ctl& c, unsigned int code, unsigned int info) {
  if (atomicCAS(&c.err->code, 0u, code) == 0u) {
    c.err->info = info;
  }
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// A waiting thread is suspended until the phase completes or this many
// nanoseconds pass, so that waiting warps take no issue slots from the warps
// they share a scheduler with; the bounded waits below re-check their limits
// after every return.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Lower bound of the time limit of a drain wait.  A drain wait (abort ==
// nullptr) waits for copies or MMAs this CTA has already issued, which finish
// without any other warp's help; a CTA must not exit, or free its TMEM, while
// they are in flight, so a short caller limit (dsv_set_wait_limit_ns) does not
// shorten these waits below this bound.
constexpr uint64_t kDrainLimitNs = 2000000000ull;

// Wait for the phase with parity `parity` of `bar` to complete.  Gives up
// (returns false) when `*abort` becomes non-zero or the per-device time
// limit passes; in the latter case it records DSV_ERR_TIMEOUT with `where`
// and raises `*abort` so that every other waiter in the CTA gives up too.
// abort == nullptr: a drain wait; only the time limit applies, and it is at
// least kDrainLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const Ctl& ctl,
                                          unsigned int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit =
      (abort == nullptr && ctl.wait_limit_ns < kDrainLimitNs) ? kDrainLimitNs : ctl.wait_limit_ns;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer() - t0 > limit || it > (1u << 30)) {
        set_error(ctl, DSV_ERR_TIMEOUT, where);
        if (abort != nullptr) *abort = 1;
        return false;
      }
    }
  }
}

// Warp-uniform variant: every lane of the warp waits and the result is the
// AND over the warp, so that .sync.aligned instructions after it are reached
// by all lanes or by none.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               const Ctl& ctl, unsigned int where) {
  bool ok = mbar_wait(bar, parity, abort, ctl, where);
  return __all_sync(0xffffffffu, ok) != 0;
}

// A wait costs a shared-memory round trip (~90 clocks measured) even when the
// phase is long complete.  Where the next wait is known early, its test is
// issued early (mbar_test, non-blocking) and consumed at the wait
// (mbar_wait_warp_tested), so the round trip overlaps other work.
__device__ __forceinline__ uint32_t mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok;
}
__device__ __forceinline__ bool mbar_wait_warp_tested(uint64_t* bar, uint32_t parity, uint32_t tested,
                                                      volatile int* abort, const Ctl& ctl, unsigned int where) {
  if (__all_sync(0xffffffffu, tested != 0u)) return true;
  return mbar_wait_warp(bar, parity, abort, ctl, where);
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Plain (untiled) bulk copy global -> shared; addresses and size multiples of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and MMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
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

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
// Fields: D format (bits 4-5) = F32, A format (7-9) = BF16, B format (10-12)
// = BF16, A major (15), B major (16) with 1 = MN-major, N>>3 (17-22),
// M>>4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  start/LBO/SBO are in
// bytes (encoded >> 4); bits 46-48 hold the fixed value 0b001; bits 61-63 the
// swizzle mode (2 = 128B).  Tiles are 1024-byte aligned, so base offset = 0.
// K-major operands: SBO = 1024 (8 rows x 128 B), LBO unused.  MN-major
// operands: LBO = distance between 64-element column chunks, SBO = 1024.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Shared-memory matrix descriptor without swizzle, K-major: the matrix is a
// grid of 8-row x 16-byte core matrices, each 128 contiguous bytes; LBO =
// bytes between core matrices adjacent along K, SBO = bytes between 8-row
// groups.  Start address 16-byte aligned.
__device__ __forceinline__ uint64_t sdesc_noswz(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Descriptor of the same matrix `byte_off` bytes further on.  The start
// address field holds (address >> 4) in 14 bits and shared-memory addresses
// stay below 2^18, so adding to the low bits never carries into LBO.  Used to
// keep the single MMA-issuing thread at a few instructions per MMA: the
// issue rate of tcgen05.mma from one thread is bounded by the scalar work
// between MMAs, not by the tensor core, when descriptors are rebuilt per MMA.
__device__ __forceinline__ uint64_t desc_off(uint64_t d, uint32_t byte_off) { return d + (uint64_t)(byte_off >> 4); }

// D[tmem] (+)= A[smem] * B[smem]  (both operands via descriptors)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Warp-wide forms of the three calls above: the whole warp runs the issuing
// code with converged control flow and elect.sync picks the one lane that
// issues, so descriptors and TMEM addresses are computed warp-uniformly.
// Measured on GB300: a converged warp issues one tcgen05.mma every ~35-48
// clocks, under the 64 clocks an M=128, N=128, K=16 MMA takes, while a single
// lane in a divergent branch needs ~100 clocks per MMA and starves the tensor
// core.  Every lane of the warp must call these together.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// TMEM -> registers: 32 lanes x 32 consecutive 32-bit columns (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// TMEM -> registers: 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// registers -> TMEM: 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// registers -> TMEM: 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// registers -> TMEM: 32 lanes x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// W consecutive columns (loads: W = 16, 32 or 64; stores: 8, 16 or 32) into /
// out of registers.
template <int W>
__device__ __forceinline__ void tmem_ld_w(uint32_t taddr, uint32_t* r) {
  static_assert(W == 16 || W == 32 || W == 64, "tmem_ld_w: W must be 16, 32 or 64");
  if constexpr (W == 64) {
    tmem_ld32(taddr, r);
    tmem_ld32(taddr + 32, r + 32);
  } else if constexpr (W == 32) {
    tmem_ld32(taddr, r);
  } else {
    tmem_ld16(taddr, r);
  }
}
template <int W>
__device__ __forceinline__ void tmem_st_w(uint32_t taddr, const uint32_t* r) {
  static_assert(W == 8 || W == 16 || W == 32, "tmem_st_w: W must be 8, 16 or 32");
  if constexpr (W == 32) tmem_st32(taddr, r); else if constexpr (W == 16) tmem_st16(taddr, r); else tmem_st8(taddr, r);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------
// Hardware base-2 exponential (MUFU.EX2), flush-to-zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs (Blackwell's two-wide fp32 FMA / add / mul): one
// instruction does the work of two, which matters in the issue-bound softmax.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (one instruction)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// The work items of a persistent CTA: rounds r = 0, 1, ... take item
// r * gridDim.x + blockIdx.x (with `snake`, odd rounds run the CTAs in reverse,
// so that a list sorted by decreasing cost spreads evenly).  Item idx is CSR
// row order[idx] (or idx itself); the row and its list bounds are read one
// item ahead, so the loads are off the critical path.
struct ItemCursor {
  const int32_t* ptr;
  const int32_t* order;
  long long items, r, row;
  int start, end;
  bool snake, valid;
  __device__ ItemCursor(const int32_t* p, const int32_t* ord, long long n, bool sn)
      : ptr(p), order(ord), items(n), r(0), row(0), start(0), end(0), snake(sn), valid(false) {
    load();
  }
  __device__ void load() {
    const long long pos = (snake && (r & 1)) ? (long long)(gridDim.x - 1 - blockIdx.x) : (long long)blockIdx.x;
    const long long idx = r * gridDim.x + pos;
    valid = idx < items;
    if (valid) {
      row = order != nullptr ? (long long)order[idx] : idx;
      start = ptr[row];
      end = ptr[row + 1];
    }
  }
  // the current item (false when there is none left); then fetch the next one
  __device__ bool next(long long& rw, int& st, int& cnt) {
    if (!valid) return false;
    rw = row;
    st = start;
    cnt = end - start;
    ++r;
    load();
    return true;
  }
};

// min of three (one instruction)
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The 1024-byte aligned start inside a dynamic shared-memory array, found by
// pointer arithmetic on the array itself, so that the compiler keeps accesses
// through it in the shared address space (ld/st/atom.shared); aligning through
// an integer round trip turns them into generic accesses.
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

template <typename T>
__device__ __forceinline__ T* align_up_ptr(void* p, uintptr_t a) {
  uintptr_t v = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<T*>((v + a - 1) & ~(a - 1));
}

// Where a wait gave up (detail word of DSV_ERR_TIMEOUT): kernel id << 8 | wait id.
enum : unsigned int {
  KID_FWD = 1,
  KID_BWD_KV = 2,
  KID_BWD_Q = 3,
  KID_MAXPOOL = 5,
};

}  // namespace dsv
