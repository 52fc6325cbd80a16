// Device-side building blocks for the sm_103a attention kernels: inline PTX for
// mbarriers, TMA bulk copies, tcgen05 (TMEM allocation, MMA, loads), bounded
// waits that report a timeout instead of hanging, and the Philox4x32-10
// generator used for in-kernel dropout.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// ---------------------------------------------------------------------------
// Device status word (its address travels in the kernel parameters). Kernels
// OR error bits into it; the host reads it back through
// fa_get_device_status(). A bounded wait that gives up sets kStatusTimeout and
// makes its CTA wind down instead of spinning forever.
// ---------------------------------------------------------------------------
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusBadLaunch = 2u;

// Wall-clock limit of one bounded wait (nanoseconds). Generous: a healthy wait
// lasts micro- to milliseconds.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// ----------------------------- mbarrier -----------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// One arrival worth `count` (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// A whole warp arrives as one operation worth 32: the lanes synchronise first
// (ordering each lane's earlier shared-memory and TMEM work before the
// release), then lane 0 arrives for all of them. Thirty-two single arrivals on
// one barrier serialise and cost about 200 cycles per warp.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_cnt(bar, 32);
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking probe of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Blocking waits let the hardware suspend the waiting warp (kPoll = false);
// polling waits spin on test_wait (kPoll = true), which wakes sooner at the
// cost of issue slots. Measured on the causal d=128 backward: polling in the
// row-math warps shortens the dK/dV kernel by ~2.5%, polling in the MMA-issuing
// warps (which share schedulers with row-math warps) lengthens it by ~5%.
constexpr bool kIssuerPoll = false;
constexpr bool kRowMathPoll = true;
// The warp that issues the MMAs consuming the row math's images (dV/dK, or the
// dQ / O accumulation) waits on the row math: its own choice.
constexpr bool kConsumerPoll = false;

// Returns false (after setting the timeout status bit and *abort) when the
// wall-clock limit passes or another role of the CTA has already aborted.
template <bool kPoll = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* status) {
  auto probe = [&]() { return kPoll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity); };
  if (probe()) return true;
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (probe()) return true;
    if ((spin & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(status, kStatusTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Every lane of the warp waits and the outcome is agreed on, so the warp leaves
// the wait together and converged (for the warp-wide issue forms below). Having
// lane 0 wait alone while the other lanes park at a shuffle measured twice as
// slow on the MMA-issuing warps.
template <bool kPoll = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* status) {
  const bool ok = mbar_wait<kPoll>(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
}

// ------------------------ packed fp32 pair arithmetic ------------------------
// The sm_100 family executes two fp32 lanes per instruction for add, mul and
// fma (.f32x2, round to nearest, no flush): bit-identical to the scalar forms,
// at half the issue slots. A pair is (lo, hi) in one 64-bit register.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Three-input maximum (one instruction on the sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------- TMA ---------------------------------------
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 4-D tiled load; c0 is the innermost (head-dim) coordinate and must be a
// multiple of 8 elements (16 bytes) — callers only pass 0 or 64.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// Plain bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// TMA tensor reduce-add: the box at tensor coordinates (c0, c1, c2) gains the
// box held in shared memory at src, element by element (fp32 add, performed at
// L2; concurrent reductions into the same elements from other CTAs are each
// applied atomically, in no defined order). c0 x element size must be a
// multiple of 16 bytes; src 128-byte aligned. Tracked by the bulk async-group
// of the issuing thread.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared-memory sources of this thread's committed bulk groups have been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's committed bulk groups have completed (their global writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// All but the most recently committed bulk group of this thread have completed.
__device__ __forceinline__ void bulk_wait_all_but_last() { asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); }
// Orders this thread's async-proxy global accesses (TMA) with its generic ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// A plain (relaxed) GPU-scope read for polling: it does not hold back this
// thread's later memory operations; acquire with fence_acq_rel_gpu once the
// value is the one waited for.
__device__ __forceinline__ unsigned int ld_relaxed_gpu(const unsigned int* ptr) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
// GPU-scope acquire-release fence: after relaxed reads, it acquires what they
// observed; before relaxed writes, it releases every earlier memory operation
// of this thread (one fence serves several flag stores).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_relaxed_gpu(unsigned int* ptr, unsigned int v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
// Wait that ignores the abort flag, used to let in-flight copies or MMAs land
// before a CTA that gave up exits. Also bounded.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned int* status) {
  unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout);
      return;
    }
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Make generic-proxy shared-memory writes visible to the async proxy (tcgen05.mma reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------ tcgen05 ------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
// Arrive once on the barrier when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 or fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A is M lanes x K, two 16-bit values per column.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-wide forms of the three issue operations: every lane of a converged
// warp executes them and elect.sync lets one lane (the lowest, the same one
// each time, so commits track that lane's MMAs) issue. Keeping the issuing
// warp converged keeps its descriptor arithmetic warp-uniform, which cuts the
// issue cost of an MMA from about 60 to about 25 cycles, and to well under half
// when busy row-math warps compete for the same scheduler.
__device__ __forceinline__ void tc_mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// ------------------------- CTA pairs (cta_group::2) -------------------------
// Store 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
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
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 8 consecutive 32-bit columns of this thread's lane from r[off .. off+8).
template <int off, int n>
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[n]) {
  static_assert(off + 8 <= n, "range");
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[off]), "r"(r[off + 1]), "r"(r[off + 2]), "r"(r[off + 3]), "r"(r[off + 4]), "r"(r[off + 5]),
               "r"(r[off + 6]), "r"(r[off + 7])
               : "memory");
}

// Writes the split image of 32 elements (see interleave_split) to the 32
// columns at taddr: rounded pairs r, residual pairs e.
__device__ __forceinline__ void tmem_st_split(uint32_t taddr, const uint32_t (&r)[16], const uint32_t (&e)[16]) {
  tmem_st8<0>(taddr, r);
  tmem_st8<0>(taddr + 8, e);
  tmem_st8<8>(taddr + 16, r);
  tmem_st8<8>(taddr + 24, e);
}

// TMEM image of a 16-bit MMA operand split into a rounded part and a residual:
// per 16-element K step, 8 columns of rounded values followed by 8 columns of
// residuals. A chunk of 32 elements therefore occupies exactly the 32 columns
// its fp32 source occupied. Given the packed rounded (r) and residual (e)
// pairs of 32 elements, builds that 32-column image.
__device__ __forceinline__ void interleave_split(const uint32_t (&r)[16], const uint32_t (&e)[16],
                                                 uint32_t (&out)[32]) {
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    out[x] = r[x];
    out[8 + x] = e[x];
    out[16 + x] = r[8 + x];
    out[24 + x] = e[8 + x];
  }
}

// Bits x of [lo, hi), clamped to [0, 32).
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > 32 ? 32 : hi;
  if (hi <= lo) return 0u;
  const uint32_t upper = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  return upper & (0xFFFFFFFFu << lo);
}

// Instruction descriptor for kind::f16 with an fp32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (0 = f16, 1 = bf16),
//   15 / 16 A / B major (0 = K-major, 1 = MN-major), 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool bf16, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle, tcgen05 version bits.
//   bits 0-13 start>>4, 16-29 leading byte offset>>4, 32-45 stride byte offset>>4,
//   46-47 version (1), 61-63 layout (2 = 128B swizzle).
// K-major operands: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO); the
// leading offset is unused. MN-major operands: 64-element MN groups LBO bytes
// apart, 8-row K groups SBO = 1024 bytes apart.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Shared-memory descriptor advanced by a byte offset (the start address field
// is the low 14 bits of the descriptor, in 16-byte units; shared addresses stay
// below 2^18 bytes, so the addition never carries out of that field).
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// 32 lanes x 32 consecutive 32-bit columns; thread t of the warp gets lane (base lane + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Wait for one outstanding 16-column load.
__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&a)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15])
               :
               : "memory");
}
// Wait for two outstanding 16-column loads (registers tied in, as below).
__device__ __forceinline__ void tmem_ld_wait16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}
// Wait for three outstanding 16-column loads.
__device__ __forceinline__ void tmem_ld_wait16x3(uint32_t (&a)[16], uint32_t (&b)[16], uint32_t (&c)[16]) {
  tmem_ld_wait16x2(a, b);
  asm volatile(""
               : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]), "+r"(c[4]), "+r"(c[5]), "+r"(c[6]), "+r"(c[7]),
                 "+r"(c[8]), "+r"(c[9]), "+r"(c[10]), "+r"(c[11]), "+r"(c[12]), "+r"(c[13]), "+r"(c[14]),
                 "+r"(c[15])
               :
               : "memory");
}
// Wait for four outstanding 16-column loads.
__device__ __forceinline__ void tmem_ld_wait16x4(uint32_t (&a)[16], uint32_t (&b)[16], uint32_t (&c)[16],
                                                 uint32_t (&d)[16]) {
  tmem_ld_wait16x3(a, b, c);
  asm volatile(""
               : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3]), "+r"(d[4]), "+r"(d[5]), "+r"(d[6]), "+r"(d[7]),
                 "+r"(d[8]), "+r"(d[9]), "+r"(d[10]), "+r"(d[11]), "+r"(d[12]), "+r"(d[13]), "+r"(d[14]),
                 "+r"(d[15])
               :
               : "memory");
}

// Wait for outstanding tcgen05.ld; the registers are tied in so that no use of
// them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                 "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                 "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                 "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait2(uint32_t (&a)[32], uint32_t (&b)[32]) {
  tmem_ld_wait(a);
  asm volatile(""
               : "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]),
                 "+r"(b[13]), "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]),
                 "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]), "+r"(b[24]),
                 "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]),
                 "+r"(b[31])
               :
               : "memory");
}

// ------------------------------ math ---------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Round two fp32 values to a packed pair of 16-bit floats (round to nearest even).
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (kBf16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// Widen a packed pair of 16-bit floats back to fp32 (exact).
template <bool kBf16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (kBf16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  } else {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
  }
}

// Rounding residual of a packed pair: lo/hi parts v - widen(round(v)), packed.
// A 16-bit MMA operand split as round(v) + residual carries ~16 significant bits.
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2_residual(float a, float b, uint32_t rounded) {
  float ra, rb;
  unpack2<kBf16>(rounded, ra, rb);
  return pack2<kBf16>(a - ra, b - rb);
}

// Probability above which a tile's P (and dS) are split into two 16-bit parts.
// Rounding an operand to 16 bits moves it by up to 2^-8 of itself, so below the
// threshold each product P*x moves by at most 2^-14*|x|; above it the residual
// tile restores ~16 significant bits.
constexpr float kSplitThreshold = 1.0f / 64.0f;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// ------------------------------ Philox -------------------------------------
// Philox-4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): per round two
// 32x32->64 multiplies, the output permutation of that paper, and a Weyl key
// schedule between rounds.
// 32 x 32 -> 64-bit product as one instruction (low word, high word).
__device__ __forceinline__ void mul_wide_u32(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b64 t;\n\tmul.wide.u32 t, %2, %3;\n\tmov.b64 {%0, %1}, t;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(a), "r"(b));
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide_u32(0xD2511F53u, c.x, lo0, hi0);
    mul_wide_u32(0xCD9E8D57u, c.z, lo1, hi1);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

struct DropoutParams {
  uint32_t on;         // dropout enabled (dropout_p > 0)
  uint32_t threshold;  // keep iff a 16-bit value >= threshold = floor(p * 2^16)
  float rp;            // 1 / (1 - p)
  uint32_t seed_lo, seed_hi, off_lo, off_hi;
  uint32_t bh_off;     // added to the launch's (batch * H + head) index: a launch over a
                       // slice of the heads or batches draws the full problem's masks
};

// Dropout keep decisions. One Philox call serves eight consecutive keys of one
// query: key 8q + 2w + h takes 16-bit half h (low for even keys) of output word
// w, at counter (g, offset) with g = (bh * N + i) * ceil(N/8) + q, and is kept
// iff that half >= threshold.

// The eight keep bits of one Philox output (bit 2w + h <-> half h of word w).
// With T16 = T << 16: the high half of x is >= T iff x >= T16, and the low half
// iff (x << 16) >= T16 (unsigned), so each decision is one compare.
__device__ __forceinline__ uint32_t keep_byte(uint4 w, uint32_t T) {
  const uint32_t T16 = T << 16;
  return (uint32_t)((w.x << 16) >= T16) | ((uint32_t)(w.x >= T16) << 1) | ((uint32_t)((w.y << 16) >= T16) << 2) |
         ((uint32_t)(w.y >= T16) << 3) | ((uint32_t)((w.z << 16) >= T16) << 4) | ((uint32_t)(w.z >= T16) << 5) |
         ((uint32_t)((w.w << 16) >= T16) << 6) | ((uint32_t)(w.w >= T16) << 7);
}

__device__ __forceinline__ uint4 philox_at(const DropoutParams& dp, uint64_t g) {
  return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), dp.off_lo, dp.off_hi), dp.seed_lo, dp.seed_hi);
}

// Keep decision for element (bh, i, j) of an N x N head.
__device__ __forceinline__ bool dropout_keep(const DropoutParams& dp, uint32_t bh, int N, int i, int j) {
  const uint64_t n8 = (uint64_t)((N + 7) >> 3);
  const uint4 w = philox_at(dp, ((uint64_t)(bh + dp.bh_off) * (uint64_t)N + (uint64_t)i) * n8 + (uint64_t)(j >> 3));
  const int ww = (j >> 1) & 3;
  const uint32_t word = ww == 0 ? w.x : ww == 1 ? w.y : ww == 2 ? w.z : w.w;
  return ((j & 1) ? (word >> 16) : (word & 0xFFFFu)) >= dp.threshold;
}

// Keep bits (bit x <-> query i0 + x) of 32 consecutive queries for this lane's
// key j, computed by the whole (converged) warp, whose lanes hold 32
// consecutive keys with j % 8 == lane % 8. One Philox call yields the bits of
// eight keys (one 8-lane group) for one query, so lane 8g + r evaluates the
// queries i0 + 8t + r (t < 4) for its group and the eight lanes trade their
// results through shuffles: 4 calls per lane instead of 32.
static __device__ __forceinline__ uint32_t keep_bits_for_key(const DropoutParams dp, uint32_t bh, int N, int i0, int j) {
  const int lane = threadIdx.x & 31, r = lane & 7;
  const uint64_t n8 = (uint64_t)((N + 7) >> 3);
  const uint64_t row0 = (uint64_t)(bh + dp.bh_off) * (uint64_t)N;
  uint32_t mine = 0;  // byte t: keep bits of the group's eight keys for query i0 + 8t + r
#pragma unroll
  for (int t = 0; t < 4; ++t)
    mine |= keep_byte(philox_at(dp, (row0 + (uint64_t)(i0 + 8 * t + r)) * n8 + (uint64_t)(j >> 3)), dp.threshold)
            << (8 * t);
  // From lane 8g + rs, this lane (8g + r) needs bit r of each byte t (the
  // queries i0 + 8t + rs), placed at bit 8t + rs: one shift brings bit r of
  // every byte to the byte's bit 0, one mask keeps those four, one shift
  // moves them to bit rs.
  uint32_t bits = 0;
#pragma unroll
  for (int rs = 0; rs < 8; ++rs) {
    const uint32_t v = __shfl_sync(0xffffffffu, mine, (lane & ~7) + rs);
    bits |= ((v >> r) & 0x01010101u) << rs;
  }
  return bits;
}

// Keep bits (bit x <-> key j0 + x) of 32 consecutive keys for one query i;
// j0 % 8 == 0, so each Philox call yields the bits of eight keys.
static __device__ __noinline__ uint32_t keep_bits_for_query(const DropoutParams dp, uint32_t bh, int N, int i, int j0) {
  const uint64_t n8 = (uint64_t)((N + 7) >> 3);
  const uint64_t g0 = ((uint64_t)(bh + dp.bh_off) * (uint64_t)N + (uint64_t)i) * n8 + (uint64_t)(j0 >> 3);
  uint32_t bits = 0;
#pragma unroll
  for (int x = 0; x < 4; ++x) bits |= keep_byte(philox_at(dp, g0 + (uint64_t)x), dp.threshold) << (8 * x);
  return bits;
}

}  // namespace fa
