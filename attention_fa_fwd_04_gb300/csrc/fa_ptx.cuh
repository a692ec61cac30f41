// fa_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA tensor
// loads, tcgen05 (TMEM alloc, MMA, commit, TMEM load/store, fences),
// mma.sync / ldmatrix, and bounded pipeline waits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// ---------------------------------------------------------------------------
// Device error word: bit 0 = a pipeline wait timed out; bits 8.. = which wait.
// ---------------------------------------------------------------------------
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrBounds = 2u;  // a global store index failed its self-check
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // default: 2 s per wait

// Time limit of a pipeline wait (mbar_wait), per device and per translation
// unit that includes this header (each kernel file has its own copy, set
// through that file's setter).  It lives in constant memory: a wait reads it
// from the constant cache, and kernels launched after the host writes it see
// the new value.  Teardown waits (mbar_wait_drain) keep the fixed
// kWaitTimeoutNs, so that loads already in flight always land before a CTA
// exits, whatever this limit is.  A limit below kWatchdogNs is a watchdog: the
// waits check the clock at every probe (see mbar_wait for when they start).
constexpr unsigned long long kWatchdogNs = 1000000ull;  // 1 ms
static __constant__ unsigned long long g_wait_limit_ns = kWaitTimeoutNs;

// Host side: set this translation unit's copy on the current device
// (0 restores the default).  Synchronous.  Returns a cudaError_t.
static inline int set_wait_limit_this_unit(unsigned long long ns) {
  const unsigned long long v = ns ? ns : kWaitTimeoutNs;
  return (int)cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof(v));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31) == 0; }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Test of the phase that may suspend the thread for a short, system-defined
// time while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the completion of the phase with the given parity.  Gives up after
// g_wait_limit_ns (or as soon as another warp of the CTA gave up), records the
// failure in *err_word and the CTA-wide abort flag, and returns false.
//
// POLL = false (prefill and backward): each probe is a try_wait, which
// suspends the thread for a short system-defined time (about 4 us measured
// on GB300) while the phase is incomplete; the clock and the abort flag are
// read every 64 probes, or at every probe after the first two under a
// watchdog limit, so a watchdog trips only waits longer than about two
// suspends.  The code is kept this small because it is inlined at every wait
// of the MMA-issuing warp, whose instruction stream paces those kernels:
// larger waits (a separate polling loop, a predicated probe, a suspend-time
// hint) measured 1-9 % slower.
// POLL = true (decode, bandwidth-bound): the first probe does not block, and
// under a watchdog limit every probe is a non-blocking test followed by a
// look at the clock and the abort flag, so a watchdog trips any wait that
// outlasts it.
template <bool POLL = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, unsigned int* err_word,
                                          unsigned int site) {
  const uint32_t a = smem_u32(bar);
  if constexpr (POLL) {
    if (mbar_test_wait(a, parity)) return true;
  } else {
    if (mbar_try_wait(a, parity)) return true;
  }
  const uint64_t t0 = globaltimer_ns();
  if constexpr (POLL) {
    if (g_wait_limit_ns < kWatchdogNs) {
      for (;;) {
        if (mbar_test_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > g_wait_limit_ns) {
          *abort_flag = 1;
          atomicOr(err_word, kErrTimeout | (site << 8));
          return false;
        }
      }
    }
  }
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0 || g_wait_limit_ns < kWatchdogNs) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > g_wait_limit_ns) {
        *abort_flag = 1;
        atomicOr(err_word, kErrTimeout | (site << 8));
        return false;
      }
    }
  }
}

// Short bounded wait used only while tearing down after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// Dynamic work schedule of a persistent, warp-specialised kernel: the
// producer warp takes the next item index from a global counter (zero when
// the launch starts) and hands it to the consumer warps through a ring of
// kSchedSlots slots in shared memory.  sfull[i] takes 1 arrival (the
// producer); sempty[i] takes one arrival per consumer warp.  (A deeper ring
// measured no faster: the producer's single Q buffer already keeps it within
// an item of its consumers.)  Both return the item, -1 when the work is
// exhausted, or -2 when a wait gave up (the CTA is aborting).
// ---------------------------------------------------------------------------
constexpr int kSchedSlots = 2;

template <bool POLL = false>
__device__ __forceinline__ int sched_produce(uint32_t k, unsigned int* ctr, int n_items,
                                             uint64_t* sfull, uint64_t* sempty,
                                             volatile int* sched, volatile int* abort_flag,
                                             unsigned int* err_word, bool leader) {
  const int slot = k % kSchedSlots;
  if (!mbar_wait<POLL>(&sempty[slot], ((k / kSchedSlots) & 1) ^ 1, abort_flag, err_word, 14))
    return -2;
  int w = -1;
  if (leader) {
    const unsigned int t = atomicAdd(ctr, 1u);
    w = t < (unsigned int)n_items ? (int)t : -1;
    sched[slot] = w;
    mbar_arrive(&sfull[slot]);
  }
  return __shfl_sync(0xffffffffu, w, 0);
}

// Whole warp: the item the producer published for step k.
template <bool POLL = false>
__device__ __forceinline__ int sched_consume(uint32_t k, uint64_t* sfull, uint64_t* sempty,
                                             volatile int* sched, volatile int* abort_flag,
                                             unsigned int* err_word, unsigned int site) {
  const int slot = k % kSchedSlots;
  if (!mbar_wait<POLL>(&sfull[slot], (k / kSchedSlots) & 1, abort_flag, err_word, site)) return -2;
  const int w = sched[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sempty[slot]);
  return w;
}

// One lane alone (the rest of its warp elsewhere): the published item.
template <bool POLL = false>
__device__ __forceinline__ int sched_consume_lane(uint32_t k, uint64_t* sfull, uint64_t* sempty,
                                                  volatile int* sched, volatile int* abort_flag,
                                                  unsigned int* err_word, unsigned int site) {
  const int slot = k % kSchedSlots;
  if (!mbar_wait<POLL>(&sfull[slot], (k / kSchedSlots) & 1, abort_flag, err_word, site)) return -2;
  const int w = sched[slot];
  mbar_arrive(&sempty[slot]);
  return w;
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor loads into shared memory, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// L2 prefetch of one 4-D tile (no shared-memory destination, no completion):
// warms L2 only.  Coordinates follow the same rules as tma_load_4d; rows
// outside the tensor are skipped.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* m, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// Relaxed (racy-by-design) load of a 32-bit value another kernel may be writing.
__device__ __forceinline__ int ld_relaxed_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* m, uint64_t* bar,
                                                 int c0, int c1, int c2, int c3,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------
// Whole warp: allocate ncols TMEM columns, base address written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
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

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two MMA forms with each shared-memory descriptor given as its two
// 32-bit halves.  Callers advance a descriptor along a tile by adding
// (byte offset >> 4) to the low half alone: the start-address field (bits
// 0-13) holds address bits 4-17 and shared-memory addresses stay below 2^18,
// so the addition never carries out of the low word, and one 32-bit add
// replaces a 64-bit add with its carry.
__device__ __forceinline__ void mma_ss_lh(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                          uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_ts_lh(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on *bar when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane
// (base lane + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Registers written by tcgen05.ld are only valid after tcgen05.wait::ld.  This
// empty statement, placed after the wait, makes every later use of r depend on
// it, so the compiler cannot move a use above the wait.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// Warpgroup register re-allocation (all 128 threads of a warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Three-input max / min (one instruction on sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
//   saddr : shared address of the first 16-byte chunk (region base plus the
//           in-row byte offset of the K step; regions are 1024-byte aligned)
//   lbo   : leading-dimension byte offset (MN-major: stride between 64-element
//           column blocks; ignored for K-major swizzled tiles)
//   sbo   : stride-dimension byte offset (stride between 8-row groups: 1024)
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2u) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
//   bf16   : A/B are bf16 (else fp16)
//   b_mn   : B is MN-major (N contiguous in shared memory) instead of K-major
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool b_mn) {
  return (1u << 4)                                   // D format: f32
         | ((bf16 ? 1u : 0u) << 7)                   // A format
         | ((bf16 ? 1u : 0u) << 10)                  // B format
         | ((b_mn ? 1u : 0u) << 16)                  // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ---------------------------------------------------------------------------
// Warp-level MMA (used by the bandwidth-bound decode path)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 f32) += A(16x16 bf16) * B(16x8 bf16)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch controls.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace fa
