// fa_prefill.cu -- dense flash-attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM), warp-specialised and persistent.
//
// What it computes (tessera #90 "compiler-generated flash_attn fwd+bwd",
// flash_attn forward commit note; "Dense flash-attention prefill (gfx950 /
// MI355X)", opening paragraph):
//   O[b,i,h,:] = sum_j p_ij V[b,j,h/G,:] / sum_j p_ij,
//   p_ij = exp(scale * <Q[b,i,h], K[b,j,h/G]> - m_i), over the keys j visible
//   to row i (all Sk keys, or j <= i + Sk - Sq when causal).
//
// Work unit ("Persistent (grid-stride) mode" of the gfx950 README): 256 query
// rows of one query head, held as two 128-row Q tiles.  A persistent grid of
// one CTA per SM takes the units in kv-head-major order (all query heads that
// share a K/V head run together, so K/V stay in L2), longest causal units
// first; each CTA claims its next unit from a work counter when it is free,
// instead of a fixed grid stride, which evens out the causal tail.
//
// CTA = 12 warps (3 warpgroups):
//   warps 0-3  softmax/epilogue for Q tile 0 (TMEM lanes 0-127)
//   warps 4-7  softmax/epilogue for Q tile 1
//   warp  8    TMA producer: Q tiles, then K_j / V_j tiles into an NSTAGE ring
//   warp  9    TMEM allocator and MMA issuer (one lane)
//   warps 10-11 idle (they complete warpgroup 2 for the register split)
// TMEM (512 columns): S0 | S1 | O0 | O1; P_i (bf16) is written over the first
// half of S_i and fed to the P@V MMA straight from TMEM (no register or shared
// memory relayout -- the role the transposed-PV lever plays on gfx950).
// MMA issue order per KV step j: PV0(j), S0(j+1), PV1(j), S1(j+1), so each
// softmax group has two MMA blocks of time to turn S_i into P_i.
// Softmax: exp2 domain with scale*log2(e) folded into one FMA; lazy rescale
// (O and l are rescaled only when a tile's row sum of P, taken against the
// stale running max, exceeds 2^60 for bf16 P or 2^15 for fp16 P; the gfx950
// README's "lazy" lever); causal and Sk-tail masks only on the tiles that need
// them (its "diagonal-only causal masking").
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <mutex>
#include <unordered_map>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ unsigned int g_prefill_err = 0;
// Rows (summed over K/V tiles) whose lazy rescale fired: the slow path of the
// softmax that rescales O and l to a new running max and recomputes P.
__device__ unsigned long long g_prefill_rescales = 0;

namespace pf {
constexpr int BM = 128;         // rows per Q tile
constexpr int BN = 128;         // keys per K/V tile
constexpr int QBLOCK = 2 * BM;  // query rows per work item
constexpr int THREADS = 384;  // 3 warpgroups
// Register split (setmaxnreg): the block launches with 168 registers per
// thread (384 x 168 = 64512).  The two softmax warpgroups take 208 each, the
// producer/MMA warpgroup keeps 88: 256*208 + 128*88 = 64512, exactly the
// launch pool (a larger sum would make setmaxnreg.inc wait forever).
constexpr uint32_t REGS_LAUNCH = 168, REGS_SOFTMAX = 208, REGS_ISSUE = 88;
static_assert(256 * REGS_SOFTMAX + 128 * REGS_ISSUE <= THREADS * REGS_LAUNCH,
              "register split exceeds the launch allocation");
constexpr int HALF_BYTES = 128 * 128;  // 128 rows x 64 elements x 2 bytes

template <int D, bool PACKED>
struct Cfg {
  static constexpr int HALVES = D / 64;
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;  // one 128-row tile
  static constexpr int NSTAGE = (D == 128) ? 4 : 9;
  static constexpr int SMEM_Q = 2 * TILE_BYTES;
  static constexpr int SMEM_KV = NSTAGE * TILE_BYTES;
  // Packed sequences: O leaves through a staging area per softmax warp (32
  // rows x 64 columns, 4 KiB, swizzled as the tensor map says) and that
  // warp's own TMA stores.
  static constexpr bool O_TMA = PACKED;
  static constexpr int OST_WARP = 32 * 128;
  static constexpr int SMEM_OST = O_TMA ? 8 * OST_WARP : 0;
  static constexpr int SMEM_BAR = 512;
  static constexpr int SMEM_TOTAL = 1024 + SMEM_Q + SMEM_KV + SMEM_OST + SMEM_BAR;
  static_assert(SMEM_TOTAL <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
};
}  // namespace pf

// TMA stores of O (the packed kernel's epilogue).
// TMA store of one 4-D tile from shared memory (laid out as the tensor map's
// swizzle says) to global memory; elements outside the tensor are not
// written.  Completion is tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* m, const void* src, int c0, int c1,
                                             int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk stores have read their shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until this thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

struct PrefillParams {
  void* o;     // [B, Sq, Hq, D]; packed sequences: [total_q, Hq, D]
  float* lse;  // [B, Hq, Sq]; packed: [Hq, total_q]; natural-log log-sum-exp, or null
  // Packed (variable-length) sequences: the work units, longest first, as
  // written by varlen_plan_kernel (two int4 per unit: {q0, k0, Sq, Sk} of its
  // sequence and {qb, b, 0, 0}), and their number (device).  Null for a dense
  // batch.  Sq is then the longest query length and Sk is unused.
  const int4* units;
  const int* n_units;
  int total_q, total_k;
  int B, Hq, Hkv, Sq, Sk, G, causal, n_qb, n_items;
  // Work counter [2] (claims, CTAs finished), zero when the launch starts:
  // each persistent CTA claims the next work item when it is free (items keep
  // their order: kv-head-major for a dense batch, the planned longest-first
  // list for packed sequences); the last CTA to finish zeroes both again.
  unsigned int* work_ctr;
  float c;  // scale * log2(e)
};

// Rows of one sequence of the batch.
struct SeqSpan {
  int q0, k0;   // first query / key row in the tensor maps' row coordinate
  int tb;       // tensor-map batch coordinate
  int Sq, Sk;   // its lengths
  size_t orow;  // packed row index of its query row 0 (O is [rows, Hq, D])
  // Packed sequences: 1 when the item is a head pair -- Q tile i is query
  // head hq + i on the block's first 128 rows (a block with at most 128 rows,
  // whose second tile would otherwise be empty); 0: tile i is rows
  // [128 i, 128 i + 128) of the block, query head hq.
  int pair;
};

// Work item w -> (b, hq, qb): kv-head-major, then batch, then query blocks in
// decreasing order (longest causal rows first), then the query heads of the
// GQA group.
__host__ __device__ __forceinline__ void prefill_item(int w, int B, int Hq, int Hkv, int n_qb,
                                                      int* b, int* hq, int* qb) {
  const int G = Hq / Hkv;
  const int per_b = n_qb * G;
  const int per_kv = B * per_b;
  const int hkv = w / per_kv;
  int r = w - hkv * per_kv;
  *b = r / per_b;
  r -= *b * per_b;
  const int qr = r / G;
  *hq = hkv * G + (r - qr * G);
  *qb = n_qb - 1 - qr;
}

void prefill_item_host(int w, int B, int Hq, int Hkv, int n_qb, int* b, int* hq, int* qb) {
  prefill_item(w, B, Hq, Hkv, n_qb, b, hq, qb);
}

// Work item w of either kind.  Dense: prefill_item.  Packed: unit w / Hq of
// the planned list (longest first) with query head w % Hq, so the query heads
// of one kv head, which read the same K/V, run side by side.
template <bool PACKED>
__device__ __forceinline__ SeqSpan work_item(const PrefillParams& p, int w, int* b, int* hq,
                                             int* qb) {
  SeqSpan s;
  if constexpr (!PACKED) {
    prefill_item(w, p.B, p.Hq, p.Hkv, p.n_qb, b, hq, qb);
    s.q0 = 0;
    s.k0 = 0;
    s.tb = *b;
    s.Sq = p.Sq;
    s.Sk = p.Sk;
    s.orow = (size_t)*b * p.Sq;
    s.pair = 0;
  } else {
    const int u = w / p.Hq;
    const int hh = w - u * p.Hq;
    const int4 a = p.units[2 * u], c = p.units[2 * u + 1];
    *qb = c.x;
    *b = c.y;
    s.q0 = a.x;
    s.k0 = a.y;
    s.tb = 0;
    s.Sk = a.w;
    s.orow = (size_t)a.x;
    s.pair = c.z;
    // A head-pair unit's items h >= Hq / 2 are empty: no rows.
    const bool empty = c.z && hh >= p.Hq / 2;
    *hq = c.z ? (empty ? 0 : 2 * hh) : hh;
    s.Sq = empty ? 0 : a.z;
  }
  return s;
}

// Number of K/V tiles Q tile rows [row0, row0+BM) need (0 if the tile is past
// Sq or sees no key).
__host__ __device__ __forceinline__ int kv_tiles_for(int row0, int Sq, int Sk, int causal) {
  if (row0 >= Sq || Sk <= 0) return 0;
  int nk = Sk;
  if (causal) {
    const int last_row = (row0 + pf::BM - 1 < Sq - 1) ? row0 + pf::BM - 1 : Sq - 1;
    const int lim = last_row + (Sk - Sq) + 1;  // keys [0, lim) visible to the last row
    nk = lim < Sk ? lim : Sk;
    if (nk <= 0) return 0;
  }
  return (nk + pf::BN - 1) / pf::BN;
}

// ---------------------------------------------------------------------------
// Packed sequences: the work plan.  One CTA reads the offsets, checks each
// sequence (0 <= cu[b] <= cu[b+1] <= total, query length <= n_qb_max * 256;
// a failing sequence is left out and sets the bounds bit of the error word),
// and lists every 256-row query block of every sequence ordered by its K/V
// tile count, largest first (longest-processing-time order; blocks past a
// sequence's end are not listed).  The gfx950 prefill README's TODO list asks
// for this: per-sequence load balance, so that short and long sequences of a
// batch do not serialise.  The plan also zeroes the prefill's work counter.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 4096;  // K/V tile counts >= 4095 share the top bucket
static_assert(kPlanBuckets == 4 * kPlanThreads, "each thread scans four buckets");

__device__ __forceinline__ bool plan_span(const int32_t* cu_q, const int32_t* cu_k, int b,
                                          int total_q, int total_k, int n_qb_max, int4* span) {
  const int q0 = cu_q[b], q1 = cu_q[b + 1], k0 = cu_k[b], k1 = cu_k[b + 1];
  const bool ok = 0 <= q0 && q0 <= q1 && q1 <= total_q && 0 <= k0 && k0 <= k1 && k1 <= total_k &&
                  (long long)(q1 - q0) <= (long long)n_qb_max * pf::QBLOCK;
  *span = make_int4(q0, k0, q1 - q0, k1 - k0);
  return ok;
}

__device__ __forceinline__ int plan_bucket(int qb, const int4& sp, int causal) {
  const int n0 = kv_tiles_for(qb * pf::QBLOCK, sp.z, sp.w, causal);
  const int n1 = kv_tiles_for(qb * pf::QBLOCK + pf::BM, sp.z, sp.w, causal);
  const int n = n0 > n1 ? n0 : n1;
  return n < kPlanBuckets - 1 ? n : kPlanBuckets - 1;
}

// pair_heads (the GQA group size is even, so heads 2h and 2h + 1 read the
// same K/V): a block of at most 128 rows becomes a head-pair unit, whose work
// items h < Hq / 2 run heads 2h and 2h + 1 as its two Q tiles (the items
// h >= Hq / 2 are empty), so its K/V steps run with both tiles full.
__global__ void __launch_bounds__(kPlanThreads)
    varlen_plan_kernel(const int32_t* cu_q, const int32_t* cu_k, int B, int total_q, int total_k,
                       int n_qb_max, int causal, int pair_heads, int4* units, int* n_units,
                       unsigned int* work_ctr) {
  __shared__ int start[kPlanBuckets];  // counts, then each bucket's next list slot
  __shared__ int warp_sum[kPlanThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int i = t; i < kPlanBuckets; i += kPlanThreads) start[i] = 0;
  __syncthreads();
  for (int b = t; b < B; b += kPlanThreads) {
    int4 sp;
    if (!plan_span(cu_q, cu_k, b, total_q, total_k, n_qb_max, &sp)) {
      atomicOr(&g_prefill_err, kErrBounds);
      continue;
    }
    const int nb = (sp.z + pf::QBLOCK - 1) / pf::QBLOCK;
    for (int qb = 0; qb < nb; ++qb) atomicAdd(&start[plan_bucket(qb, sp, causal)], 1);
  }
  __syncthreads();
  // Exclusive prefix sum over the buckets from the largest tile count down:
  // thread t owns buckets kPlanBuckets-1-4t .. kPlanBuckets-4-4t.
  int c[4], sum = 0;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    c[x] = start[kPlanBuckets - 1 - (4 * t + x)];
    sum += c[x];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    warp_sum[lane] = ws;  // inclusive over warps
  }
  __syncthreads();
  int run = incl - sum + (warp > 0 ? warp_sum[warp - 1] : 0);  // exclusive
  const int total = warp_sum[kPlanThreads / 32 - 1];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    start[kPlanBuckets - 1 - (4 * t + x)] = run;
    run += c[x];
  }
  __syncthreads();
  for (int b = t; b < B; b += kPlanThreads) {
    int4 sp;
    if (!plan_span(cu_q, cu_k, b, total_q, total_k, n_qb_max, &sp)) continue;
    const int nb = (sp.z + pf::QBLOCK - 1) / pf::QBLOCK;
    for (int qb = 0; qb < nb; ++qb) {
      const int pos = atomicAdd(&start[plan_bucket(qb, sp, causal)], 1);
      const int pair = pair_heads && sp.z - qb * pf::QBLOCK <= pf::BM ? 1 : 0;
      units[2 * pos] = sp;
      units[2 * pos + 1] = make_int4(qb, b, pair, 0);
    }
  }
  if (t == 0) {
    *n_units = total;
    work_ctr[0] = 0u;
    work_ctr[1] = 0u;
  }
}

template <typename T>
struct Pack2;
template <>
struct Pack2<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct Pack2<__half> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

template <typename T>
struct IsBF16 {
  static constexpr bool value = false;
};
template <>
struct IsBF16<__nv_bfloat16> {
  static constexpr bool value = true;
};

// PACKED: the batch is packed sequences, whose work items come from the list
// varlen_plan_kernel wrote; otherwise a dense batch.  Both claim items from
// the work counter.  (Separate instantiations: the dense kernel carries none
// of the packed-sequence code.)
// POLL: the waits poll without suspending under a watchdog limit (mbar_wait);
// the host launches this instantiation (dense batches only) while the
// device's wait limit is below kWatchdogNs, and the lean-wait one otherwise.
template <int D, typename T, bool PACKED, bool POLL = false>
__global__ void __launch_bounds__(pf::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const PrefillParams p) {
  using C = pf::Cfg<D, PACKED>;
  constexpr bool kBF16 = IsBF16<T>::value;
  // Largest row sum of unnormalised P a step may leave (see the lazy rescale
  // below): 2^60 for bf16 P (range to 2^127), 2^15 for fp16 P (max 65504).
  constexpr float PBIG = kBF16 ? 1.152921504606846976e18f : 32768.f;
  constexpr int NSTAGE = C::NSTAGE;
  constexpr bool PAIRED = NSTAGE % 2 == 0;  // ring slots released in fixed pairs
  constexpr int NPAIR = NSTAGE / 2;
  constexpr float NEG_INF = -INFINITY;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::SMEM_Q;
  uint8_t* sOst = sKV + C::SMEM_KV;  // [8] O staging areas (packed sequences)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOst + C::SMEM_OST);
  uint64_t* full = bars;
  uint64_t* empty = bars + NSTAGE;
  uint64_t* q_full = bars + 2 * NSTAGE;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_full + 2;  // [2]
  uint64_t* p_full = q_full + 4;  // [2]
  uint64_t* o_full = q_full + 6;  // [2]
  uint64_t* drain = q_full + 8;
  uint64_t* sched_full = q_full + 9;                 // [kSchedSlots] work-item ring
  uint64_t* sched_empty = sched_full + kSchedSlots;  // [kSchedSlots]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sched_empty + kSchedSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* sched = abort_flag + 1;  // [kSchedSlots]
  // The producer's loads that may still be in flight if the CTA aborts,
  // written by the producer when it leaves its loop: [0] ring positions
  // issued (loads [n - NSTAGE, n) may be in flight), [1] q_full phase parity
  // of the last Q issued, [2] whether any Q was issued.
  volatile uint32_t* prod_info = reinterpret_cast<volatile uint32_t*>(sched + kSchedSlots);
  static_assert(2 * C::NSTAGE * 8 + (9 + 2 * kSchedSlots) * 8 + 8 + 4 * (kSchedSlots + 3) <=
                    C::SMEM_BAR,
                "barrier block overflow");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], pf::BM);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(&sched_full[i], 1);
      mbar_init(&sched_empty[i], 9);  // the MMA warp and the 8 softmax warps
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // The producer warp runs its loop with all 32 lanes converged: every lane
  // waits on the barriers, lane 0 alone issues TMA loads, and __syncwarp()
  // follows each issue.  The MMA warp's loop runs on lane 0 alone, the other
  // lanes waiting at its end.  (A warp must never reach the warp-aligned CTA
  // barrier below, or tcgen05.dealloc, with lanes still inside a role loop.)
  const bool leader = lane == 0;
  // Work items: the producer claims each item from the counter and hands it
  // to the MMA and softmax warps (sched_*).
  if (warp >= 8) {
   // ------------------ warpgroup 2: TMA producer and MMA issuer ------------------
   regs_decrease<pf::REGS_ISSUE>();
   if (warp == 8) {
    // ============================ TMA producer ============================
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();
    uint32_t kv_cnt = 0, local = 0, q_par = 0;
    bool ok = true, q_any = false;
    const int n_items = PACKED ? p.Hq * *p.n_units : p.n_items;
    for (uint32_t k = 0; ok; ++k, ++local) {
      const int w = sched_produce<POLL>(k, p.work_ctr, n_items, sched_full, sched_empty, sched,
                                  abort_flag, &g_prefill_err, leader);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hq, qb;
      const SeqSpan sq = work_item<PACKED>(p, w, &b, &hq, &qb);
      const int hkv = hq / p.G;
      const int row0 = qb * pf::QBLOCK;
      const int n0 = kv_tiles_for(row0, sq.Sq, sq.Sk, p.causal);
      const int n1 = kv_tiles_for(row0 + (sq.pair ? 0 : pf::BM), sq.Sq, sq.Sk, p.causal);
      const int n = n0 > n1 ? n0 : n1;
      if (local > 0 && !(ok = mbar_wait<POLL>(q_empty, (local - 1) & 1, abort_flag, &g_prefill_err, 1)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h)
            tma_load_4d_hint(sQ + i * C::TILE_BYTES + h * pf::HALF_BYTES, &tmQ, q_full, h * 64,
                             hq + (sq.pair ? i : 0), sq.q0 + row0 + (sq.pair ? 0 : i * pf::BM),
                             sq.tb, pol_q);
      }
      __syncwarp();
      q_par = local & 1;  // (Q of earlier items has landed: q_empty was waited for)
      q_any = true;
      // Ring order K_0, V_0, K_1, V_1, ...  V_j and K_{j+1} are consumed
      // together (P V_j, then S of step j + 1), so V_j completes on K_{j+1}'s
      // barrier, armed for both tiles, and V_j's own barrier gets a plain
      // arrival that keeps its phases in step: the MMA warp waits once per
      // K/V step.  K_0 and the last V stand alone.
      // An even ring pairs its slots for good: ring positions 2g - 1 (a V) and
      // 2g (the K after it) always share a pair of slots, released together
      // by one commit on empty[g % NPAIR] (see the MMA warp).  Loading either
      // position of pair g waits for the release of pair g - NPAIR.
      auto slot_free = [&](uint32_t cnt) {
        if constexpr (PAIRED) {
          const uint32_t g = (cnt + 1) >> 1;
          return mbar_wait<POLL>(&empty[g % NPAIR], ((g / NPAIR) & 1) ^ 1, abort_flag,
                                 &g_prefill_err, 2);
        } else {
          return mbar_wait<POLL>(&empty[cnt % NSTAGE], ((cnt / NSTAGE) & 1) ^ 1, abort_flag,
                                 &g_prefill_err, 2);
        }
      };
      auto load_tile = [&](uint32_t cnt, const CUtensorMap* m, int kv_tile, uint64_t* bar) {
        const int s = cnt % NSTAGE;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h)
          tma_load_4d_hint(sKV + s * C::TILE_BYTES + h * pf::HALF_BYTES, m, bar, h * 64, hkv,
                           sq.k0 + kv_tile * pf::BN, sq.tb, pol_kv);
      };
      if (n > 0) {
        if ((ok = slot_free(kv_cnt))) {
          if (leader) {
            mbar_arrive_expect_tx(&full[kv_cnt % NSTAGE], C::TILE_BYTES);
            load_tile(kv_cnt, &tmK, 0, &full[kv_cnt % NSTAGE]);
          }
          __syncwarp();
          ++kv_cnt;
        }
      }
      for (int j = 0; j < n && ok; ++j) {
        const uint32_t cv = kv_cnt;  // V_j
        if (j + 1 < n) {
          const uint32_t ck = kv_cnt + 1;  // K_{j+1}
          if (!(ok = slot_free(cv))) break;
          if (!PAIRED && !(ok = slot_free(ck))) break;  // paired: ck shares cv's pair
          if (leader) {
            uint64_t* bar = &full[ck % NSTAGE];
            mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
            mbar_arrive(&full[cv % NSTAGE]);
            load_tile(cv, &tmV, j, bar);
            load_tile(ck, &tmK, j + 1, bar);
          }
          __syncwarp();
          kv_cnt += 2;
        } else {
          if (!(ok = slot_free(cv))) break;
          if (leader) {
            mbar_arrive_expect_tx(&full[cv % NSTAGE], C::TILE_BYTES);
            load_tile(cv, &tmV, j, &full[cv % NSTAGE]);
          }
          __syncwarp();
          kv_cnt += 1;
        }
      }
    }
    if (leader) {
      prod_info[0] = kv_cnt;
      prod_info[1] = q_par;
      prod_info[2] = q_any ? 1u : 0u;
    }
    __syncwarp();
  } else if (warp == 9) {
    // ============================ MMA issuer ============================
    // Lane 0 alone runs the issuer loop (waits, MMAs, commits); the other
    // lanes wait at the __syncwarp below, so the warp reconverges before the
    // CTA barrier and tcgen05.dealloc.  (With all 32 lanes in the loop, every
    // issue and commit was followed by a __syncwarp: a single-lane loop took
    // those, and the leader tests, out of the issuer's instruction stream.)
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16(pf::BM, pf::BN, kBF16, false);
      constexpr uint32_t IDESC_O = idesc_f16(pf::BM, D, kBF16, true);
      const uint32_t sq_addr = smem_u32(sQ);
      const uint32_t skv_addr = smem_u32(sKV);
      uint32_t kv_cnt = 0, local = 0, p_cnt0 = 0, p_cnt1 = 0;
      bool ok = true;

      // Descriptors advance by adding (byte offset >> 4) to their low 32 bits
      // (the start-address field holds address bits 4-17 and shared-memory
      // addresses stay below 2^18, so the addition never carries out of it):
      // one 32-bit add per operand and MMA.  The high halves are constants.
      const uint64_t dq0 = sdesc_sw128(sq_addr, 16, 1024);
      const uint64_t dkv = sdesc_sw128(skv_addr, 16, 1024);          // K, stage 0
      const uint64_t dv = sdesc_sw128(skv_addr, pf::HALF_BYTES, 1024);  // V, stage 0
      const uint32_t q_lo[2] = {(uint32_t)dq0, (uint32_t)dq0 + (C::TILE_BYTES >> 4)};
      const uint32_t sd_hi = (uint32_t)(dq0 >> 32);  // SBO, version, swizzle: shared
      const uint32_t k_lo0 = (uint32_t)dkv, v_lo0 = (uint32_t)dv;
      // S_i = Q_i K^T over D/16 k-steps (K-major A and B, 128-byte swizzle).
      auto issue_s = [&](int i, int stage) {
        const uint32_t d_tmem = tmem + (i ? C::COL_S1 : C::COL_S0);
        const uint32_t a0 = q_lo[i];
        const uint32_t b0 = k_lo0 + stage * (C::TILE_BYTES >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t hoff16 = ((k >> 2) * pf::HALF_BYTES + (k & 3) * 32) >> 4;
          mma_ss_lh(d_tmem, a0 + hoff16, sd_hi, b0 + hoff16, sd_hi, IDESC_S, k > 0 ? 1u : 0u);
        }
      };
      // O_i (+)= P_i V over BN/16 k-steps; P_i from TMEM, V MN-major in smem.
      auto issue_pv = [&](int i, int stage, bool accumulate) {
        const uint32_t d_tmem = tmem + (i ? C::COL_O1 : C::COL_O0);
        const uint32_t p_tmem = tmem + (i ? C::COL_S1 : C::COL_S0);
        const uint32_t b0 = v_lo0 + stage * (C::TILE_BYTES >> 4);
#pragma unroll
        for (int k = 0; k < pf::BN / 16; ++k) {
          mma_ts_lh(d_tmem, p_tmem + k * 8, b0 + (uint32_t)((k * 16 * 128) >> 4), sd_hi, IDESC_O,
                    (accumulate || k > 0) ? 1u : 0u);
        }
      };
      // tcgen05.commit from the issuing lane: arrive on *bar once its MMAs are done.
      auto commit = [&](uint64_t* bar) { mma_commit(bar); };

      // K_j / V_j of an item sit at ring positions kb + 2j / kb + 2j + 1; V_j
      // and K_{j+1} complete together on K_{j+1}'s barrier (see the producer).
      auto ring_wait = [&](uint32_t idx, unsigned int site) {
        return mbar_wait<POLL>(&full[idx % NSTAGE], (idx / NSTAGE) & 1, abort_flag, &g_prefill_err, site);
      };
      for (uint32_t it = 0; ok; ++it, ++local) {
        const int w = sched_consume_lane<POLL>(it, sched_full, sched_empty, sched, abort_flag,
                                             &g_prefill_err, 15);
        if (w < 0) {
          ok = w == -1;
          break;
        }
        int b, hq, qb;
        const SeqSpan sq = work_item<PACKED>(p, w, &b, &hq, &qb);
        const int row0 = qb * pf::QBLOCK;
        const int nt0 = kv_tiles_for(row0, sq.Sq, sq.Sk, p.causal);
        const int nt1 = kv_tiles_for(row0 + (sq.pair ? 0 : pf::BM), sq.Sq, sq.Sk, p.causal);
        const int n = nt0 > nt1 ? nt0 : nt1;
        if (!(ok = mbar_wait<POLL>(q_full, local & 1, abort_flag, &g_prefill_err, 3))) break;
        tc_fence_after();
        if (n == 0) {
          commit(q_empty);
          continue;
        }
        const uint32_t kb = kv_cnt;
        kv_cnt += 2 * n;
        // K_0 -> S_0(0), S_1(0)
        if (!(ok = ring_wait(kb, 4))) break;
        tc_fence_after();
        if (nt0 > 0) {
          issue_s(0, kb % NSTAGE);
          commit(&s_full[0]);
        }
        if (nt1 > 0) {
          issue_s(1, kb % NSTAGE);
          commit(&s_full[1]);
        }
        // Paired: K_0 (position kb, even) completes pair kb / 2 with the
        // previous item's last V.
        commit(PAIRED ? &empty[(kb >> 1) % NPAIR] : &empty[kb % NSTAGE]);
        if (n == 1) commit(q_empty);
        // Operands of step 0: V_0 and K_1 (one barrier: K_1's), or V_0 alone.
        if (!(ok = ring_wait(n > 1 ? kb + 2 : kb + 1, 5))) break;
        tc_fence_after();

        // Per step j: PV0(j), S0(j+1), PV1(j), S1(j+1), then the operand wait
        // of step j+1 (V_{j+1} and K_{j+2}; K_{j+1} was waited for a step
        // earlier).  The wait sits behind a whole batch of issued MMAs, so its
        // latency leaves less of the tensor pipe idle.
        for (int j = 0; j < n && ok; ++j) {
          const int sV = (kb + 2 * j + 1) % NSTAGE;
          const int sK = (kb + 2 * j + 2) % NSTAGE;  // K_{j+1}
          if (j < nt0) {
            if (!(ok = mbar_wait<POLL>(&p_full[0], p_cnt0 & 1, abort_flag, &g_prefill_err, 7))) break;
            ++p_cnt0;
            tc_fence_after();
            issue_pv(0, sV, j > 0);
            if (j == nt0 - 1) commit(&o_full[0]);
            if (j + 1 < nt0) {
              issue_s(0, sK);
              commit(&s_full[0]);
            }
          }
          if (j < nt1) {
            if (!(ok = mbar_wait<POLL>(&p_full[1], p_cnt1 & 1, abort_flag, &g_prefill_err, 8))) break;
            ++p_cnt1;
            tc_fence_after();
            issue_pv(1, sV, j > 0);
            if (j == nt1 - 1) commit(&o_full[1]);
          }
          if (!PAIRED) commit(&empty[sV]);  // paired: released with K_{j+1} below
          if (j + 1 < n) {
            if (j + 1 < nt1) {
              issue_s(1, sK);
              commit(&s_full[1]);
            }
            // Paired: V_j and K_{j+1} (positions kb + 2j + 1, + 2) are pair
            // kb / 2 + j + 1.  The last V of an item waits for the next item's K_0.
            commit(PAIRED ? &empty[((kb >> 1) + j + 1) % NPAIR] : &empty[sK]);
            if (j + 1 == n - 1) commit(q_empty);
            // V_{j+1} and K_{j+2} on K_{j+2}'s barrier, or the last V alone.
            if (!(ok = ring_wait(j + 2 < n ? kb + 2 * j + 4 : kb + 2 * j + 3, 6))) break;
            tc_fence_after();
          }
        }
      }
      // Every MMA this lane issued has completed (and its commits have
      // landed) before the CTA barrier that precedes the TMEM dealloc.
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
   }
  } else {
    // ======================= softmax + epilogue (2 groups) =======================
    regs_increase<pf::REGS_SOFTMAX>();
    const int i = warp >> 2;          // Q tile handled by this warpgroup
    const int wq = warp & 3;          // TMEM lane quarter
    const int r = wq * 32 + lane;     // row within the Q tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = t_lane + (i ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = t_lane + (i ? C::COL_O1 : C::COL_O0);
    const float c = p.c;
    const bool neg_scale = c < 0.f;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    T* const O = static_cast<T*>(p.o);
    // 32-byte O stores (D = 128, O's base 32-byte aligned; rows are multiples
    // of 256 bytes): see the epilogue.
    const bool o_wide = D == 128 && (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;

    for (uint32_t it = 0; ok; ++it) {
      const int w =
          sched_consume<POLL>(it, sched_full, sched_empty, sched, abort_flag, &g_prefill_err, 16);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hq, qb;
      const SeqSpan sq = work_item<PACKED>(p, w, &b, &hq, &qb);
      const int Sq = sq.Sq, Sk = sq.Sk, off = Sk - Sq;  // bottom-right causal offset
      const int row0 = qb * pf::QBLOCK + (sq.pair ? 0 : i * pf::BM);
      const int hq_i = hq + (sq.pair ? i : 0);  // this tile's query head
      const int grow = row0 + r;
      const int n_i = kv_tiles_for(row0, Sq, Sk, p.causal);
      T* const orow = O + (sq.orow + grow) * (size_t)p.Hq * D + (size_t)hq_i * D;
      float* const lse_row =
          p.lse ? p.lse + (PACKED ? (size_t)hq_i * p.total_q + sq.orow + grow
                                  : ((size_t)b * p.Hq + hq_i) * p.Sq + grow)
                : nullptr;
      // Self-check: the row must lie inside O (records and skips otherwise).
      const bool row_ok = grow < Sq && b < p.B && hq_i < p.Hq &&
                          (!PACKED || sq.orow + grow < (size_t)p.total_q);
      if (n_i == 0) {
        if (row_ok) {
#pragma unroll
          for (int x = 0; x < D / 8; ++x)
            reinterpret_cast<uint4*>(orow)[x] = make_uint4(0u, 0u, 0u, 0u);
          if (lse_row) *lse_row = NEG_INF;
        }
        continue;
      }
      float m_used = NEG_INF;  // running max in the log2 domain (scaled units)
      float l = 0.f;
      for (int j = 0; j < n_i; ++j) {
        if (!(ok = mbar_wait<POLL>(&s_full[i], s_cnt & 1, abort_flag, &g_prefill_err, 9 + i))) break;
        ++s_cnt;
        __syncwarp();  // tcgen05.ld below is warp-collective
        tc_fence_after();
        const int kv0 = j * pf::BN;
        const bool need_mask =
            (kv0 + pf::BN > Sk) || (p.causal && kv0 + pf::BN - 1 > row0 + off);
        int lim = pf::BN;  // keys [0, lim) of this tile are visible to this row
        if (need_mask) {
          const int lim_c = p.causal ? grow + off + 1 : Sk;
          lim = (lim_c < Sk ? lim_c : Sk) - kv0;
        }
        // Raw-domain fill for hidden keys: becomes -inf once multiplied by c.
        const float hide = neg_scale ? -NEG_INF : NEG_INF;
        uint32_t sr[4][32];
        float mx = hide;  // running max (min if c < 0) of this tile's raw scores
        float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);  // tile row sum

        // Chunk q (32 keys): hide masked keys, fold into the running max.
        auto mask_and_max = [&](uint32_t (&r)[32], int q) {
          float* v = reinterpret_cast<float*>(r);
          if (need_mask) {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (q * 32 + x >= lim) v[x] = hide;
          }
          float a = v[0], b = v[1];
          if (!neg_scale) {
#pragma unroll
            for (int x = 2; x < 30; x += 4) {
              a = max3f(a, v[x], v[x + 1]);
              b = max3f(b, v[x + 2], v[x + 3]);
            }
            mx = max3f(mx, max3f(a, b, v[30]), v[31]);
          } else {
#pragma unroll
            for (int x = 2; x < 30; x += 4) {
              a = min3f(a, v[x], v[x + 1]);
              b = min3f(b, v[x + 2], v[x + 3]);
            }
            mx = min3f(mx, min3f(a, b, v[30]), v[31]);
          }
        };
        // Chunk q: P = exp2(s*c - base) packed to the input type, written over
        // S at columns [16q, 16q+16) (keys 32q..32q+31); row sum into la/lb.
        auto exp_store = [&](uint32_t (&r)[32], int q, float base) {
          const float* v = reinterpret_cast<const float*>(r);
          const float2 c2 = make_float2(c, c), nb2 = make_float2(-base, -base);
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float2 a = __ffma2_rn(make_float2(v[2 * t], v[2 * t + 1]), c2, nb2);
            const float2 pp = make_float2(fast_exp2(a.x), fast_exp2(a.y));
            if (t & 1)
              lb = __fadd2_rn(lb, pp);
            else
              la = __fadd2_rn(la, pp);
            pk[t] = Pack2<T>::pack(pp.x, pp.y);
          }
          tmem_st16(tS + q * 16, pk);
        };

        // All four 32-column loads in flight at once: tcgen05.wait::ld waits
        // for every outstanding load, so finer pipelining would serialise on
        // the TMEM load latency.
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tS + q4 * 32, sr[q4]);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) reg_fence32(sr[q4]);
        if (j == 0) {
          // First tile of the item: no running max yet -- max first, then P.
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) mask_and_max(sr[q4], q4);
          m_used = mx * c;
          const float base = (m_used == NEG_INF) ? 0.f : m_used;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) exp_store(sr[q4], q4, base);
        } else {
          // Later tiles: exponentiate against the running max m_used without
          // computing this tile's max.  Every P of a row is bounded by the
          // row's tile sum, so a sum <= PBIG guarantees P fits the input type
          // and the fp32 sums (the lazy-rescale idea of the gfx950 README with
          // the threshold moved from the max to the sum).  Rows above it (their
          // max grew by ~log2(PBIG)), and rows that had no visible key before
          // (m_used = -inf: P was taken against 0), take the slow path, which
          // finds the true max from the scores still in registers.
          const float base_old = (m_used == NEG_INF) ? 0.f : m_used;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            if (need_mask) {
              float* v = reinterpret_cast<float*>(sr[q4]);
#pragma unroll
              for (int x = 0; x < 32; ++x)
                if (q4 * 32 + x >= lim) v[x] = hide;
            }
            exp_store(sr[q4], q4, base_old);
          }
          const float lt = (la.x + la.y) + (lb.x + lb.y);
          const bool resc = !(lt <= PBIG) || (m_used == NEG_INF && lim > 0);
          const uint32_t resc_rows = __ballot_sync(0xffffffffu, resc);
          if (resc_rows) {
            // Rare: rescale l and O by 2^(m_used - m_new) for those rows and
            // rewrite this tile's P.  P_i(j-1) @ V has completed (it was
            // issued before S_i(j)); P_i(j) is not read before p_full below.
            if (lane == 0) atomicAdd(&g_prefill_rescales, (unsigned long long)__popc(resc_rows));
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) mask_and_max(sr[q4], q4);
            float f = 1.f;
            if (resc) {
              const float m_new = fmaxf(m_used, mx * c);
              f = (m_used == NEG_INF) ? 0.f : fast_exp2(m_used - m_new);
              l *= f;
              m_used = m_new;
            }
            const float base = (m_used == NEG_INF) ? 0.f : m_used;
            tmem_wait_st();
            la = make_float2(0.f, 0.f);
            lb = make_float2(0.f, 0.f);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) exp_store(sr[q4], q4, base);
#pragma unroll
            for (int q4 = 0; q4 < D / 32; ++q4) {
              uint32_t orr[32];
              tmem_ld32(tO + q4 * 32, orr);
              tmem_wait_ld();
              reg_fence32(orr);
#pragma unroll
              for (int x = 0; x < 32; ++x) orr[x] = __float_as_uint(__uint_as_float(orr[x]) * f);
              tmem_st32(tO + q4 * 32, orr);
            }
          }
        }
        l += (la.x + la.y) + (lb.x + lb.y);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[i]);
      }
      if (!ok) break;
      // Epilogue: O / l, rounded once; TMA stores (packed sequences), else
      // 32- or 16-byte stores.
      if (!(ok = mbar_wait<POLL>(&o_full[i], o_cnt & 1, abort_flag, &g_prefill_err, 11 + i))) break;
      ++o_cnt;
      __syncwarp();
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // log sum_j exp(s_j) = ln2 * (m_used + log2 l): m_used is the row max of
      // s * log2(e) the P values were taken against.
      if (lse_row && row_ok)
        *lse_row = l > 0.f ? 0.6931471805599453f * (m_used + __log2f(l)) : NEG_INF;
      // Packed sequences: the warp's 32 rows go out through its
      // staging area and its own TMA stores, 64 columns at a time, when all of
      // them belong to this sequence (rows past its end would be the next
      // sequence's).  Stores from the threads, each its own row, leave the
      // load-store unit a queue of transactions that this warp's next
      // shared-memory operations (its waits on the next item's S) sit behind;
      // packed batches have many short items, so that cost recurs often.
      const int wrow0 = row0 + wq * 32;
      const bool o_tma = C::O_TMA && b < p.B && hq_i < p.Hq && wrow0 + 32 <= Sq &&
                         sq.orow + wrow0 + 32 <= (size_t)p.total_q;
      if (o_tma) {
        uint8_t* const ost = sOst + warp * C::OST_WARP;  // this warp's staging area
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          uint32_t pk[2][16];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            uint32_t orr[32];
            tmem_ld32(tO + (hh * 2 + q2) * 32, orr);
            tmem_wait_ld();
            reg_fence32(orr);
#pragma unroll
            for (int x = 0; x < 16; ++x)
              pk[q2][x] = Pack2<T>::pack(__uint_as_float(orr[2 * x]) * inv,
                                         __uint_as_float(orr[2 * x + 1]) * inv);
          }
          // The staging area is free once the warp's previous store has read it.
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
          // Row `lane`, 16-byte chunk c at lane * 128 + ((c ^ (lane & 7)) << 4):
          // the tensor map's 128-byte swizzle (each 8 lanes hit distinct banks).
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(smem_u32(ost) + lane * 128 + ((c ^ (lane & 7)) << 4),
                         pk[c >> 2][4 * (c & 3)], pk[c >> 2][4 * (c & 3) + 1],
                         pk[c >> 2][4 * (c & 3) + 2], pk[c >> 2][4 * (c & 3) + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&tmO, ost, hh * 64, hq_i, sq.q0 + wrow0, sq.tb);
            bulk_commit_group();
          }
        }
      }
#pragma unroll
      for (int q4 = 0; q4 < D / 32 && !o_tma; ++q4) {
        uint32_t orr[32];
        tmem_ld32(tO + q4 * 32, orr);
        tmem_wait_ld();
        reg_fence32(orr);
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          pk[x] = Pack2<T>::pack(__uint_as_float(orr[2 * x]) * inv,
                                 __uint_as_float(orr[2 * x + 1]) * inv);
        if (grow < Sq) {
          if (!row_ok) {
            atomicOr(&g_prefill_err, kErrBounds);
            continue;
          }
          if (o_wide) {
            // 32-byte stores.  Each thread stores its own row, so every store
            // instruction touches 32 rows; the load-store unit works through
            // them for a couple of thousand clocks after the last one issues,
            // and this warpgroup's next shared-memory operations (its waits on
            // the next item's S) queue behind them.  Half as many instructions
            // halve that drain.
#pragma unroll
            for (int x = 0; x < 2; ++x)
              asm volatile(
                  "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                      orow + q4 * 32 + x * 16),
                  "r"(pk[8 * x]), "r"(pk[8 * x + 1]), "r"(pk[8 * x + 2]), "r"(pk[8 * x + 3]),
                  "r"(pk[8 * x + 4]), "r"(pk[8 * x + 5]), "r"(pk[8 * x + 6]), "r"(pk[8 * x + 7])
                  : "memory");
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
      }
      tc_fence_before();
    }
    // The TMA stores this warp issued complete before the CTA ends.
    if (C::O_TMA && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Aborted CTA (a wait gave up, here or in another warp, possibly after the
  // producer issued its last loads): wait, bounded, for every load that may
  // still be in flight before the CTA exits.  A ring load older than the last
  // NSTAGE has landed (its slot was released before the producer reused it),
  // and so has the Q of any item before the last.
  if (warp == 8 && *abort_flag) {
    const uint32_t issued = prod_info[0];
    const uint32_t first = issued > (uint32_t)NSTAGE ? issued - NSTAGE : 0u;
    for (uint32_t u = first; u < issued; ++u) mbar_wait_drain(&full[u % NSTAGE], (u / NSTAGE) & 1);
    if (prod_info[2]) mbar_wait_drain(q_full, prod_info[1]);
    __syncwarp();
  }
  // Every CTA has made its last claim once it gets here.  The last CTA out
  // sets the work counter back to zero for the next launch that uses it.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.work_ctr + 1, 1u) == gridDim.x - 1) {
      p.work_ctr[0] = 0u;
      p.work_ctr[1] = 0u;
    }
  }
}

// Sk == 0: no key is visible to any row, O = 0 and log-sum-exp -inf.
template <typename T>
__global__ void prefill_zero_kernel(T* o, size_t n, float* lse, size_t nl) {
  for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < n;
       x += (size_t)gridDim.x * blockDim.x)
    o[x] = T(0.f);
  if (lse)
    for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < nl;
         x += (size_t)gridDim.x * blockDim.x)
      lse[x] = -INFINITY;
}

// Host copy of each device's wait limit: the launch picks the POLL
// instantiation while it is a watchdog limit.
static unsigned long long g_host_wait_limit[64];

static bool watchdog_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const unsigned long long v = __atomic_load_n(&g_host_wait_limit[dev], __ATOMIC_RELAXED);
  return v != 0 && v < kWatchdogNs;
}

// Dense batch: cu_q == nullptr, rows = Sq / Sk per sequence.  Packed
// sequences: cu_q / cu_k device prefix sums, Sq = longest query length,
// rows_q / rows_k = total packed rows.
struct PrefillShape {
  int B, Hq, Hkv, Sq, Sk;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
};

// units / n_units: the packed-sequence plan (device; null for a dense batch).
template <int D, typename T>
static int launch_prefill_t(const void* q, const void* k, const void* v, void* o, float* lse,
                            const PrefillShape& sh, float scale, int causal,
                            unsigned int* work_ctr, const int4* units, const int* n_units,
                            cudaStream_t stream) {
  using CD = pf::Cfg<D, false>;  // dense batches
  using CP = pf::Cfg<D, true>;   // packed sequences
  const bool packed = sh.cu_q != nullptr;
  // to: O in 32-row boxes, for the packed kernel's TMA stores.
  CUtensorMap tq, tk, tv, to{};  // to stays unused (zero) for a dense batch
  if (packed) {
    if (encode_tmap_rows(&to, o, D, sh.Hq, sh.total_q, 1, 32)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tq, q, D, sh.Hq, sh.total_q, 1, pf::BM)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tk, k, D, sh.Hkv, sh.total_k, 1, pf::BN)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tv, v, D, sh.Hkv, sh.total_k, 1, pf::BN)) return cudaErrorInvalidValue;
  } else {
    if (encode_tmap_rows(&tq, q, D, sh.Hq, sh.Sq, sh.B, pf::BM)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tk, k, D, sh.Hkv, sh.Sk, sh.B, pf::BN)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tv, v, D, sh.Hkv, sh.Sk, sh.B, pf::BN)) return cudaErrorInvalidValue;
  }
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, T, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CD::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_kernel<D, T, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, CP::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_kernel<D, T, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, CD::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  PrefillParams p;
  p.o = o;
  p.lse = lse;
  p.units = units;
  p.n_units = n_units;
  p.total_q = sh.total_q;
  p.total_k = sh.total_k;
  p.B = sh.B;
  p.Hq = sh.Hq;
  p.Hkv = sh.Hkv;
  p.Sq = sh.Sq;
  p.Sk = sh.Sk;
  p.G = sh.Hq / sh.Hkv;
  p.causal = causal ? 1 : 0;
  p.n_qb = (sh.Sq + pf::QBLOCK - 1) / pf::QBLOCK;
  p.n_items = sh.B * sh.Hq * p.n_qb;
  p.work_ctr = work_ctr;
  p.c = scale * 1.4426950408889634f;
  // scale == 0: every visible score is 0.  A tiny positive c keeps that (all
  // exp2 arguments round to 0) while hidden keys still map to -inf, never NaN.
  if (p.c == 0.f) p.c = 1e-30f;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  const int grid = p.n_items < sms ? p.n_items : sms;
  if (grid == 0) return cudaSuccess;  // packed: no sequence fits max_seqlen_q (bounds bit set)
  if (packed)
    prefill_kernel<D, T, true><<<grid, pf::THREADS, CP::SMEM_TOTAL, stream>>>(tq, tk, tv, to, p);
  else if (watchdog_on_current_device())
    prefill_kernel<D, T, false, true><<<grid, pf::THREADS, CD::SMEM_TOTAL, stream>>>(tq, tk, tv, to,
                                                                                  p);
  else
    prefill_kernel<D, T, false><<<grid, pf::THREADS, CD::SMEM_TOTAL, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

// Per-stream work counters of the prefill kernel: two uint32 per stream
// (claims, CTAs finished), zero between launches because the last CTA of
// every launch zeroes them.  Streams are told apart by cudaStreamGetId, which
// is unique for the life of the process (so two streams never share a slot,
// and launches that share one are ordered by their stream).  Slots come from
// zero-filled chunks of device memory that live as long as the process.
// Returns null -- the caller then uses stream-ordered scratch zeroed by a
// memset -- while the stream is being captured (each captured graph then owns
// its counter, so two graphs recorded on one stream may replay concurrently)
// or when the device is out of memory.
static unsigned int* work_counter_for_stream(cudaStream_t stream) {
  constexpr int kChunkSlots = 4096;
  struct Pool {
    std::unordered_map<unsigned long long, unsigned int*> slot;
    unsigned int* chunk = nullptr;
    int used = kChunkSlots;
  };
  static std::mutex mu;
  static Pool pools[64];
  int dev = 0;
  unsigned long long id = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return nullptr;
  if (cudaStreamGetId(stream, &id) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Pool& pl = pools[dev];
  auto it = pl.slot.find(id);
  if (it != pl.slot.end()) return it->second;
  if (pl.used == kChunkSlots) {
    void* c = nullptr;
    if (cudaMalloc(&c, kChunkSlots * 2 * sizeof(unsigned int)) != cudaSuccess) return nullptr;
    if (cudaMemset(c, 0, kChunkSlots * 2 * sizeof(unsigned int)) != cudaSuccess) {
      cudaFree(c);
      return nullptr;
    }
    pl.chunk = static_cast<unsigned int*>(c);
    pl.used = 0;
  }
  unsigned int* s = pl.chunk + 2 * pl.used++;
  pl.slot.emplace(id, s);
  return s;
}

static int launch_prefill_shape(const void* q, const void* k, const void* v, void* o,
                                float* lse, const PrefillShape& sh, int D, float scale,
                                int causal, bool bf16, cudaStream_t stream) {
  const bool packed = sh.cu_q != nullptr;
  const int rows_q = packed ? sh.total_q : sh.B * sh.Sq;
  if (sh.B == 0 || sh.Hq == 0 || rows_q == 0) return cudaSuccess;
  if ((packed ? sh.total_k : sh.Sk) == 0) {
    // No key anywhere: O = 0 and every log-sum-exp -inf.
    const size_t n = (size_t)rows_q * sh.Hq * D, nl = (size_t)rows_q * sh.Hq;
    const unsigned blocks = (unsigned)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
    if (bf16)
      prefill_zero_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
          static_cast<__nv_bfloat16*>(o), n, lse, nl);
    else
      prefill_zero_kernel<__half><<<blocks, 256, 0, stream>>>(static_cast<__half*>(o), n, lse,
                                                              nl);
    return cudaGetLastError();
  }
  // The kernel's work counter.  Dense batch: the stream's own slot (zero
  // between launches), or, while the stream is being captured, stream-ordered
  // scratch zeroed here (an allocation and a memset node of the graph).
  // Packed sequences: stream-ordered scratch holding the counter, the number
  // of planned units and the plan itself (two int4 per 256-row query block),
  // all written by varlen_plan_kernel before the prefill starts.
  const int n_qb = (sh.Sq + pf::QBLOCK - 1) / pf::QBLOCK;
  const size_t plan_units = packed ? (size_t)sh.B * n_qb : 0;
  void* ctr = packed ? nullptr : work_counter_for_stream(stream);
  const bool own = ctr == nullptr;
  cudaError_t e = cudaSuccess;
  if (own) {
    const size_t bytes = packed ? 16 + plan_units * 2 * sizeof(int4) : 2 * sizeof(unsigned int);
    e = cudaMallocAsync(&ctr, bytes, stream);
    if (e != cudaSuccess) return e;
    if (!packed) e = cudaMemsetAsync(ctr, 0, 2 * sizeof(unsigned int), stream);
  }
  unsigned int* c = static_cast<unsigned int*>(ctr);
  int4* units = packed ? reinterpret_cast<int4*>(static_cast<uint8_t*>(ctr) + 16) : nullptr;
  int* n_units = packed ? reinterpret_cast<int*>(c + 2) : nullptr;
  if (e == cudaSuccess && packed) {
    const int pair_heads = sh.Hkv > 0 && (sh.Hq / sh.Hkv) % 2 == 0 ? 1 : 0;
    varlen_plan_kernel<<<1, kPlanThreads, 0, stream>>>(sh.cu_q, sh.cu_k, sh.B, sh.total_q,
                                                       sh.total_k, n_qb, causal, pair_heads,
                                                       units, n_units, c);
    e = cudaGetLastError();
  }
  int r = e;
  if (e == cudaSuccess) {
    if (D == 64)
      r = bf16 ? launch_prefill_t<64, __nv_bfloat16>(q, k, v, o, lse, sh, scale, causal, c, units,
                                                     n_units, stream)
               : launch_prefill_t<64, __half>(q, k, v, o, lse, sh, scale, causal, c, units,
                                              n_units, stream);
    else
      r = bf16 ? launch_prefill_t<128, __nv_bfloat16>(q, k, v, o, lse, sh, scale, causal, c,
                                                      units, n_units, stream)
               : launch_prefill_t<128, __half>(q, k, v, o, lse, sh, scale, causal, c, units,
                                               n_units, stream);
  }
  const cudaError_t ef = own ? cudaFreeAsync(ctr, stream) : cudaSuccess;
  return r != 0 ? r : (int)ef;
}

int launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal, bool bf16,
                   cudaStream_t stream) {
  const PrefillShape sh{B, Hq, Hkv, Sq, Sk, nullptr, nullptr, 0, 0};
  return launch_prefill_shape(q, k, v, o, lse, sh, D, scale, causal, bf16, stream);
}

int launch_prefill_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* cu_q, const int32_t* cu_k, int B, int Hq, int Hkv,
                          int total_q, int total_k, int max_seqlen_q, int D, float scale,
                          int causal, bool bf16, cudaStream_t stream) {
  const PrefillShape sh{B, Hq, Hkv, max_seqlen_q, 0, cu_q, cu_k, total_q, total_k};
  return launch_prefill_shape(q, k, v, o, lse, sh, D, scale, causal, bf16, stream);
}

int read_prefill_rescales(unsigned long long* out, int reset) {
  unsigned long long v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_rescales, sizeof(v));
  if (e != cudaSuccess) return e;
  if (reset && v) {
    const unsigned long long z = 0;
    e = cudaMemcpyToSymbol(g_prefill_rescales, &z, sizeof(z));
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

int set_prefill_wait_limit(unsigned long long ns) {
  const int e = set_wait_limit_this_unit(ns);
  int dev = 0;
  if (e == 0 && cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64)
    __atomic_store_n(&g_host_wait_limit[dev], ns, __ATOMIC_RELAXED);
  return e;
}

int read_prefill_error(unsigned int* out, int reset) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (reset && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_prefill_err, &z, sizeof(z));
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace fa
