// fa_backward.cu -- attention backward pass on the 5th-generation tensor cores.
//
// Gradients of the loss l = sum(O * dO) with respect to Q, K and V, in the
// three passes of the flash-attention backward commit note of tessera #90
// ("compiler-generated flash_attn fwd+bwd"):
//   pre :  Delta_i = sum_d dO_id O_id                       (per query row)
//   dq  :  per 128-row query tile, over its visible key tiles:
//            S = Q K^T, P = exp(scale S - lse), dP = dO V^T,
//            dS = P * (dP - Delta),  dQ += scale * dS K
//   dkdv:  per 128-key tile, over the query tiles (and query heads of the
//          GQA group) that see it:
//            S^T = K Q^T, P^T, dP^T = V dO^T, dS^T = P^T * (dP^T - Delta),
//            dV += P^T dO,  dK += scale * dS^T Q
// lse is the forward pass's per-row log-sum-exp (fa_prefill_fwd_lse), so P is
// recomputed exactly as the forward computed it, with no row max or sum.
//
// The tensor-core kernels are persistent (one CTA per SM) and
// warp-specialised: element-wise warps turn the S / dP accumulators into dS
// (and P) one TMEM lane per thread and write the results back into TMEM as
// the next MMA's A operand; the next warp issues TMA tile loads, and the one
// after it allocates TMEM and issues tcgen05.mma.  The dq kernel has 4
// element-wise warps (warps 0-3; producer 4, MMA 5).  The dkdv kernels have
// 8, two per TMEM lane quarter, each on half of the query columns (warps
// 0-7; producer 8, MMA 9): at D = 64 64-row query sub-tiles, double-buffered
// in TMEM; at D = 128 128-row sub-tiles with one TMEM buffer (see each
// kernel).  All waits are bounded (see fa_ptx.cuh).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ unsigned int g_backward_err = 0;

namespace bw {
constexpr int BT = 128;                // rows of every tile
constexpr int HALF_BYTES = 128 * 128;  // 128 rows x 64 elements x 2 bytes
constexpr int QS = 64;                 // query rows of a dkdv sub-tile
constexpr int SUB_HALF = QS * 128;     // 64 rows x 64 elements x 2 bytes
constexpr int THREADS = 192;           // dq: warps 0-3 elementwise, 4 producer, 5 MMA
constexpr uint32_t TMEM_COLS = 512;
constexpr int KRING = 3, VRING = 2;    // dq kernel: K and V tile rings
constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct Cfg {
  static constexpr int HALVES = D / 64;
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;  // one 128-row tile
  static constexpr int NSTAGE_DQ = 5;    // dq: K ring (KRING slots) + V ring (VRING slots)
  static constexpr int NSTAGE_DKV = 4;   // (Q, dO) sub-tile ring of the D = 64 dkdv kernel
  // D = 64 dkdv kernel: 8 element-wise warps, then the producer and MMA warps.
  static constexpr int DKV_EW = 8;
  static constexpr int DKV_THREADS = (DKV_EW + 2) * 32;
  static constexpr int SMEM_BAR = 512;
  static constexpr int SMEM_DQ = 1024 + 2 * TILE_BYTES + NSTAGE_DQ * TILE_BYTES + SMEM_BAR;
  // dkdv stage: a 64-row Q sub-tile and its dO sub-tile (1 KiB aligned); the
  // stages' lse*log2(e) and Delta rows follow the ring.
  static constexpr int SUB_BYTES = HALVES * SUB_HALF;
  static constexpr int STAGE_DKV = 2 * SUB_BYTES;
  static constexpr int SMEM_DKV =
      1024 + 2 * TILE_BYTES + NSTAGE_DKV * (STAGE_DKV + 2 * QS * 4) + SMEM_BAR;
};
// dkdv kernel at D = 128 (128-row query sub-tiles): K, V, a Q ring, a dO ring
// and a ring of lse / Delta rows.  The rings fill the 227 KiB a CTA may use,
// leaving PAD_MAX bytes to align the tiles to 1 KiB.
struct Wide {
  static constexpr int QSLOTS = 3, DOSLOTS = 2, LDSLOTS = 2;
  static constexpr int TILE = 2 * HALF_BYTES;  // a 128-row, D = 128 tile
  static constexpr int BAR_BYTES = 256;
  static constexpr int CORE = (2 + QSLOTS + DOSLOTS) * TILE + LDSLOTS * 2 * BT * 4 + BAR_BYTES;
  static constexpr int SMEM = 227 * 1024;
  static constexpr int PAD_MAX = SMEM - CORE;
  static_assert(PAD_MAX >= 0, "wide dkdv layout exceeds the shared memory of a CTA");
};
}  // namespace bw

struct BwdParams {
  void* dq;             // [B, Sq, Hq, D]
  void* dk;             // [B, Sk, Hkv, D]
  void* dv;             // [B, Sk, Hkv, D]
  const float* lse;     // [B, Hq, Sq] natural log
  const float* delta;   // [B, Hq, Sq]
  // Work counter of the kernel (zeroed by the Delta kernel before it runs):
  // persistent CTAs take items in index order, so items are numbered longest
  // first and every CTA takes the next one when it is free.
  unsigned int* work_ctr;
  int B, Hq, Hkv, Sq, Sk, G, causal;
  int n_qt, n_kt, n_items;
  float c;              // scale * log2(e)
  float scale;
};

template <typename T>
struct BPack;
template <>
struct BPack<__nv_bfloat16> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
  }
};
template <>
struct BPack<__half> {
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    return __half22float2(v);
  }
};
template <typename T>
struct BIsBF16 {
  static constexpr bool value = false;
};
template <>
struct BIsBF16<__nv_bfloat16> {
  static constexpr bool value = true;
};

// ------------------------------------------------------------------------------
// pre: Delta[b, h, i] = sum_d dO[b,i,h,d] * O[b,i,h,d].  Rows are taken in
// memory order ([B, Sq, Hq]); D / 8 lanes share a row, each loading 16 bytes
// of O and of dO, and a warp issues the loads of PRE_STEPS steps of rows (8 KiB
// at D = 128) before it reduces any of them, so enough bytes are in flight to
// keep HBM busy.
// ------------------------------------------------------------------------------
constexpr int PRE_STEPS = 4;

template <int D, typename T>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const T* __restrict__ o,
                                                      const T* __restrict__ dout,
                                                      float* __restrict__ delta, int B, int Sq,
                                                      int Hq, unsigned int* __restrict__ ctr) {
  // The dq and dkdv kernels, launched after this one, take work from ctr[0], ctr[1].
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    ctr[0] = 0u;
    ctr[1] = 0u;
  }
  constexpr int LPR = D / 8;          // lanes per row
  constexpr int RPS = 32 / LPR;       // rows per warp and step
  constexpr int RPI = RPS * PRE_STEPS;  // rows per warp and iteration
  const size_t rows = (size_t)B * Sq * Hq;
  const int lane = threadIdx.x & 31, sub = lane / LPR, l = lane % LPR;
  const size_t warps = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t r0 = ((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5) * RPI; r0 < rows;
       r0 += warps * RPI) {
    uint4 a[PRE_STEPS], g[PRE_STEPS];
#pragma unroll
    for (int st = 0; st < PRE_STEPS; ++st) {
      const size_t r = r0 + st * RPS + sub;
      a[st] = g[st] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        a[st] = reinterpret_cast<const uint4*>(o + r * D)[l];
        g[st] = reinterpret_cast<const uint4*>(dout + r * D)[l];
      }
    }
#pragma unroll
    for (int st = 0; st < PRE_STEPS; ++st) {
      const uint32_t av[4] = {a[st].x, a[st].y, a[st].z, a[st].w};
      const uint32_t gv[4] = {g[st].x, g[st].y, g[st].z, g[st].w};
      float acc = 0.f;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float2 fa = BPack<T>::unpack(av[x]), fg = BPack<T>::unpack(gv[x]);
        acc += fa.x * fg.x + fa.y * fg.y;
      }
#pragma unroll
      for (int m = LPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
      const size_t r = r0 + st * RPS + sub;
      if (l == 0 && r < rows) {
        // r indexes [B, Sq, Hq] rows of O; Delta is stored [B, Hq, Sq].  Row
        // counts below 2^32 (every tensor that fits in memory) divide in 32 bits.
        size_t h, i, b;
        if (rows <= 0xffffffffull) {
          const uint32_t ru = (uint32_t)r, bi = ru / (uint32_t)Hq;
          h = ru - bi * (uint32_t)Hq;
          b = bi / (uint32_t)Sq;
          i = bi - (uint32_t)b * (uint32_t)Sq;
        } else {
          const size_t bi = r / Hq;
          h = r - bi * Hq;
          b = bi / Sq;
          i = bi - b * Sq;
        }
        delta[(b * Hq + h) * Sq + i] = acc;
      }
    }
  }
}

// Work items, numbered longest first (the order CTAs take them in).
// dq: (b, hq, query tile), query tiles descending (a causal tile sees more
// keys the later it is); within a tile, batch-major then head, so the query
// heads of one kv head run side by side and share its K/V tiles in L2.
// dkdv: (b, hkv, key tile), key tiles ascending (the earliest key tile is
// seen by the most query tiles); within a tile, batch-major then kv head.
__device__ __forceinline__ void dq_item(int w, const BwdParams& p, int* b, int* hq, int* qt) {
  const int per_t = p.B * p.Hq;
  const int qr = w / per_t;
  const int r = w - qr * per_t;
  *b = r / p.Hq;
  *hq = r - *b * p.Hq;
  *qt = p.n_qt - 1 - qr;
}
__device__ __forceinline__ void dkv_item(int w, const BwdParams& p, int* b, int* hkv, int* kt) {
  const int per_t = p.B * p.Hkv;
  *kt = w / per_t;
  const int r = w - *kt * per_t;
  *b = r / p.Hkv;
  *hkv = r - *b * p.Hkv;
}

// Key tiles seen by query tile rows [r0, r0 + 128).
__device__ __forceinline__ int bw_key_tiles(int r0, const BwdParams& p) {
  if (r0 >= p.Sq || p.Sk <= 0) return 0;
  int nk = p.Sk;
  if (p.causal) {
    const int last = (r0 + bw::BT - 1 < p.Sq - 1 ? r0 + bw::BT - 1 : p.Sq - 1) + (p.Sk - p.Sq);
    nk = last + 1 < p.Sk ? last + 1 : p.Sk;
    if (nk <= 0) return 0;
  }
  return (nk + bw::BT - 1) / bw::BT;
}
// First query tile that sees key tile rows [k0, k0 + 128) (n_qt if none).
__device__ __forceinline__ int bw_first_query_tile(int k0, const BwdParams& p) {
  if (!p.causal) return 0;
  const int i0 = k0 - (p.Sk - p.Sq);  // the first query row that sees key k0
  if (i0 >= p.Sq) return p.n_qt;
  return i0 <= 0 ? 0 : i0 / bw::BT;
}

// ------------------------------------------------------------------------------
// dq
//
// TMEM: S(0) | S(1) | dP | dQ (128 + 128 + 128 + D columns).  S is
// double-buffered and dP is handed back early, so the element-wise pass of key
// tile j overlaps the MMAs around it:
//   S(j+1) is issued a whole step ahead, into the other S buffer;
//   the element-wise warps read all of dP(j) into registers first and say so
//   (ld_done), which lets dP(j+1) be issued while they compute dS(j);
//   dQ += dS(j) K_j follows once dS(j) is in TMEM, then S(j+2) into the buffer
//   dQ(j) has just read.
// K and V tiles sit in two rings: K (3 slots; K_j is read by S(j) and dQ(j)
// and released after dQ(j)) and V (2 slots; V_j is released after dP(j)).
// Each ring frees a slot about a step before its next tile is due.
// ------------------------------------------------------------------------------
template <int D, typename T>
__global__ void __launch_bounds__(bw::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  using C = bw::Cfg<D>;
  constexpr bool kBF16 = BIsBF16<T>::value;
  constexpr int NS = C::NSTAGE_DQ;
  constexpr float NEG_INF = -INFINITY;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::TILE_BYTES;
  uint8_t* sKV = smem + 2 * C::TILE_BYTES;  // K ring slots 0-2, then V ring slots 0-1
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + NS * C::TILE_BYTES);
  uint64_t* full = bars;            // [NS] (K ring: 0-2, V ring: 3-4)
  uint64_t* empty = bars + NS;      // [NS]
  uint64_t* q_full = bars + 2 * NS;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_full + 2;    // [2] S of buffer b in TMEM
  uint64_t* dp_full = q_full + 4;   // dP in TMEM
  uint64_t* ld_done = q_full + 5;   // dP read into registers (128 arrivals)
  uint64_t* ds_full = q_full + 6;   // dS in TMEM (128 arrivals)
  uint64_t* o_full = q_full + 7;    // dQ complete
  uint64_t* drain = q_full + 8;
  uint64_t* sched_full = q_full + 9;                 // [kSchedSlots]
  uint64_t* sched_empty = sched_full + kSchedSlots;  // [kSchedSlots]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sched_empty + kSchedSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* sched = abort_flag + 1;  // [kSchedSlots]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(ld_done, bw::BT);
    mbar_init(ds_full, bw::BT);
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(&sched_full[i], 1);
      mbar_init(&sched_empty[i], 5);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, bw::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const bool leader = lane == 0;
  const int off = p.Sk - p.Sq;
  // The producer's loads that may still be in flight if the CTA aborts (the
  // last KRING K and VRING V tiles, the Q/dO tiles of its last item); drained
  // after the final CTA barrier.
  uint32_t prod_k = 0, prod_v = 0, prod_q_par = 0;
  bool prod_q_any = false;

  if (warp == 4) {
    // ================================ producer ================================
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();
    uint32_t k_iss = 0, v_iss = 0, local = 0;  // K / V tiles issued so far
    bool ok = true;
    for (uint32_t k = 0; ok; ++k, ++local) {
      const int w = sched_produce(k, p.work_ctr, p.n_items, sched_full, sched_empty, sched,
                                  abort_flag, &g_backward_err, leader);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hq, qt;
      dq_item(w, p, &b, &hq, &qt);
      const int hkv = hq / p.G;
      const int n = bw_key_tiles(qt * bw::BT, p);
      if (local > 0 && !(ok = mbar_wait(q_empty, (local - 1) & 1, abort_flag, &g_backward_err, 1)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_4d_hint(sQ + h * bw::HALF_BYTES, &tmQ, q_full, h * 64, hq, qt * bw::BT, b, pol_q);
          tma_load_4d_hint(sDO + h * bw::HALF_BYTES, &tmDO, q_full, h * 64, hq, qt * bw::BT, b,
                           pol_q);
        }
      }
      __syncwarp();
      prod_q_par = local & 1;  // (Q of earlier items has landed: q_empty was waited for)
      prod_q_any = true;
      for (int j = 0; j < n && ok; ++j) {
#pragma unroll
        for (int sel = 0; sel < 2; ++sel) {  // K_j, then V_j
          const uint32_t t = sel ? v_iss : k_iss;  // the tile's count in its ring
          const uint32_t nr = sel ? bw::VRING : bw::KRING;
          const int s = (sel ? bw::KRING : 0) + (int)(t % nr);
          if (!(ok = mbar_wait(&empty[s], ((t / nr) & 1) ^ 1, abort_flag, &g_backward_err, 2)))
            break;
          if (leader) {
            mbar_arrive_expect_tx(&full[s], C::TILE_BYTES);
            const CUtensorMap* m = sel ? &tmV : &tmK;
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h)
              tma_load_4d_hint(sKV + s * C::TILE_BYTES + h * bw::HALF_BYTES, m, &full[s], h * 64,
                               hkv, j * bw::BT, b, pol_kv);
          }
          __syncwarp();
          if (sel) ++v_iss; else ++k_iss;
          prod_k = k_iss;
          prod_v = v_iss;
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ================================== MMA ===================================
    // Lane 0 alone runs the issuer loop; the other lanes wait at the
    // __syncwarp below (the warp reconverges before the CTA barrier and
    // tcgen05.dealloc).  Descriptors advance on their low 32 bits (see
    // mma_ss_lh); the high halves (SBO, version, swizzle) are one constant.
    if (lane == 0) {
      const uint32_t sd_hi = (uint32_t)(sdesc_sw128(0u, 16, 1024) >> 32);
      constexpr uint32_t IDESC_S = idesc_f16(bw::BT, bw::BT, kBF16, false);
      constexpr uint32_t IDESC_ACC = idesc_f16(bw::BT, D, kBF16, true);
      const uint32_t sq_addr = smem_u32(sQ), sdo_addr = smem_u32(sDO), skv_addr = smem_u32(sKV);
      uint32_t kv_cnt = 0, local = 0, g = 0;  // g: key-tile steps so far (buffers, parities)
      bool ok = true;
      constexpr uint32_t COL_DP = 256, COL_DQ = 384;
      // D_tmem = A (K-major smem) x B^T (K-major smem) over D/16 k-steps.
      auto issue_nt = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
        const uint32_t a0 = (uint32_t)sdesc_sw128(a_addr, 16, 1024);
        const uint32_t b0 = (uint32_t)sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t hoff16 = ((k >> 2) * bw::HALF_BYTES + (k & 3) * 32) >> 4;
          mma_ss_lh(tmem + d_col, a0 + hoff16, sd_hi, b0 + hoff16, sd_hi, IDESC_S, k > 0 ? 1u : 0u);
        }
      };
      auto commit = [&](uint64_t* bar) { mma_commit(bar); };
      // Tile t (a global count of key tiles) of the K ring or the V ring.
      auto kslot = [&](uint32_t t) { return (int)(t % bw::KRING); };
      auto vslot = [&](uint32_t t) { return bw::KRING + (int)(t % bw::VRING); };
      auto wait_k = [&](uint32_t t, unsigned int site) {
        const bool r = mbar_wait(&full[kslot(t)], (t / bw::KRING) & 1, abort_flag,
                                 &g_backward_err, site);
        tc_fence_after();
        return r;
      };
      auto wait_v = [&](uint32_t t, unsigned int site) {
        const bool r = mbar_wait(&full[vslot(t)], (t / bw::VRING) & 1, abort_flag,
                                 &g_backward_err, site);
        tc_fence_after();
        return r;
      };
      auto addr = [&](int s) { return skv_addr + s * C::TILE_BYTES; };
      for (uint32_t it = 0; ok; ++it, ++local) {
        const int w =
            sched_consume_lane(it, sched_full, sched_empty, sched, abort_flag, &g_backward_err,
                               11);
        if (w < 0) {
          ok = w == -1;
          break;
        }
        int b, hq, qt;
        dq_item(w, p, &b, &hq, &qt);
        const int n = bw_key_tiles(qt * bw::BT, p);
        if (!(ok = mbar_wait(q_full, local & 1, abort_flag, &g_backward_err, 3))) break;
        tc_fence_after();
        if (n == 0) {
          commit(q_empty);
          commit(o_full);  // dQ = 0 for this tile (accumulator not written)
          continue;
        }
        const uint32_t kb = kv_cnt;  // K_j and V_j are tile kb + j of their rings
        kv_cnt += n;
        // Prologue: S(0), dP(0), S(1).
        if (!(ok = wait_k(kb, 4))) break;
        issue_nt((g & 1) * 128, sq_addr, addr(kslot(kb)));
        commit(&s_full[g & 1]);
        if (!(ok = wait_v(kb, 5))) break;
        issue_nt(COL_DP, sdo_addr, addr(vslot(kb)));
        commit(dp_full);
        commit(&empty[vslot(kb)]);
        if (n == 1) commit(q_empty);
        if (n > 1) {
          if (!(ok = wait_k(kb + 1, 4))) break;
          issue_nt(((g + 1) & 1) * 128, sq_addr, addr(kslot(kb + 1)));
          commit(&s_full[(g + 1) & 1]);
        }
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t gj = g + j;
          // dP(j) is in the element-wise warps' registers: dP(j+1) may go.
          if (!(ok = mbar_wait(ld_done, gj & 1, abort_flag, &g_backward_err, 6))) break;
          tc_fence_after();
          if (j + 1 < n) {
            if (!(ok = wait_v(kb + j + 1, 5))) break;
            issue_nt(COL_DP, sdo_addr, addr(vslot(kb + j + 1)));
            commit(dp_full);
            commit(&empty[vslot(kb + j + 1)]);
            if (j + 1 == n - 1) commit(q_empty);  // the last S and dP are issued
          }
          // dQ += dS(j) K_j: dS (16-bit) in the first 64 columns of S buffer j.
          if (!(ok = mbar_wait(ds_full, gj & 1, abort_flag, &g_backward_err, 6))) break;
          tc_fence_after();
          const uint32_t b0 = (uint32_t)sdesc_sw128(addr(kslot(kb + j)), bw::HALF_BYTES, 1024);
#pragma unroll
          for (int k = 0; k < bw::BT / 16; ++k) {
            mma_ts_lh(tmem + COL_DQ, tmem + (gj & 1) * 128 + k * 8,
                      b0 + (uint32_t)((k * 16 * 128) >> 4), sd_hi, IDESC_ACC,
                      (j > 0 || k > 0) ? 1u : 0u);
          }
          commit(&empty[kslot(kb + j)]);
          // S(j+2) into the buffer dQ(j) has just read.
          if (j + 2 < n) {
            if (!(ok = wait_k(kb + j + 2, 4))) break;
            issue_nt((gj & 1) * 128, sq_addr, addr(kslot(kb + j + 2)));
            commit(&s_full[gj & 1]);
          }
        }
        if (!ok) break;
        g += n;
        commit(o_full);
      }
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // ============================ dS (warps 0-3) ============================
    const int r = warp * 32 + lane;  // TMEM lane = query row within the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint32_t g = 0, o_cnt = 0;  // g: key-tile steps so far (buffers, parities)
    bool ok = true;
    T* const DQ = static_cast<T*>(p.dq);
    constexpr uint32_t COL_DP = 256, COL_DQ = 384;
    for (uint32_t it = 0; ok; ++it) {
      const int w =
          sched_consume(it, sched_full, sched_empty, sched, abort_flag, &g_backward_err, 12);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hq, qt;
      dq_item(w, p, &b, &hq, &qt);
      const int n = bw_key_tiles(qt * bw::BT, p);
      const int i = qt * bw::BT + r;  // query row
      const bool row_ok = i < p.Sq;
      const size_t lrow = ((size_t)b * p.Hq + hq) * p.Sq + (row_ok ? i : 0);
      const float l2 = row_ok ? p.lse[lrow] * bw::LOG2E : 0.f;
      const float dl = row_ok ? p.delta[lrow] : 0.f;
      const bool any_key = row_ok && p.lse[lrow] != NEG_INF;
      const int lim_c = p.causal ? i + off + 1 : p.Sk;  // keys [0, lim) visible
      const int lim = any_key ? (lim_c < p.Sk ? lim_c : p.Sk) : 0;
      for (int j = 0; j < n && ok; ++j, ++g) {
        const uint32_t cs = (g & 1) * 128;  // this step's S buffer
        if (!(ok = mbar_wait(&s_full[g & 1], (g >> 1) & 1, abort_flag, &g_backward_err, 7)))
          break;
        if (!(ok = mbar_wait(dp_full, g & 1, abort_flag, &g_backward_err, 7))) break;
        __syncwarp();
        tc_fence_after();
        // All of dP(j) into registers first, then hand the dP columns back so
        // that dP(j+1) can be computed while dS(j) is.
        uint32_t pr[4][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(t_lane + COL_DP + q4 * 32, pr[q4]);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) reg_fence32(pr[q4]);
        tc_fence_before();
        mbar_arrive(ld_done);
        // Keys [0, lim) of this row are visible: columns from lim_t on are
        // hidden (selected to 0), which only the tile holding key lim has.
        const int lim_t = lim - j * bw::BT;
        const bool edge = __any_sync(0xffffffffu, lim_t < bw::BT);
        const float2 c2 = make_float2(p.c, p.c), nl2 = make_float2(-l2, -l2);
        const float2 nd2 = make_float2(-dl, -dl);
        // S in 32-column chunks, one chunk ahead.
        uint32_t sr[2][32];
        tmem_ld32(t_lane + cs, sr[0]);
        tmem_wait_ld();
        reg_fence32(sr[0]);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int cur = q4 & 1;
          if (q4 < 3) tmem_ld32(t_lane + cs + (q4 + 1) * 32, sr[cur ^ 1]);
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[cur][2 * x]),
                                                    __uint_as_float(sr[cur][2 * x + 1])),
                                        c2, nl2);
            float2 pv = make_float2(fast_exp2(a.x), fast_exp2(a.y));
            if (edge) {
              const int col = q4 * 32 + 2 * x;
              pv.x = col < lim_t ? pv.x : 0.f;
              pv.y = col + 1 < lim_t ? pv.y : 0.f;
            }
            const float2 dd = __fadd2_rn(make_float2(__uint_as_float(pr[q4][2 * x]),
                                                     __uint_as_float(pr[q4][2 * x + 1])),
                                         nd2);
            const float2 ds = __fmul2_rn(pv, dd);
            pk[x] = BPack<T>::pack(ds.x, ds.y);
          }
          // 16-bit dS of these 32 keys over the S columns already read.
          tmem_st16(t_lane + cs + q4 * 16, pk);
          if (q4 < 3) {
            tmem_wait_ld();
            reg_fence32(sr[cur ^ 1]);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (!ok) break;
      // Epilogue: dQ = scale * accumulator, rounded once.
      if (!(ok = mbar_wait(o_full, o_cnt & 1, abort_flag, &g_backward_err, 8))) break;
      ++o_cnt;
      __syncwarp();
      tc_fence_after();
      T* const drow = DQ + (((size_t)b * p.Sq + (row_ok ? i : 0)) * p.Hq + hq) * D;
#pragma unroll
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t ar[32];
        if (n > 0) {
          tmem_ld32(t_lane + COL_DQ + q4 * 32, ar);
          tmem_wait_ld();
          reg_fence32(ar);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ar[x] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          pk[x] = BPack<T>::pack(__uint_as_float(ar[2 * x]) * p.scale,
                                 __uint_as_float(ar[2 * x + 1]) * p.scale);
        if (row_ok) {
          if (b >= p.B || hq >= p.Hq) {
            atomicOr(&g_backward_err, kErrBounds);
            continue;
          }
          uint4* dst = reinterpret_cast<uint4*>(drow + q4 * 32);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, bw::TMEM_COLS);
  }
  // Aborted CTA: wait, bounded, for the loads that may still be in flight
  // (older ones have landed: their slot was released before it was reused).
  if (warp == 4 && *abort_flag) {
    for (uint32_t u = prod_k > (uint32_t)bw::KRING ? prod_k - bw::KRING : 0u; u < prod_k; ++u)
      mbar_wait_drain(&full[u % bw::KRING], (u / bw::KRING) & 1);
    for (uint32_t u = prod_v > (uint32_t)bw::VRING ? prod_v - bw::VRING : 0u; u < prod_v; ++u)
      mbar_wait_drain(&full[bw::KRING + u % bw::VRING], (u / bw::VRING) & 1);
    if (prod_q_any) mbar_wait_drain(q_full, prod_q_par);
    __syncwarp();
  }
}

// ------------------------------------------------------------------------------
// dk, dv at D = 64
//
// Per 128-key tile, the visible query rows are taken 64 at a time (a
// sub-tile) so that S^T / dP^T can be double-buffered in TMEM:
//   columns [0, 64) S^T(0), [64, 128) dP^T(0), [128, 192) S^T(1),
//   [192, 256) dP^T(1), then dV and dK (D columns each).
// While the element-wise warps turn buffer b into P^T / dS^T, the MMA warp
// already computes the next sub-tile's S^T / dP^T into buffer b ^ 1; then it
// issues dV += P^T dO and dK += dS^T Q for buffer b.  MMA issue order:
//   S(u), dP(u), [wait P/dS(u-1)], dV(u-1), dK(u-1), S(u+1), ...
// ------------------------------------------------------------------------------
template <int D, typename T>
__global__ void __launch_bounds__(bw::Cfg<D>::DKV_THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using C = bw::Cfg<D>;
  constexpr bool kBF16 = BIsBF16<T>::value;
  constexpr int NS = C::NSTAGE_DKV;
  constexpr int QS = bw::QS;
  static_assert(D == 64, "the 64-row sub-tile dkdv kernel serves D = 64");
  constexpr int EW = C::DKV_EW;                 // element-wise warps 0 .. EW-1
  constexpr int PRODUCER = EW, MMA = EW + 1;    // then the producer and MMA warps
  // 16-bit P^T / dS^T of query half h start at column PST * h of S^T / dP^T:
  // two threads share each TMEM lane, one per half, and each writes within
  // the 32 columns it has read.
  constexpr int PST = 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::TILE_BYTES;
  uint8_t* sStage = smem + 2 * C::TILE_BYTES;  // [NS] x (Q sub-tile, dO sub-tile)
  float* sLD = reinterpret_cast<float*>(sStage + NS * C::STAGE_DKV);  // [NS][lse*log2e, Delta][QS]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sLD + NS * 2 * QS);
  uint64_t* full = bars;          // [NS]: producer (expect_tx) + producer (after lse/Delta)
  uint64_t* empty = bars + NS;    // [NS]: MMA commit + one arrival per element-wise thread
  uint64_t* kv_full = bars + 2 * NS;
  uint64_t* kv_empty = kv_full + 1;
  uint64_t* st_full = kv_full + 2;  // [2] S^T and dP^T of buffer b in TMEM
  uint64_t* pd_full = kv_full + 4;  // [2] P^T and dS^T of buffer b in TMEM (all element-wise threads)
  uint64_t* o_full = kv_full + 6;   // dK, dV complete
  uint64_t* drain = kv_full + 7;
  uint64_t* sched_full = kv_full + 8;                // [kSchedSlots]
  uint64_t* sched_empty = sched_full + kSchedSlots;  // [kSchedSlots]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sched_empty + kSchedSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* sched = abort_flag + 1;  // [kSchedSlots]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 2);
      mbar_init(&empty[s], 1 + EW * 32);
    }
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&pd_full[i], EW * 32);
    }
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(&sched_full[i], 1);
      mbar_init(&sched_empty[i], EW + 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA) {
    tmem_alloc(tmem_holder, bw::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const bool leader = lane == 0;
  const int off = p.Sk - p.Sq;
  const int n_qs = (p.Sq + QS - 1) / QS;
  // First query sub-tile that sees key row k0 (n_qs if none).
  auto first_sub = [&](int k0) {
    if (!p.causal) return 0;
    const int i0 = k0 - off;  // the first query row that sees key k0
    if (i0 >= p.Sq) return n_qs;
    return i0 <= 0 ? 0 : i0 / QS;
  };
  constexpr uint32_t COL_DV = 256, COL_DK = 256 + D;
  // The producer's loads that may still be in flight if the CTA aborts (the
  // last NS sub-tile stages, the K/V tiles of its last item); drained after
  // the final CTA barrier.
  uint32_t prod_st = 0, prod_kv_par = 0;
  bool prod_kv_any = false;

  if (warp == PRODUCER) {
    // ================================ producer ================================
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    uint32_t st_cnt = 0, local = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k, ++local) {
      const int w = sched_produce(k, p.work_ctr, p.n_items, sched_full, sched_empty, sched,
                                  abort_flag, &g_backward_err, leader);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hkv, kt;
      dkv_item(w, p, &b, &hkv, &kt);
      const int q0 = first_sub(kt * bw::BT);
      if (local > 0 &&
          !(ok = mbar_wait(kv_empty, (local - 1) & 1, abort_flag, &g_backward_err, 1)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_4d_hint(sK + h * bw::HALF_BYTES, &tmK, kv_full, h * 64, hkv, kt * bw::BT, b,
                           pol_kv);
          tma_load_4d_hint(sV + h * bw::HALF_BYTES, &tmV, kv_full, h * 64, hkv, kt * bw::BT, b,
                           pol_kv);
        }
      }
      __syncwarp();
      prod_kv_par = local & 1;  // (K/V of earlier items has landed: kv_empty was waited for)
      prod_kv_any = true;
      // Query sub-tiles descending, the group's heads innermost: the items of
      // one kv head then read the same Q / dO tiles at about the same time.
      for (int qs = n_qs - 1; qs >= q0 && ok; --qs) {
        for (int g = 0; g < p.G && ok; ++g) {
          const int hq = hkv * p.G + g;
          const int s = st_cnt % NS;
          const uint32_t ph = (st_cnt / NS) & 1;
          if (!(ok = mbar_wait(&empty[s], ph ^ 1, abort_flag, &g_backward_err, 2))) break;
          uint8_t* st = sStage + s * C::STAGE_DKV;
          float* sL = sLD + s * 2 * QS;
          float* sD = sL + QS;
          if (leader) {
            mbar_arrive_expect_tx(&full[s], 2 * C::SUB_BYTES);
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h) {
              tma_load_4d_hint(st + h * bw::SUB_HALF, &tmQ, &full[s], h * 64, hq, qs * QS, b,
                               pol_q);
              tma_load_4d_hint(st + C::SUB_BYTES + h * bw::SUB_HALF, &tmDO, &full[s], h * 64, hq,
                               qs * QS, b, pol_q);
            }
          }
          // lse * log2(e) and Delta of the sub-tile's 64 query rows (+inf / 0
          // past Sq: those columns get P = 0).
          const size_t base = ((size_t)b * p.Hq + hq) * p.Sq;
#pragma unroll
          for (int x = 0; x < QS / 32; ++x) {
            const int i = qs * QS + x * 32 + lane;
            sL[x * 32 + lane] = i < p.Sq ? p.lse[base + i] * bw::LOG2E : INFINITY;
            sD[x * 32 + lane] = i < p.Sq ? p.delta[base + i] : 0.f;
          }
          __syncwarp();
          if (leader) mbar_arrive(&full[s]);  // the second arrival, after the smem writes
          __syncwarp();
          ++st_cnt;
          prod_st = st_cnt;
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA) {
    // ================================== MMA ===================================
    // Lane 0 alone runs the issuer loop; the other lanes wait at the
    // __syncwarp below (the warp reconverges before the CTA barrier and
    // tcgen05.dealloc).  Descriptors advance on their low 32 bits (see
    // mma_ss_lh); the high halves (SBO, version, swizzle) are one constant.
    if (lane == 0) {
      const uint32_t sd_hi = (uint32_t)(sdesc_sw128(0u, 16, 1024) >> 32);
      constexpr uint32_t IDESC_S = idesc_f16(bw::BT, QS, kBF16, false);
      constexpr uint32_t IDESC_ACC = idesc_f16(bw::BT, D, kBF16, true);
      const uint32_t sk_addr = smem_u32(sK), sv_addr = smem_u32(sV), sst = smem_u32(sStage);
      uint32_t st_cnt = 0, local = 0, gcnt = 0;
      bool ok = true;
      // D_tmem (128 x 64) = A (128-row tile, K-major) x B^T (64-row sub-tile, K-major).
      auto issue_nt = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
        const uint32_t a0 = (uint32_t)sdesc_sw128(a_addr, 16, 1024);
        const uint32_t b0 = (uint32_t)sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ka16 = ((k >> 2) * bw::HALF_BYTES + (k & 3) * 32) >> 4;
          const uint32_t kb16 = ((k >> 2) * bw::SUB_HALF + (k & 3) * 32) >> 4;
          mma_ss_lh(tmem + d_col, a0 + ka16, sd_hi, b0 + kb16, sd_hi, IDESC_S, k > 0 ? 1u : 0u);
        }
      };
      // acc += A (TMEM, 16-bit) x B (64-row sub-tile, MN-major).  A's 64 query
      // columns are two halves of 32, half h packed from column PST * h, so
      // k-steps 2h and 2h + 1 read columns PST * h and PST * h + 8.
      auto issue_acc = [&](uint32_t d_col, uint32_t a_col, uint32_t b_addr, bool accumulate) {
        const uint32_t b0 = (uint32_t)sdesc_sw128(b_addr, bw::SUB_HALF, 1024);
#pragma unroll
        for (int k = 0; k < QS / 16; ++k) {
          mma_ts_lh(tmem + d_col, tmem + a_col + (k >> 1) * PST + (k & 1) * 8,
                    b0 + (uint32_t)((k * 16 * 128) >> 4),
                    sd_hi, IDESC_ACC, (accumulate || k > 0) ? 1u : 0u);
        }
      };
      auto commit = [&](uint64_t* bar) { mma_commit(bar); };
      // dV += P^T dO and dK += dS^T Q of the sub-step held in buffer gb, stage s.
      auto issue_grads = [&](uint32_t gb, int s, bool accumulate) {
        const int bb = gb & 1;
        if (!mbar_wait(&pd_full[bb], (gb >> 1) & 1, abort_flag, &g_backward_err, 5)) return false;
        tc_fence_after();
        const uint32_t sq = sst + s * C::STAGE_DKV, sdo = sq + C::SUB_BYTES;
        issue_acc(COL_DV, bb * 128, sdo, accumulate);      // dV += P^T dO
        issue_acc(COL_DK, bb * 128 + 64, sq, accumulate);  // dK += dS^T Q
        commit(&empty[s]);
        return true;
      };
      for (uint32_t it = 0; ok; ++it, ++local) {
        const int w =
            sched_consume_lane(it, sched_full, sched_empty, sched, abort_flag, &g_backward_err,
                               11);
        if (w < 0) {
          ok = w == -1;
          break;
        }
        int b, hkv, kt;
        dkv_item(w, p, &b, &hkv, &kt);
        const int steps = p.G * (n_qs - first_sub(kt * bw::BT));
        if (!(ok = mbar_wait(kv_full, local & 1, abort_flag, &g_backward_err, 3))) break;
        tc_fence_after();
        int s_prev = 0;
        for (int u = 0; u < steps && ok; ++u, ++gcnt) {
          const int s = st_cnt % NS;
          const uint32_t ph = (st_cnt / NS) & 1;
          ++st_cnt;
          if (!(ok = mbar_wait(&full[s], ph, abort_flag, &g_backward_err, 4))) break;
          tc_fence_after();
          const uint32_t bb = gcnt & 1;
          const uint32_t sq = sst + s * C::STAGE_DKV, sdo = sq + C::SUB_BYTES;
          issue_nt(bb * 128, sk_addr, sq);       // S^T = K Q^T
          issue_nt(bb * 128 + 64, sv_addr, sdo); // dP^T = V dO^T
          commit(&st_full[bb]);
          if (u > 0 && !(ok = issue_grads(gcnt - 1, s_prev, u > 1))) break;
          s_prev = s;
        }
        if (!ok) break;
        if (steps > 0 && !(ok = issue_grads(gcnt - 1, s_prev, steps > 1))) break;
        commit(kv_empty);
        commit(o_full);
      }
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // ================== P^T and dS^T (element-wise warps) ==================
    // Warp w serves TMEM lane quarter w % 4 and takes the query half w / 4 of
    // each sub-tile.  The pass is element-wise given lse and Delta, so the
    // halves never talk.
    const int quarter = warp & 3, qh0 = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane = key row within the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t ph_cnt = 0, gcnt = 0, o_cnt = 0;
    bool ok = true;
    T* const DK = static_cast<T*>(p.dk);
    T* const DV = static_cast<T*>(p.dv);
    const float2 c2 = make_float2(p.c, p.c);
    for (uint32_t it = 0; ok; ++it) {
      const int w =
          sched_consume(it, sched_full, sched_empty, sched, abort_flag, &g_backward_err, 12);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hkv, kt;
      dkv_item(w, p, &b, &hkv, &kt);
      const int q0 = first_sub(kt * bw::BT);
      const int j = kt * bw::BT + r;  // key row
      for (int qs = n_qs - 1; qs >= q0 && ok; --qs) {
        for (int g = 0; g < p.G && ok; ++g, ++gcnt) {
          const int s = ph_cnt % NS;
          const uint32_t fph = (ph_cnt / NS) & 1;
          ++ph_cnt;
          const uint32_t bb = gcnt & 1;
          // The stage's lse / Delta rows are written by the producer before
          // its second arrival on full[s].
          if (!(ok = mbar_wait(&full[s], fph, abort_flag, &g_backward_err, 9))) break;
          if (!(ok = mbar_wait(&st_full[bb], (gcnt >> 1) & 1, abort_flag, &g_backward_err, 7)))
            break;
          __syncwarp();
          tc_fence_after();
          const float* sL = sLD + s * 2 * QS;
          const float* sD = sL + QS;
          // Query row i = qs * 64 + ic sees key j when i < Sq and (not causal or
          // j <= i + off).  Rows past Sq have lse = +inf in the stage, so their
          // P is 0 without a test; key rows past Sk read zeros (TMA fill) and
          // only feed dK / dV rows that are never stored.  What remains is the
          // causal edge: columns below ic_lo are hidden (P selected to 0),
          // which only a sub-tile on the diagonal has.
          const int ic_lo = p.causal ? j - off - qs * QS : 0;
          const bool edge = __any_sync(0xffffffffu, ic_lo > 0);
          // P^T, dS^T of query half qh from registers sr / pr (its S^T, dP^T),
          // stored 16-bit from column PST * qh: over columns this thread has
          // already read, never over another thread's.
          auto half_pass = [&](int qh, const uint32_t (&sr)[32], const uint32_t (&pr)[32]) {
            uint32_t pp[16], pd[16];
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {
              // lse*log2(e) and Delta of 4 query columns (broadcast loads).
              const float4 l4 = reinterpret_cast<const float4*>(sL)[qh * 8 + x4];
              const float4 d4 = reinterpret_cast<const float4*>(sD)[qh * 8 + x4];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int x = x4 * 2 + h;  // column pair within the half
                const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
                const float2 nd = h ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
                const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[2 * x]),
                                                        __uint_as_float(sr[2 * x + 1])),
                                            c2, nl);
                float2 pv = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                if (edge) {
                  const int col = qh * 32 + 2 * x;
                  pv.x = col < ic_lo ? 0.f : pv.x;
                  pv.y = col + 1 < ic_lo ? 0.f : pv.y;
                }
                const float2 dd = __fadd2_rn(make_float2(__uint_as_float(pr[2 * x]),
                                                         __uint_as_float(pr[2 * x + 1])),
                                             nd);
                const float2 ds = __fmul2_rn(pv, dd);
                pp[x] = BPack<T>::pack(pv.x, pv.y);
                pd[x] = BPack<T>::pack(ds.x, ds.y);
              }
            }
            tmem_st16(t_lane + bb * 128 + qh * PST, pp);
            tmem_st16(t_lane + bb * 128 + 64 + qh * PST, pd);
          };
          uint32_t sr[32], pr[32];
          tmem_ld32(t_lane + bb * 128 + qh0 * 32, sr);
          tmem_ld32(t_lane + bb * 128 + 64 + qh0 * 32, pr);
          tmem_wait_ld();
          reg_fence32(sr);
          reg_fence32(pr);
          half_pass(qh0, sr, pr);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&pd_full[bb]);
          mbar_arrive(&empty[s]);  // this thread is done with the stage's lse / Delta
        }
      }
      if (!ok) break;
      // Epilogue: dV, dK (= scale * accumulator) of this thread's key row; each
      // warp of a lane quarter stores half of the D columns.
      if (!(ok = mbar_wait(o_full, o_cnt & 1, abort_flag, &g_backward_err, 8))) break;
      ++o_cnt;
      __syncwarp();
      tc_fence_after();
      const bool any = p.G * (n_qs - q0) > 0;
      const bool row_ok = j < p.Sk;
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
        T* const row =
            (which ? DK : DV) + (((size_t)b * p.Sk + (row_ok ? j : 0)) * p.Hkv + hkv) * D;
        const float mul = which ? p.scale : 1.f;
        constexpr int NQ = D / 64;  // 32-column chunks per thread
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq) {
          const int q4 = qh0 * NQ + qq;
          uint32_t ar[32];
          if (any) {
            tmem_ld32(t_lane + (which ? COL_DK : COL_DV) + q4 * 32, ar);
            tmem_wait_ld();
            reg_fence32(ar);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) ar[x] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            pk[x] = BPack<T>::pack(__uint_as_float(ar[2 * x]) * mul,
                                   __uint_as_float(ar[2 * x + 1]) * mul);
          if (row_ok) {
            if (b >= p.B || hkv >= p.Hkv) {
              atomicOr(&g_backward_err, kErrBounds);
              continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(row + q4 * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, bw::TMEM_COLS);
  }
  // Aborted CTA: wait, bounded, for the loads that may still be in flight.
  if (warp == PRODUCER && *abort_flag) {
    const uint32_t first = prod_st > (uint32_t)NS ? prod_st - NS : 0u;
    for (uint32_t u = first; u < prod_st; ++u) mbar_wait_drain(&full[u % NS], (u / NS) & 1);
    if (prod_kv_any) mbar_wait_drain(kv_full, prod_kv_par);
    __syncwarp();
  }
}


// ------------------------------------------------------------------------------
// dkdv, D = 128: 128-row query sub-tiles, one TMEM buffer.
//
// TMEM: S^T [0, 128) | dP^T [128, 256) | dV [256, 384) | dK [384, 512).
// S^T = K Q^T and dP^T = V dO^T are N = 128 products (a 64-row sub-tile
// makes them N = 64, whose shared-memory operand reads, not the tensor math,
// set their rate).  There is no room for a second S^T / dP^T buffer, so the
// steps overlap this way:
//   the element-wise warps read all of S^T(u) into registers and say so
//   (s_free); S^T(u+1) is issued then, so P(u+1) is computed while the MMAs
//   of step u still run;
//   P^T and dS^T (16-bit) of query half h go over the dP^T columns of that
//   half, and each half is signalled on its own, so dV, dK of half 0 run
//   while half 1 is computed;
//   dP^T(u+1) follows dV, dK of half 1, the last readers of its columns.
// Shared memory holds K, V, a 3-slot Q ring, a 2-slot dO ring and a 2-slot
// ring of the sub-tiles' lse and Delta rows, each ring with its own
// barriers: S^T(u+1) waits only for Q(u+1), whose slot frees two steps
// earlier than a combined Q / dO stage would.
// Eight element-wise warps: warp w serves TMEM lane quarter w % 4 and query
// columns 32 (w / 4) + [0, 32) of each half.  A thread writes its 16-bit
// results only over columns it has already read, so the two warps of a lane
// quarter never touch each other's columns.
// ------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(10 * 32, 1)
    bwd_dkdv_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  constexpr int D = 128;
  using C = bw::Cfg<D>;
  using W = bw::Wide;
  constexpr bool kBF16 = BIsBF16<T>::value;
  constexpr int QN = W::QSLOTS, DN = W::DOSLOTS, LN = W::LDSLOTS;
  constexpr int QW = bw::BT;                 // query rows of a sub-tile
  constexpr int EW = 8, PRODUCER = 8, MMA = 9;
  extern __shared__ uint8_t smem_raw[];
  // The launch reserves W::PAD_MAX bytes for aligning the tiles to 1 KiB.  A
  // base needing more (not seen: the dynamic shared window starts aligned)
  // is reported, and the CTA leaves before touching shared memory.
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > (uint32_t)W::PAD_MAX) {
    if (threadIdx.x == 0) atomicOr(&g_backward_err, kErrBounds | (15u << 8));
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::TILE_BYTES;
  uint8_t* sQ = smem + 2 * C::TILE_BYTES;  // [QN] Q tiles
  uint8_t* sDO = sQ + QN * C::TILE_BYTES;  // [DN] dO tiles
  float* sLD = reinterpret_cast<float*>(sDO + DN * C::TILE_BYTES);  // [LN][lse*log2e, Delta][QW]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sLD + LN * 2 * QW);
  uint64_t* q_full = bars;              // [QN] producer (expect_tx)
  uint64_t* q_empty = q_full + QN;      // [QN] MMA commit
  uint64_t* do_full = q_empty + QN;     // [DN] producer (expect_tx)
  uint64_t* do_empty = do_full + DN;    // [DN] MMA commit
  uint64_t* ld_full = do_empty + DN;    // [LN] producer, after its shared-memory writes
  uint64_t* ld_empty = ld_full + LN;    // [LN] one arrival per element-wise thread
  uint64_t* kv_full = ld_empty + LN;
  uint64_t* kv_empty = kv_full + 1;
  uint64_t* s_full = kv_full + 2;   // S^T(u) in TMEM
  uint64_t* dp_full = kv_full + 3;  // dP^T(u) in TMEM
  uint64_t* h_ready = kv_full + 4;  // [2] P^T / dS^T of query half h (all element-wise threads)
  uint64_t* o_full = kv_full + 6;   // dK, dV complete
  uint64_t* drain = kv_full + 7;
  uint64_t* s_free = kv_full + 8;   // S^T(u) read into registers (all element-wise threads)
  uint64_t* sched_full = kv_full + 9;                // [kSchedSlots]
  uint64_t* sched_empty = sched_full + kSchedSlots;  // [kSchedSlots]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sched_empty + kSchedSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* sched = abort_flag + 1;  // [kSchedSlots]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < QN; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < DN; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    for (int s = 0; s < LN; ++s) {
      mbar_init(&ld_full[s], 1);
      mbar_init(&ld_empty[s], EW * 32);
    }
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(&h_ready[0], EW * 32);
    mbar_init(&h_ready[1], EW * 32);
    mbar_init(s_free, EW * 32);
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(&sched_full[i], 1);
      mbar_init(&sched_empty[i], EW + 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA) {
    tmem_alloc(tmem_holder, bw::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const bool leader = lane == 0;
  const int off = p.Sk - p.Sq;
  const int n_qw = (p.Sq + QW - 1) / QW;
  // First query sub-tile that sees key row k0 (n_qw if none).
  auto first_sub = [&](int k0) {
    if (!p.causal) return 0;
    const int i0 = k0 - off;  // the first query row that sees key k0
    if (i0 >= p.Sq) return n_qw;
    return i0 <= 0 ? 0 : i0 / QW;
  };
  constexpr uint32_t COL_DP = 128, COL_DV = 256, COL_DK = 384;
  // The producer's loads that may still be in flight if the CTA aborts: the
  // last QN Q tiles, the last DN dO tiles, the K / V tiles of its last item.
  uint32_t prod_q = 0, prod_do = 0, prod_kv_par = 0;
  bool prod_kv_any = false;

  if (warp == PRODUCER) {
    // ================================ producer ================================
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
    }
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    uint32_t st = 0, local = 0;  // st: sub-tile steps so far (slots, parities)
    bool ok = true;
    for (uint32_t k = 0; ok; ++k, ++local) {
      const int w = sched_produce(k, p.work_ctr, p.n_items, sched_full, sched_empty, sched,
                                  abort_flag, &g_backward_err, leader);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hkv, kt;
      dkv_item(w, p, &b, &hkv, &kt);
      const int q0 = first_sub(kt * bw::BT);
      if (local > 0 &&
          !(ok = mbar_wait(kv_empty, (local - 1) & 1, abort_flag, &g_backward_err, 1)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_4d_hint(sK + h * bw::HALF_BYTES, &tmK, kv_full, h * 64, hkv, kt * bw::BT, b,
                           pol_kv);
          tma_load_4d_hint(sV + h * bw::HALF_BYTES, &tmV, kv_full, h * 64, hkv, kt * bw::BT, b,
                           pol_kv);
        }
      }
      __syncwarp();
      prod_kv_par = local & 1;
      prod_kv_any = true;
      // Query sub-tiles descending, the group's heads innermost: the items of
      // one kv head then read the same Q / dO tiles at about the same time.
      for (int qs = n_qw - 1; qs >= q0 && ok; --qs) {
        for (int g = 0; g < p.G && ok; ++g, ++st) {
          const int hq = hkv * p.G + g;
          // lse * log2(e) and Delta of the sub-tile's query rows (+inf / 0
          // past Sq: those columns get P = 0), read before the waits so that
          // their latency is off the rings' paths.
          const size_t base = ((size_t)b * p.Hq + hq) * p.Sq;
          float lv[QW / 32], dv[QW / 32];
#pragma unroll
          for (int x = 0; x < QW / 32; ++x) {
            const int i = qs * QW + x * 32 + lane;
            lv[x] = i < p.Sq ? p.lse[base + i] * bw::LOG2E : INFINITY;
            dv[x] = i < p.Sq ? p.delta[base + i] : 0.f;
          }
          // Q first (S^T needs only Q), then dO, then the lse / Delta rows.
          const int qsl = st % QN, dsl = st % DN, lsl = st % LN;
          if (!(ok = mbar_wait(&q_empty[qsl], ((st / QN) & 1) ^ 1, abort_flag, &g_backward_err,
                               2)))
            break;
          if (leader) {
            mbar_arrive_expect_tx(&q_full[qsl], C::TILE_BYTES);
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h)
              tma_load_4d_hint(sQ + qsl * C::TILE_BYTES + h * bw::HALF_BYTES, &tmQ, &q_full[qsl],
                               h * 64, hq, qs * QW, b, pol_q);
          }
          __syncwarp();
          prod_q = st + 1;
          if (!(ok = mbar_wait(&do_empty[dsl], ((st / DN) & 1) ^ 1, abort_flag, &g_backward_err,
                               2)))
            break;
          if (leader) {
            mbar_arrive_expect_tx(&do_full[dsl], C::TILE_BYTES);
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h)
              tma_load_4d_hint(sDO + dsl * C::TILE_BYTES + h * bw::HALF_BYTES, &tmDO,
                               &do_full[dsl], h * 64, hq, qs * QW, b, pol_q);
          }
          __syncwarp();
          prod_do = st + 1;
          if (!(ok = mbar_wait(&ld_empty[lsl], ((st / LN) & 1) ^ 1, abort_flag, &g_backward_err,
                               2)))
            break;
          float* sL = sLD + lsl * 2 * QW;
          float* sD = sL + QW;
#pragma unroll
          for (int x = 0; x < QW / 32; ++x) {
            sL[x * 32 + lane] = lv[x];
            sD[x * 32 + lane] = dv[x];
          }
          __syncwarp();
          if (leader) mbar_arrive(&ld_full[lsl]);  // after the shared-memory writes
          __syncwarp();
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA) {
    // ================================== MMA ===================================
    // Lane 0 alone runs the issuer loop; descriptors advance on their low 32
    // bits (see mma_ss_lh).
    if (lane == 0) {
      const uint32_t sd_hi = (uint32_t)(sdesc_sw128(0u, 16, 1024) >> 32);
      constexpr uint32_t IDESC_S = idesc_f16(bw::BT, QW, kBF16, false);
      constexpr uint32_t IDESC_ACC = idesc_f16(bw::BT, D, kBF16, true);
      const uint32_t sk_addr = smem_u32(sK), sv_addr = smem_u32(sV);
      const uint32_t sq_addr = smem_u32(sQ), sdo_addr = smem_u32(sDO);
      uint32_t st = 0, local = 0;
      bool ok = true;
      // D_tmem (128 x 128) = A (128-row tile, K-major) x B^T (128-row tile, K-major).
      auto issue_nt = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
        const uint32_t a0 = (uint32_t)sdesc_sw128(a_addr, 16, 1024);
        const uint32_t b0 = (uint32_t)sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t k16 = ((k >> 2) * bw::HALF_BYTES + (k & 3) * 32) >> 4;
          mma_ss_lh(tmem + d_col, a0 + k16, sd_hi, b0 + k16, sd_hi, IDESC_S, k > 0 ? 1u : 0u);
        }
      };
      // acc += A (TMEM, 16-bit) x B (rows 64 h .. 64 h + 63 of a 128-row
      // tile, MN-major).  The half's 16-bit A columns are two runs of 16, one
      // per element-wise warp of the lane quarter, 32 columns apart: k-steps
      // 2e and 2e + 1 read columns a_col + 32 e and a_col + 32 e + 8.
      auto issue_acc = [&](uint32_t d_col, uint32_t a_col, uint32_t b_addr, int h,
                           bool accumulate) {
        const uint32_t b0 =
            (uint32_t)sdesc_sw128(b_addr + h * (QW / 2) * 128, bw::HALF_BYTES, 1024);
#pragma unroll
        for (int k = 0; k < QW / 2 / 16; ++k) {
          mma_ts_lh(tmem + d_col, tmem + a_col + (k >> 1) * 32 + (k & 1) * 8,
                    b0 + (uint32_t)((k * 16 * 128) >> 4), sd_hi, IDESC_ACC,
                    (accumulate || k > 0) ? 1u : 0u);
        }
      };
      auto commit = [&](uint64_t* bar) { mma_commit(bar); };
      auto q_addr = [&](uint32_t t) { return sq_addr + (t % QN) * C::TILE_BYTES; };
      auto do_addr = [&](uint32_t t) { return sdo_addr + (t % DN) * C::TILE_BYTES; };
      auto wait_q = [&](uint32_t t) {
        return mbar_wait(&q_full[t % QN], (t / QN) & 1, abort_flag, &g_backward_err, 4);
      };
      auto wait_do = [&](uint32_t t) {
        return mbar_wait(&do_full[t % DN], (t / DN) & 1, abort_flag, &g_backward_err, 4);
      };
      for (uint32_t it = 0; ok; ++it, ++local) {
        const int w =
            sched_consume_lane(it, sched_full, sched_empty, sched, abort_flag, &g_backward_err,
                               11);
        if (w < 0) {
          ok = w == -1;
          break;
        }
        int b, hkv, kt;
        dkv_item(w, p, &b, &hkv, &kt);
        const int steps = p.G * (n_qw - first_sub(kt * bw::BT));
        if (!(ok = mbar_wait(kv_full, local & 1, abort_flag, &g_backward_err, 3))) break;
        tc_fence_after();
        if (steps > 0) {
          if (!(ok = wait_q(st))) break;
          tc_fence_after();
          issue_nt(0, sk_addr, q_addr(st));  // S^T(0) = K Q^T
          commit(s_full);
          if (!(ok = wait_do(st))) break;
          tc_fence_after();
          issue_nt(COL_DP, sv_addr, do_addr(st));  // dP^T(0) = V dO^T
          commit(dp_full);
        }
        for (int u = 0; u < steps && ok; ++u, ++st) {
          const uint32_t g = st;  // step counter shared with the element-wise warps
          // S^T(u+1) as soon as the element-wise warps hold S^T(u) in
          // registers: no 16-bit result is written over S^T.
          if (!(ok = mbar_wait(s_free, g & 1, abort_flag, &g_backward_err, 5))) break;
          if (u + 1 < steps) {
            if (!(ok = wait_q(st + 1))) break;
            tc_fence_after();
            issue_nt(0, sk_addr, q_addr(st + 1));
            commit(s_full);
          }
          // Half 0: P^T and dS^T over dP^T columns [128, 192).
          if (!(ok = mbar_wait(&h_ready[0], g & 1, abort_flag, &g_backward_err, 5))) break;
          tc_fence_after();
          issue_acc(COL_DV, COL_DP, do_addr(st), 0, u > 0);       // dV += P^T dO
          issue_acc(COL_DK, COL_DP + 16, q_addr(st), 0, u > 0);   // dK += dS^T Q
          // Half 1: P^T and dS^T over dP^T columns [192, 256).
          if (!(ok = mbar_wait(&h_ready[1], g & 1, abort_flag, &g_backward_err, 5))) break;
          tc_fence_after();
          issue_acc(COL_DK, COL_DP + 80, q_addr(st), 1, true);
          commit(&q_empty[st % QN]);
          issue_acc(COL_DV, COL_DP + 64, do_addr(st), 1, true);
          commit(&do_empty[st % DN]);
          if (u + 1 < steps) {
            if (!(ok = wait_do(st + 1))) break;
            tc_fence_after();
            issue_nt(COL_DP, sv_addr, do_addr(st + 1));
            commit(dp_full);
          }
        }
        if (!ok) break;
        commit(kv_empty);
        commit(o_full);
      }
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    // ================== P^T and dS^T (element-wise warps) ==================
    const int quarter = warp & 3, e = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane = key row within the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t st = 0, o_cnt = 0;
    bool ok = true;
    T* const DK = static_cast<T*>(p.dk);
    T* const DV = static_cast<T*>(p.dv);
    const float2 c2 = make_float2(p.c, p.c);
    for (uint32_t it = 0; ok; ++it) {
      const int w =
          sched_consume(it, sched_full, sched_empty, sched, abort_flag, &g_backward_err, 12);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      int b, hkv, kt;
      dkv_item(w, p, &b, &hkv, &kt);
      const int q0 = first_sub(kt * bw::BT);
      const int j = kt * bw::BT + r;  // key row
      for (int qs = n_qw - 1; qs >= q0 && ok; --qs) {
        for (int g = 0; g < p.G && ok; ++g, ++st) {
          const int lsl = st % LN;
          if (!(ok = mbar_wait(&ld_full[lsl], (st / LN) & 1, abort_flag, &g_backward_err, 9)))
            break;
          if (!(ok = mbar_wait(s_full, st & 1, abort_flag, &g_backward_err, 7))) break;
          __syncwarp();
          tc_fence_after();
          const float* sL = sLD + lsl * 2 * QW;
          const float* sD = sL + QW;
          // Query row i = qs * 128 + ic sees key j when i < Sq and (not causal
          // or j <= i + off).  Rows past Sq have lse = +inf (P = 0); key rows
          // past Sk read zeros and feed only dK / dV rows never stored.  Only
          // a sub-tile on the causal edge hides columns (ic < ic_lo).
          const int ic_lo = p.causal ? j - off - qs * QW : 0;
          const bool edge = __any_sync(0xffffffffu, ic_lo > 0);
          // P of this thread's 32 columns of both halves, from S^T.
          uint32_t pv[2][32];
          tmem_ld32(t_lane + e * 32, pv[0]);
          tmem_ld32(t_lane + 64 + e * 32, pv[1]);
          tmem_wait_ld();
          reg_fence32(pv[0]);
          reg_fence32(pv[1]);
          tc_fence_before();
          mbar_arrive(s_free);  // S^T(u+1) may now be written over S^T(u)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {
              const float4 l4 = reinterpret_cast<const float4*>(sL)[h * 16 + e * 8 + x4];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int x = x4 * 2 + hh;
                const float2 nl = hh ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
                const float2 a = __ffma2_rn(make_float2(__uint_as_float(pv[h][2 * x]),
                                                        __uint_as_float(pv[h][2 * x + 1])),
                                            c2, nl);
                float2 pf = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                if (edge) {
                  const int col = h * 64 + e * 32 + 2 * x;
                  pf.x = col < ic_lo ? 0.f : pf.x;
                  pf.y = col + 1 < ic_lo ? 0.f : pf.y;
                }
                pv[h][2 * x] = __float_as_uint(pf.x);
                pv[h][2 * x + 1] = __float_as_uint(pf.y);
              }
            }
          }
          if (!(ok = mbar_wait(dp_full, st & 1, abort_flag, &g_backward_err, 7))) break;
          __syncwarp();
          tc_fence_after();
          uint32_t pr[2][32];
          tmem_ld32(t_lane + COL_DP + e * 32, pr[0]);
          tmem_ld32(t_lane + COL_DP + 64 + e * 32, pr[1]);
          tmem_wait_ld();
          reg_fence32(pr[0]);
          reg_fence32(pr[1]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pp[16], pd[16];
#pragma unroll
            for (int x4 = 0; x4 < 8; ++x4) {
              const float4 d4 = reinterpret_cast<const float4*>(sD)[h * 16 + e * 8 + x4];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int x = x4 * 2 + hh;
                const float2 nd = hh ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
                const float2 pf = make_float2(__uint_as_float(pv[h][2 * x]),
                                              __uint_as_float(pv[h][2 * x + 1]));
                const float2 dd = __fadd2_rn(make_float2(__uint_as_float(pr[h][2 * x]),
                                                         __uint_as_float(pr[h][2 * x + 1])),
                                             nd);
                const float2 ds = __fmul2_rn(pf, dd);
                pp[x] = BPack<T>::pack(pf.x, pf.y);
                pd[x] = BPack<T>::pack(ds.x, ds.y);
              }
            }
            // P^T, then dS^T, over the 32 dP^T columns of half h this thread read.
            tmem_st16(t_lane + COL_DP + h * 64 + e * 32, pp);
            tmem_st16(t_lane + COL_DP + h * 64 + e * 32 + 16, pd);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&h_ready[h]);
          }
          mbar_arrive(&ld_empty[lsl]);  // this thread is done with the slot's lse / Delta
        }
      }
      if (!ok) break;
      // Epilogue: dV, dK (= scale * accumulator) of this thread's key row;
      // each warp of a lane quarter stores half of the D columns.
      if (!(ok = mbar_wait(o_full, o_cnt & 1, abort_flag, &g_backward_err, 8))) break;
      ++o_cnt;
      __syncwarp();
      tc_fence_after();
      const bool any = p.G * (n_qw - q0) > 0;
      const bool row_ok = j < p.Sk;
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
        T* const row =
            (which ? DK : DV) + (((size_t)b * p.Sk + (row_ok ? j : 0)) * p.Hkv + hkv) * D;
        const float mul = which ? p.scale : 1.f;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int q4 = e * 2 + qq;
          uint32_t ar[32];
          if (any) {
            tmem_ld32(t_lane + (which ? COL_DK : COL_DV) + q4 * 32, ar);
            tmem_wait_ld();
            reg_fence32(ar);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) ar[x] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            pk[x] = BPack<T>::pack(__uint_as_float(ar[2 * x]) * mul,
                                   __uint_as_float(ar[2 * x + 1]) * mul);
          if (row_ok) {
            if (b >= p.B || hkv >= p.Hkv) {
              atomicOr(&g_backward_err, kErrBounds);
              continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(row + q4 * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, bw::TMEM_COLS);
  }
  // Aborted CTA: wait, bounded, for the loads that may still be in flight.
  if (warp == PRODUCER && *abort_flag) {
    for (uint32_t t = prod_q > (uint32_t)QN ? prod_q - QN : 0u; t < prod_q; ++t)
      mbar_wait_drain(&q_full[t % QN], (t / QN) & 1);
    for (uint32_t t = prod_do > (uint32_t)DN ? prod_do - DN : 0u; t < prod_do; ++t)
      mbar_wait_drain(&do_full[t % DN], (t / DN) & 1);
    if (prod_kv_any) mbar_wait_drain(kv_full, prod_kv_par);
    __syncwarp();
  }
}

// ------------------------------------------------------------------------------
// Host
// ------------------------------------------------------------------------------
template <int D, typename T>
static int launch_backward_t(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             float* delta, int B, int Hq, int Hkv, int Sq, int Sk, float scale,
                             int causal, cudaStream_t stream) {
  using C = bw::Cfg<D>;
  // The two work counters follow Delta in the scratch.
  unsigned int* ctr = reinterpret_cast<unsigned int*>(delta + (size_t)B * Hq * Sq);
  // pre: Delta
  {
    // A grid-stride loop over as many blocks as fit on the SMs at once (each
    // warp with PRE_STEPS steps of loads in flight), fewer when the rows run
    // out first.
    static int per_sm = 0;
    if (per_sm <= 0 &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bwd_pre_kernel<D, T>, 256, 0) !=
            cudaSuccess)
      per_sm = 2;
    if (per_sm <= 0) per_sm = 1;
    const size_t rows = (size_t)B * Sq * Hq;
    const size_t rows_per_block = (size_t)8 * (32 / (D / 8)) * PRE_STEPS;
    const size_t cap = (size_t)(sm_count() > 0 ? sm_count() : 148) * per_sm;
    const size_t want = (rows + rows_per_block - 1) / rows_per_block;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    bwd_pre_kernel<D, T><<<blocks, 256, 0, stream>>>(static_cast<const T*>(o),
                                                     static_cast<const T*>(dout), delta, B, Sq,
                                                     Hq, ctr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tq, tk, tv, tdo;
  if (encode_tmap_rows(&tq, q, D, Hq, Sq, B, bw::BT)) return cudaErrorInvalidValue;
  if (encode_tmap_rows(&tdo, dout, D, Hq, Sq, B, bw::BT)) return cudaErrorInvalidValue;
  if (encode_tmap_rows(&tk, k, D, Hkv, Sk, B, bw::BT)) return cudaErrorInvalidValue;
  if (encode_tmap_rows(&tv, v, D, Hkv, Sk, B, bw::BT)) return cudaErrorInvalidValue;
  // The D = 64 dkdv kernel reads Q and dO in 64-row sub-tiles.
  CUtensorMap tq64, tdo64;
  if (D == 64) {
    if (encode_tmap_rows(&tq64, q, D, Hq, Sq, B, bw::QS)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tdo64, dout, D, Hq, Sq, B, bw::QS)) return cudaErrorInvalidValue;
  }
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D, T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_DQ);
    if (e != cudaSuccess) return e;
    if constexpr (D == 128) {
      e = cudaFuncSetAttribute(bwd_dkdv_wide_kernel<T>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, bw::Wide::SMEM);
    } else {
      e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, T>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_DKV);
    }
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  BwdParams p;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.lse = lse;
  p.delta = delta;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.G = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.n_qt = (Sq + bw::BT - 1) / bw::BT;
  p.n_kt = (Sk + bw::BT - 1) / bw::BT;
  p.scale = scale;
  p.c = scale * bw::LOG2E;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  p.n_items = B * Hq * p.n_qt;
  p.work_ctr = ctr;
  if (p.n_items > 0) {
    const int grid = p.n_items < sms ? p.n_items : sms;
    bwd_dq_kernel<D, T><<<grid, bw::THREADS, C::SMEM_DQ, stream>>>(tq, tk, tv, tdo, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  p.n_items = B * Hkv * p.n_kt;
  p.work_ctr = ctr + 1;
  if (p.n_items > 0) {
    const int grid = p.n_items < sms ? p.n_items : sms;
    if constexpr (D == 128)
      bwd_dkdv_wide_kernel<T><<<grid, 10 * 32, bw::Wide::SMEM, stream>>>(tq, tk, tv, tdo, p);
    else
      bwd_dkdv_kernel<D, T><<<grid, C::DKV_THREADS, C::SMEM_DKV, stream>>>(tq64, tk, tv, tdo64, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int launch_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, float* delta, int B, int Hq,
                    int Hkv, int Sq, int Sk, int D, float scale, int causal, bool bf16,
                    cudaStream_t stream) {
  if (D == 64)
    return bf16 ? launch_backward_t<64, __nv_bfloat16>(q, k, v, o, dout, lse, dq, dk, dv, delta,
                                                       B, Hq, Hkv, Sq, Sk, scale, causal, stream)
                : launch_backward_t<64, __half>(q, k, v, o, dout, lse, dq, dk, dv, delta, B, Hq,
                                                Hkv, Sq, Sk, scale, causal, stream);
  return bf16 ? launch_backward_t<128, __nv_bfloat16>(q, k, v, o, dout, lse, dq, dk, dv, delta, B,
                                                      Hq, Hkv, Sq, Sk, scale, causal, stream)
              : launch_backward_t<128, __half>(q, k, v, o, dout, lse, dq, dk, dv, delta, B, Hq,
                                               Hkv, Sq, Sk, scale, causal, stream);
}

int set_backward_wait_limit(unsigned long long ns) { return set_wait_limit_this_unit(ns); }

int read_backward_error(unsigned int* out, int reset) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_backward_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (reset && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_backward_err, &z, sizeof(z));
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return 0;
}

}  // namespace fa
