// fa_decode.cu -- single-token decode: split-KV kernel + log-sum-exp combine.
//
// What it computes: for every query head h of every batch entry b,
//   O[b,h,:] = sum_{j<L} p_j V[b,j,h/G,:] / sum_{j<L} p_j,
//   p_j = exp(scale * <q[b,h], K[b,j,h/G]> - max),
// over the first L tokens of a token-major [B, cap, Hkv, D] cache, where L is
// an int32 in device memory (rocm-libraries #13108 "minimal single-token
// attention decode", interface description).  The same PR's review showed that
// loading whole tiles lets NaN in unused capacity reach P@V through 0*NaN; here
// every K/V row at a token >= L is overwritten with zeros in shared memory
// before any MMA touches the tile, and its score is set to -inf.  Split-KV is
// the step that PR names as its next optimisation.
//
// Design (HBM-bound: 2*L*Hkv*D*2 bytes read, ~4 flop per byte):
//   grid   = (nsplit, Hkv * ceil(G/16), B), one CTA per SM, sized from cap and
//            the SM count (not from L, which the host never reads);
//   CTA    = 1 producer warp issuing TMA tile loads (64 tokens x D, K and V,
//            128-byte swizzle) into a 6-stage mbarrier ring (12 for D = 64,
//            192 KiB in flight), and 3 consumer warps that each own whole
//            tiles (paged caches whose pages are not a multiple of 64 tokens:
//            32-token tiles over 4 warps):
//            S^T = K Q^T and O^T += V^T P^T with mma.sync m16n8k16,
//            tokens as the MMA's M and the group's query heads as its N (8 per
//            block, so a GQA group of 4 wastes half of N instead of 3/4 of a
//            16-row M), an exp2 online softmax per warp, then a cross-warp
//            merge in shared memory into one (max, sum, o[D]) partial per head
//            and split;
//   combine= one CTA per (32 columns, head, b) merges the split partials with
//            weights exp2(m_s - M).
// Both kernels are launched as programmatic dependents of the grid before
// them.  Before its griddepcontrol.wait the split kernel only initialises its
// barriers and prefetches (tensor maps, and its first K/V tiles into L2), so
// in a sequence of calls the next call's prologue and first HBM reads overlap
// the current call's merge, combine and grid boundaries.
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ unsigned int g_decode_err = 0;

namespace dec {
constexpr int TT = 32;        // the smallest tile: pages are multiples of it
constexpr int NWARPS = 4;     // consumer warps, at most (32-token tiles)
constexpr int THREADS = (NWARPS + 1) * 32;
constexpr int HB = 16;        // row stride of the merge buffers (query rows per CTA at most)
// Bytes of K/V per CTA warmed in L2 before the grid wait: with one CTA per SM
// that is at most about half of L2 in flight, whatever the cache length.
constexpr int PREFETCH_BYTES = 384 * 1024;

// Tile t lives in stage t % NSTAGE and is consumed by warp t % NW.  With
// NSTAGE a multiple of NW every stage belongs to exactly one warp, which
// therefore waits on that stage's phases strictly in order.  (A parity wait
// must never run ahead by a phase: if two warps shared a stage, the faster one
// could see the stage's previous phase as "complete" and consume a tile that
// has not landed.)
// TILE = 64: 64-token tiles (64-row TMA boxes; an SM takes in 32-row boxes
// more slowly), 3 consumer warps with 2 stages each, 192 KiB in flight: the
// bytes in flight per SM set the rate of a long stream from HBM.
// Pages that are not a multiple of 64 tokens take TILE = 32 (32-token tiles
// over 4 warps).
template <int D, bool PAGED = false, int TILE = 64>
struct Cfg {
  static constexpr int HALVES = D / 64;
  static constexpr int TT = TILE;  // tokens per tile (32 or 64)
  static constexpr int NW = TILE == 64 ? 3 : dec::NWARPS;  // consumer warps
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int HALF_BYTES = TT * 128;  // TT rows x 64 elements x 2 bytes
  static constexpr int NSTAGE = (D == 128 ? 1 : 2) * (PAGED ? (TILE == 64 ? 6 : 12) : 6);
  static constexpr int KV_BYTES = HALVES * HALF_BYTES;  // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;      // K tile + V tile
  static constexpr int SMEM_STAGES = NSTAGE * STAGE_BYTES;
  static_assert(NSTAGE % NW == 0, "each stage must belong to one consumer warp");
  static constexpr int SMEM_RED = NW * HB * D * 4 + NW * HB * 2 * 4 + NW * HB * 4;
  static constexpr int SMEM_BAR = 2 * NSTAGE * 8 + 16 + NSTAGE * 4;
  static_assert(HALF_BYTES % 1024 == 0, "128-byte-swizzled tiles need 1 KiB alignment");
  static constexpr int SMEM_TOTAL = 1024 + SMEM_STAGES + SMEM_RED + SMEM_BAR;
  static_assert(SMEM_TOTAL <= 227 * 1024, "shared memory per CTA");
};
}  // namespace dec

struct DecodeParams {
  const __nv_bfloat16* q;    // [B, Hq, D]
  const int32_t* valid_len;  // device: L of batch entry b is valid_len[b * len_stride]
  int len_stride;            // 0: one L for the batch; 1: one per sequence
  // Paged caches: K/V pages [num_pages, page_size, Hkv, D], page_table
  // [B, max_pages] (device).  Null for contiguous [B, cap, Hkv, D] caches.
  const int32_t* page_table;
  int page_size, max_pages, num_pages;
  float* part_o;             // [B, Hq, nsplit, D] unnormalised partial outputs
  float* part_ml;            // [B, Hq, nsplit, 2] (row max in log2 units, row sum)
  __nv_bfloat16* o;          // [B, Hq, D]
  float* lse;                // [B, Hq] natural-log log-sum-exp per head, or null
  int B, Hq, Hkv, cap, G, nsplit, n_hb;
  // Balanced splits (paged caches only): the grid is nsplit CTAs in x, and
  // each finds its (sequence, kv head, row block, split) from the lengths;
  // partials are indexed by CTA (part_o [nsplit, HB, D], part_ml
  // [nsplit, HB, 2]), and CTA 0 writes unit_map[u] = (first CTA, splits) of
  // every unit u = (b * Hkv + hkv) * n_hb + hb for the combine.  0: the grid
  // is (nsplit, Hkv * n_hb, B).
  int balanced;
  int2* unit_map;
  // New query tokens per sequence (paged path; 1 otherwise).  The MMA's 16
  // rows are (token, head) pairs r = s * G + g of one kv head; token s sees
  // the keys [0, L - Sq + s] (bottom-right causal).
  int Sq;
  float c;                   // scale * log2(e)
};

// Query row of MMA row r (r = s * G + g) of kv head hkv in batch entry b: the
// index of (b, s, hkv * G + g) in [B, Sq, Hq].
__device__ __forceinline__ size_t decode_qrow(const DecodeParams& p, int b, int hkv, int r,
                                              int Sq) {
  const int s = r / p.G, g = r - s * p.G;
  return ((size_t)b * Sq + s) * p.Hq + (size_t)hkv * p.G + g;
}

// Balanced splits for a batch of sequences of different lengths (the lengths
// are device data, so the host cannot size the splits).  A unit is one
// (sequence, kv head, row block); a unit of sequence b has T_b = ceil(L_b / TT)
// K/V tiles.  Each unit of b gets S_b = ceil(T_b / lam) splits, lam being the
// smallest tile budget per split for which all units' splits fit the nsplit
// CTAs (binary search; lam = max T_b always fits, since there are fewer units
// than CTAs).  So no split holds more than lam tiles, and lam is within about
// one tile per unit of the even share.  The units of b take the CTAs (and
// partial slots) sP[b] + j * S_b + k, j = hkv * n_hb + hb, k < S_b.
// Block-cooperative, one thread per sequence (B <= blockDim.x); every thread
// of the block must call it, after griddepcontrol.wait; ends with
// __syncthreads().  sRed: 2 * warps entries.
__device__ void balanced_splits(const DecodeParams& p, int* sS, int* sP, long long* sRed, int tt) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = (blockDim.x + 31) >> 5;
  const int U = p.Hkv * p.n_hb;
  int T = 0;
  if (t < p.B) {
    int L = p.valid_len[(size_t)t * p.len_stride];
    L = L < 0 ? 0 : (L > p.cap ? p.cap : L);
    T = (L + tt - 1) / tt;
  }
  // Block sum of a (per thread) and block max of m, into every thread.
  auto reduce = [&](long long a, long long m, long long* sum, long long* mx) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      const long long y = __shfl_xor_sync(0xffffffffu, m, o);
      m = y > m ? y : m;
    }
    __syncthreads();  // the previous reduction has read sRed
    if (lane == 0) {
      sRed[2 * warp] = a;
      sRed[2 * warp + 1] = m;
    }
    __syncthreads();
    long long s2 = 0, m2 = 0;
    for (int w = 0; w < nw; ++w) {
      s2 += sRed[2 * w];
      m2 = sRed[2 * w + 1] > m2 ? sRed[2 * w + 1] : m2;
    }
    *sum = s2;
    *mx = m2;
  };
  long long all_tiles, max_t;
  reduce((long long)T * U, T, &all_tiles, &max_t);
  long long lam = 1;
  if (all_tiles > 0) {
    long long lo = (all_tiles + p.nsplit - 1) / p.nsplit, hi = max_t;
    if (lo < 1) lo = 1;
    if (lo > hi) lo = hi;
    while (lo < hi) {  // block-uniform: every thread sees the same sums
      const long long mid = (lo + hi) / 2;
      long long need, unused;
      reduce(T > 0 ? (long long)U * ((T + mid - 1) / mid) : 0, 0, &need, &unused);
      if (need <= p.nsplit)
        hi = mid;
      else
        lo = mid + 1;
    }
    lam = lo;
  }
  const int S = T > 0 ? (int)((T + lam - 1) / lam) : 0;
  // Exclusive prefix sum of U * S over the sequences.
  const int v = U * S;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();  // every thread has read sRed above
  if (lane == 31) sRed[warp] = inc;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += (int)sRed[w];
  if (t < p.B) {
    sS[t] = S;
    sP[t] = before + inc - v;
  }
  __syncthreads();
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Transpose of an 8x8 matrix of 16-bit elements held one 32-bit pair per lane
// (row lane/4, columns 2(lane%4), +1), returned in the same distribution.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// PAGED: K/V tiles are addressed through the page table (instantiated
// separately so the contiguous path carries none of the paging code).
// NB: query rows per CTA in blocks of 8 (the MMA's N): 1 when a kv head has at
// most 8 rows (GQA groups up to 8 with one new token), else 2.
template <int D, bool PAGED, int NB, int TILE>
__global__ void __launch_bounds__(dec::THREADS, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = dec::Cfg<D, PAGED, TILE>;
  constexpr int TT = C::TT, NSTAGE = C::NSTAGE, HB = dec::HB, NW = C::NW;
  constexpr int RB = 8 * NB;  // query rows of this CTA (HB is the buffers' row stride)
  static_assert(RB <= HB, "row blocks must fit the merge buffers");
  constexpr float NEG_INF = -INFINITY;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  float* red_o = reinterpret_cast<float*>(smem + C::SMEM_STAGES);  // [NW][HB][D]
  float* red_ml = red_o + NW * HB * D;                             // [NW][HB][2]
  float* red_w = red_ml + NW * HB * 2;                             // [NW][HB] merge weights
  uint64_t* full = reinterpret_cast<uint64_t*>(red_w + NW * HB);
  uint64_t* empty = full + NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NSTAGE);
  // Per stage: 1 when the producer could not map the tile to a valid page (its
  // tokens then count as masked); written before the stage's full barrier.
  volatile int* stage_bad = abort_flag + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This CTA's sequence, kv head, row block and split: from the grid, or in
  // balanced mode from the lengths once they can be read (below).
  int split = blockIdx.x;
  int hkv = blockIdx.y / p.n_hb, hb = blockIdx.y % p.n_hb;
  int b = blockIdx.z;

  // The combine grid may become resident now; it blocks until this grid ends.
  pdl_launch_dependents();
  // Prologue that reads nothing an earlier kernel may still be writing (the
  // tensor maps are kernel parameters); this kernel is launched as a
  // programmatic dependent, so it overlaps the tail of the previous grid.
  if (threadIdx.x == NW * 32) {  // producer lane 0: fetch the maps early
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  } else if (!PAGED && lane == 0 && warp < NW) {
    // Consumer lanes warm L2 with this CTA's first tiles while the previous
    // grid finishes (HBM is otherwise idle then).  L is read without ordering
    // here, so the tile range may be stale; that only wastes the prefetch --
    // nothing read before griddepcontrol.wait below reaches shared memory or
    // registers, and L2 stays coherent with any write still to come.
    int Ls = ld_relaxed_gpu(p.valid_len);
    Ls = Ls < 0 ? 0 : (Ls > p.cap ? p.cap : Ls);
    const int tt = (Ls + TT - 1) / TT;
    const int tp = (tt + p.nsplit - 1) / p.nsplit;
    const int tb = split * tp;
    int nt = tt - tb;
    nt = nt < 0 ? 0 : (nt > tp ? tp : nt);
    if (nt > dec::PREFETCH_BYTES / C::STAGE_BYTES) nt = dec::PREFETCH_BYTES / C::STAGE_BYTES;
    for (int t = warp; t < nt; t += NW) {
      const int tok = (tb + t) * TT;
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h) {
        tma_prefetch_l2_4d(&tmK, h * 64, hkv, tok, b);
        tma_prefetch_l2_4d(&tmV, h * 64, hkv, tok, b);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Everything below reads q, L and the caches, and writes the partials (which
  // the previous call's combine may still be reading): wait for the previous
  // grid in the stream to complete.
  pdl_wait_primary();

  int nsplit = p.nsplit;  // splits of this CTA's unit
  bool idle = false;      // balanced mode: a CTA beyond the splits in use
  if constexpr (PAGED) {
    if (p.balanced) {
      // The merge buffers are free until the end: scratch for the assignment.
      int* sS = reinterpret_cast<int*>(red_o);
      int* sP = sS + dec::THREADS;
      int* sRes = sP + dec::THREADS;
      long long* sRed = reinterpret_cast<long long*>(sRes + 8);
      if (threadIdx.x == 0) sRes[0] = -1;
      balanced_splits(p, sS, sP, sRed, TT);
      const int c = blockIdx.x, U = p.Hkv * p.n_hb;
      if (c == 0 && threadIdx.x < p.B) {  // the combine's map of every unit
        const int t = threadIdx.x;
        for (int j = 0; j < U; ++j) p.unit_map[t * U + j] = make_int2(sP[t] + j * sS[t], sS[t]);
      }
      if (threadIdx.x < p.B) {
        const int t = threadIdx.x, S = sS[t], first = sP[t];
        if (S > 0 && c >= first && c < first + U * S) {
          sRes[0] = t;
          sRes[1] = (c - first) / S;
          sRes[2] = (c - first) % S;
          sRes[3] = S;
        }
      }
      __syncthreads();
      if (sRes[0] < 0) {
        idle = true;
        b = 0;
        hkv = 0;
        hb = 0;
        split = 0;
        nsplit = 1;
      } else {
        b = sRes[0];
        hkv = sRes[1] / p.n_hb;
        hb = sRes[1] % p.n_hb;
        split = sRes[2];
        nsplit = sRes[3];
      }
    }
  }
  int L = idle ? 0 : (PAGED ? p.valid_len[(size_t)b * p.len_stride] : *p.valid_len);
  const int Sq = PAGED ? p.Sq : 1;  // compile-time 1 on the contiguous path
  L = L < 0 ? 0 : (L > p.cap ? p.cap : L);
  const int tiles_total = (L + TT - 1) / TT;
  const int tps = (tiles_total + nsplit - 1) / nsplit;
  const int t_begin = split * tps;
  int n_tiles = tiles_total - t_begin;
  n_tiles = n_tiles < 0 ? 0 : (n_tiles > tps ? tps : n_tiles);
  __syncthreads();

  const int g = lane >> 2, tq = lane & 3;
  // Tiles the producer issued (drained at the end if the CTA aborted).
  int prod_t = 0;

  if (warp == NW) {
    // ---------------- producer warp: lanes stay converged, lane 0 issues ----------------
    const bool leader = lane == 0;
    const uint64_t pol = l2_policy_evict_first();
    // Paged caches: lane l holds the page id of logical page pg_base + l, so
    // the page-table reads of 32 pages cost one load latency.
    int pg_base = -(1 << 30), pid_lane = 0;
    // Paged caches: the page of the next tile and the tile's row in it.  Tiles
    // advance by TT tokens and page_size is a multiple of TT, so they step
    // without a division per tile (the producer's issue rate paces long
    // streams).
    int page = 0, pos = 0;
    if constexpr (PAGED) {
      page = t_begin * TT / p.page_size;
      pos = t_begin * TT - page * p.page_size;
    }
    int t = 0;
    for (; t < n_tiles; ++t) {
      const int s = t % NSTAGE;
      const uint32_t ph = (t / NSTAGE) & 1;
      const int tok = (t_begin + t) * TT;
      int row = tok, tb = b, bad = 0;  // tensor-map row / batch coordinates of the tile
      if constexpr (PAGED) {
        if (page < pg_base || page >= pg_base + 32) {  // warp-uniform
          pg_base = page;
          const int pg = pg_base + lane;
          pid_lane = pg < p.max_pages ? p.page_table[(size_t)b * p.max_pages + pg] : -1;
        }
        const int pid = __shfl_sync(0xffffffffu, pid_lane, page - pg_base);
        bad = (pid < 0 || pid >= p.num_pages) ? 1 : 0;
        row = pos;
        tb = bad ? 0 : pid;  // a bad id loads page 0, and the tile is masked
        pos += TT;
        if (pos == p.page_size) {
          pos = 0;
          ++page;
        }
      }
      if (!mbar_wait<true>(&empty[s], ph ^ 1, abort_flag, &g_decode_err, 1)) break;
      if (leader) {
        if constexpr (PAGED) {
          stage_bad[s] = bad;
          if (bad) atomicOr(&g_decode_err, kErrBounds);
        }
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        uint8_t* st = stages + s * C::STAGE_BYTES;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h)
          tma_load_4d_hint(st + h * C::HALF_BYTES, &tmK, &full[s], h * 64, hkv, row, tb, pol);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h)
          tma_load_4d_hint(st + C::KV_BYTES + h * C::HALF_BYTES, &tmV, &full[s], h * 64, hkv,
                           row, tb, pol);
      }
      __syncwarp();
    }
    prod_t = t;
    __syncwarp();
  } else {
    // ---------------- consumers: whole tiles, round-robin over warps ----------------
    // Transposed products, so that the tile's tokens fill the MMA's M and the
    // CTA's few query rows only its N (8 per block):
    //   S^T = K Q^T   (A = K rows from shared memory, B = Q from registers),
    //   O^T += V^T P^T (A = V through transposing ldmatrix, B = P^T, which is
    //                   the S^T accumulator transposed per 8x8 by movmatrix).
    // Lane (g, tq) holds, for row block nb, rows nb*8 + 2tq + {0,1} of tokens
    // g and g + 8 of each 16-token block, and O^T at d = 16 dm + g (+8).
    const int rows_all = Sq * p.G;
    uint32_t qb[NB][D / 16][2];
    int vis[NB][2];  // keys [0, vis) visible to the lane's rows (paged: causal new tokens)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int r = hb * RB + nb * 8 + g;
      const bool ok = r < rows_all;
      const uint32_t* qr = reinterpret_cast<const uint32_t*>(
          p.q + decode_qrow(p, b, hkv, ok ? r : 0, Sq) * D);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qb[nb][kk][0] = ok ? qr[kk * 8 + tq] : 0u;
        qb[nb][kk][1] = ok ? qr[kk * 8 + 4 + tq] : 0u;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int rc = hb * RB + nb * 8 + 2 * tq + e;
        vis[nb][e] = L - Sq + 1 + (rc < rows_all ? rc / p.G : 0);
      }
    }
    float mr[NB][2], lr[NB][2];
    float acc[NB][D / 16][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mr[nb][e] = NEG_INF;
        lr[nb][e] = 0.f;
      }
#pragma unroll
      for (int dm = 0; dm < D / 16; ++dm) acc[nb][dm][0] = acc[nb][dm][1] = acc[nb][dm][2] = acc[nb][dm][3] = 0.f;
    }

    for (int t = warp; t < n_tiles; t += NW) {
      const int s = t % NSTAGE;
      const uint32_t ph = (t / NSTAGE) & 1;
      if (!mbar_wait<true>(&full[s], ph, abort_flag, &g_decode_err, 2)) break;
      __syncwarp();  // ldmatrix / mma.sync below are warp-collective
      uint8_t* st = stages + s * C::STAGE_BYTES;
      const int tok0 = (t_begin + t) * TT;
      // Tokens >= L (and every token of a tile with no valid page) are masked.
      const int nvalid = (PAGED && stage_bad[s]) ? 0 : ((L - tok0) < TT ? (L - tok0) : TT);
      if (nvalid < TT) {
        // Masked tokens: zero their K and V rows before any MMA reads the tile.
        const int nz = TT - nvalid;
        for (int x = lane; x < 2 * C::HALVES * nz * 8; x += 32) {
          const int chunk = x & 7;
          int r = x >> 3;
          const int row = nvalid + r % nz;
          r /= nz;
          const int half = r % C::HALVES;
          const int kv = r / C::HALVES;
          *reinterpret_cast<uint4*>(st + kv * C::KV_BYTES + half * C::HALF_BYTES + row * 128 +
                                    chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }

      // S^T: TT/16 token blocks x NB row blocks, 16 d per MMA.
      constexpr int MB = TT / 16;
      float sc[NB][MB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) sc[nb][mb][0] = sc[nb][mb][1] = sc[nb][mb][2] = sc[nb][mb][3] = 0.f;
      const uint32_t kbase = smem_u32(st);
      const int mi = lane >> 3;
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int tok = mb * 16 + (mi & 1) * 8 + (lane & 7);
          const int chunk = kk * 2 + (mi >> 1);
          const uint32_t addr = kbase + (chunk >> 3) * C::HALF_BYTES + tok * 128 +
                                ((((chunk & 7) ^ (tok & 7))) << 4);
          uint32_t a[4];
          ldsm_x4(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(sc[nb][mb], a, qb[nb][kk][0], qb[nb][kk][1]);
        }
      }
      // Scale into the log2 domain; mask tokens >= L (and, with several new
      // tokens, the keys after each row's own position).
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int mb = 0; mb < MB; ++mb)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tl = mb * 16 + g + (i >> 1) * 8;  // token within the tile
            sc[nb][mb][i] *= p.c;
            if constexpr (PAGED) {
              if (tok0 + tl >= vis[nb][i & 1] || tl >= nvalid) sc[nb][mb][i] = NEG_INF;
            } else {
              if (nvalid < TT && tl >= nvalid) sc[nb][mb][i] = NEG_INF;
            }
          }
      // Online softmax per row (column of S^T): the max over the tile's
      // tokens is over the lane's 2 x MB values and the 8 lanes of its tq.
      uint32_t pb[NB][MB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        float f[2], base[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx = NEG_INF;
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) mx = fmaxf(mx, fmaxf(sc[nb][mb][e], sc[nb][mb][2 + e]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(mr[nb][e], mx);
          base[e] = mn == NEG_INF ? 0.f : mn;
          f[e] = fast_exp2(mr[nb][e] - base[e]);
          mr[nb][e] = mn;
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sc[nb][mb][i] = fast_exp2(sc[nb][mb][i] - base[i & 1]);
            rs[i & 1] += sc[nb][mb][i];
          }
          // P^T B operand: rows tq-pairs of tokens g / g + 8, transposed per 8x8.
          pb[nb][mb][0] = movmatrix_trans(pack_bf16(sc[nb][mb][0], sc[nb][mb][1]));
          pb[nb][mb][1] = movmatrix_trans(pack_bf16(sc[nb][mb][2], sc[nb][mb][3]));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) lr[nb][e] = lr[nb][e] * f[e] + rs[e];
#pragma unroll
        for (int dm = 0; dm < D / 16; ++dm) {
          acc[nb][dm][0] *= f[0];
          acc[nb][dm][1] *= f[1];
          acc[nb][dm][2] *= f[0];
          acc[nb][dm][3] *= f[1];
        }
      }
      // O^T += V^T P^T: A = V^T (16 d x 16 tokens) by transposing ldmatrix.
      const uint32_t vbase = kbase + C::KV_BYTES;
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
        for (int dm = 0; dm < D / 16; ++dm) {
          const int tok = mb * 16 + (mi >> 1) * 8 + (lane & 7);
          const int chunk = dm * 2 + (mi & 1);
          const uint32_t addr = vbase + (chunk >> 3) * C::HALF_BYTES + tok * 128 +
                                ((((chunk & 7) ^ (tok & 7))) << 4);
          uint32_t a[4];
          ldsm_x4_t(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(acc[nb][dm], a, pb[nb][mb][0], pb[nb][mb][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // Per-warp row sums over the 8 lanes that share tq, then this warp's
    // (max, sum) and unnormalised O rows (only the CTA's real rows are kept).
    __syncwarp();
    const int nh_rows = (rows_all - hb * RB) < RB ? (rows_all - hb * RB) : RB;
    float* my_o = red_o + warp * HB * D;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = lr[nb][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int row = nb * 8 + 2 * tq + e;
        if (g == 0) {
          red_ml[(warp * HB + row) * 2 + 0] = mr[nb][e];
          red_ml[(warp * HB + row) * 2 + 1] = l;
        }
        if (row < nh_rows) {
#pragma unroll
          for (int dm = 0; dm < D / 16; ++dm) {
            my_o[row * D + dm * 16 + g] = acc[nb][dm][e];
            my_o[row * D + dm * 16 + g + 8] = acc[nb][dm][2 + e];
          }
        }
      }
    }
  }
  __syncthreads();

  // Merge the warps' partials (weights exp2(m_w - M)) and write this split's
  // partial for the CTA's heads: the weights once per row, then the outputs
  // four columns per thread.
  int nh = (Sq * p.G - hb * RB) < RB ? (Sq * p.G - hb * RB) : RB;
  // Query row of CTA row `row` (partials and outputs are indexed by it).
  auto qrow = [&](int row) { return decode_qrow(p, b, hkv, hb * RB + row, Sq); };
  // Partial slot of CTA row `row`: (query row, split), or in balanced mode
  // (CTA, row).
  const bool bal = PAGED && p.balanced;
  auto pslot = [&](int row) -> size_t {
    return bal ? (size_t)blockIdx.x * HB + row : qrow(row) * p.nsplit + split;
  };
  if (idle) nh = 0;  // no unit: nothing to write
  // Self-check: partial rows must lie inside the scratch (records and skips).
  if (b >= p.B || split >= nsplit || (!bal && split >= p.nsplit) ||
      (bal && (int)blockIdx.x >= p.nsplit) ||
      (nh > 0 && qrow(nh - 1) >= (size_t)p.B * Sq * p.Hq)) {
    if (threadIdx.x == 0) atomicOr(&g_decode_err, kErrBounds);
    nh = 0;
  }
  if (threadIdx.x < nh) {
    const int row = threadIdx.x;
    float M = NEG_INF;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_ml[(w * HB + row) * 2]);
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = red_ml[(w * HB + row) * 2];
      const float wt = (mw == NEG_INF) ? 0.f : fast_exp2(mw - M);
      red_w[w * HB + row] = wt;
      Ls += red_ml[(w * HB + row) * 2 + 1] * wt;
    }
    p.part_ml[pslot(row) * 2 + 0] = M;
    p.part_ml[pslot(row) * 2 + 1] = Ls;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < nh * (D / 4); x += C::THREADS) {
    const int row = x / (D / 4), d4 = x % (D / 4);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float wt = red_w[w * HB + row];
      const float4 v = reinterpret_cast<const float4*>(red_o + (w * HB + row) * D)[d4];
      o.x += v.x * wt;
      o.y += v.y * wt;
      o.z += v.z * wt;
      o.w += v.w * wt;
    }
    reinterpret_cast<float4*>(p.part_o + pslot(row) * D)[d4] = o;
  }
  // Aborted CTA (a wait gave up, in any warp, possibly after the producer
  // issued its last tile): wait, bounded, for the loads that may still be in
  // flight before the CTA exits.  Tiles older than the last NSTAGE have landed
  // (their stage was released before the producer reused it).
  if (warp == NW && *abort_flag) {
    for (int u = (prod_t - NSTAGE > 0 ? prod_t - NSTAGE : 0); u < prod_t; ++u)
      mbar_wait_drain(&full[u % NSTAGE], (u / NSTAGE) & 1);
    __syncwarp();
  }
}

// Combine: one CTA per (32 output columns, head, batch), 8 warps, up to
// kMaxSplits splits.  Every load is issued before any result is needed -- the
// split statistics (thread t: split t) and the partial outputs (lane = column,
// warp w: splits w, w+8, ...) -- so the kernel costs about one L2 round trip:
//   M = max over splits that saw a token (l_s > 0),
//   O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// Splits with l_s == 0 get weight 0 (their m_s may be -inf).  Launched with
// programmatic dependent launch; waits for the split grid in
// griddepcontrol.wait.
constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = kCombineWarps * 32;
constexpr int kMaxSplits = kCombineThreads;
constexpr int kSplitsPerWarp = kMaxSplits / kCombineWarps;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeParams p) {
  // A programmatic dependent launched after this grid (the next call's split
  // kernel) may start its prologue now; it waits for this grid to complete
  // before it reads or writes anything.
  pdl_launch_dependents();
  pdl_wait_primary();
  __shared__ float sW[kMaxSplits];
  __shared__ float sRed[kCombineWarps];
  __shared__ float sAcc[kCombineWarps][32];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int d = blockIdx.x * 32 + lane;
  const int h = blockIdx.y, b = blockIdx.z;
  if (h >= p.Sq * p.Hq || b >= p.B || p.nsplit > kMaxSplits) {
    if (t == 0) atomicOr(&g_decode_err, kErrBounds << 4);
    return;
  }
  const size_t base = ((size_t)b * p.Sq * p.Hq + h) * p.nsplit;  // h: row in [Sq, Hq]
  const int ns = p.nsplit;
  float ov[kSplitsPerWarp];
#pragma unroll
  for (int k = 0; k < kSplitsPerWarp; ++k) {
    const int sp = warp + k * kCombineWarps;
    ov[k] = (sp < ns && d < D) ? p.part_o[(base + sp) * D + d] : 0.f;
  }
  // (max, sum) of split t as one 8-byte load: selecting on the sum after a
  // second, dependent load would cost a second L2 round trip.
  float m_t = -INFINITY, l_t = 0.f;
  if (t < ns) {
    const float2 ml = reinterpret_cast<const float2*>(p.part_ml)[base + t];
    l_t = ml.y;
    m_t = l_t > 0.f ? ml.x : -INFINITY;
  }
  // M = block max of m_t.
  float M = m_t;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) sRed[warp] = M;
  __syncthreads();
  M = sRed[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, sRed[w]);
  const float w_t = (m_t == -INFINITY) ? 0.f : fast_exp2(m_t - M);  // M = -inf -> all 0
  sW[t] = w_t;
  float den = w_t * l_t;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  __syncthreads();  // sW complete; sRed (max) consumed
  if (lane == 0) sRed[warp] = den;
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kSplitsPerWarp; ++k) {
    const int sp = warp + k * kCombineWarps;
    if (sp < ns) acc += ov[k] * sW[sp];
  }
  sAcc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float num = 0.f, dsum = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      num += sAcc[w][lane];
      dsum += sRed[w];
    }
    const float out = dsum > 0.f ? num / dsum : 0.f;
    if (d < D) p.o[((size_t)b * p.Sq * p.Hq + h) * D + d] = __float2bfloat16_rn(out);
    // log sum_j exp(s_j) = ln2 * (M + log2 sum_s 2^(m_s - M) l_s), M in log2 units.
    if (p.lse && lane == 0 && blockIdx.x == 0)
      p.lse[(size_t)b * p.Sq * p.Hq + h] = dsum > 0.f ? 0.6931471805599453f * (M + __log2f(dsum))
                                               : -INFINITY;
  }
}

// Combine for balanced splits (paged batches): one warp per output row
// (b, s, hq), lane l holding columns [l * D/32, (l + 1) * D/32).  The row's
// unit lists its splits' partials (unit map from the split grid's first CTA);
// a row has few of them, so they are loaded four at a time and merged online:
// running max M, and the output and the sum l rescaled by 2^(M_old - M_new)
// when M grows -- O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s as in the
// other combine.  Splits with l_s == 0 get weight 0.  No shared memory and no
// block barrier: a block is 8 independent rows.
constexpr int kRowWarps = 8;
template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) decode_combine_rows_kernel(const DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait_primary();
  constexpr int CPL = D / 32;  // columns per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * kRowWarps + warp;  // in [B, Sq, Hq]
  const size_t rows_per_b = (size_t)p.Sq * p.Hq;
  if (row >= (size_t)p.B * rows_per_b) return;
  const int b = (int)(row / rows_per_b), h = (int)(row - (size_t)b * rows_per_b);
  const int s = h / p.Hq, hq = h - s * p.Hq, hkv = hq / p.G;
  const int r = s * p.G + (hq - hkv * p.G), hb = r / dec::HB;
  const int2 um = p.unit_map[((size_t)b * p.Hkv + hkv) * p.n_hb + hb];
  int ns = um.y;
  if (um.x < 0 || ns < 0 || um.x + ns > p.nsplit) {  // self-check: inside the partials
    if (lane == 0) atomicOr(&g_decode_err, kErrBounds << 4);
    ns = 0;
  }
  const size_t base = (size_t)(um.x < 0 ? 0 : um.x) * dec::HB + (r - hb * dec::HB);
  float M = -INFINITY, den = 0.f, acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int k0 = 0; k0 < ns; k0 += 4) {
    float2 ml[4];
    float ov[4][CPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // every load of the batch before any use
      const size_t slot = base + (size_t)(k0 + u) * dec::HB;
      if (k0 + u < ns) {
        ml[u] = reinterpret_cast<const float2*>(p.part_ml)[slot];
        const float* src = p.part_o + slot * D + lane * CPL;
        if constexpr (CPL == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          ov[u][0] = v.x; ov[u][1] = v.y; ov[u][2] = v.z; ov[u][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          ov[u][0] = v.x; ov[u][1] = v.y;
        }
      } else {
        ml[u] = make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int c = 0; c < CPL; ++c) ov[u][c] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float m_u = ml[u].y > 0.f ? ml[u].x : -INFINITY;
      if (m_u > M) {  // rescale what was merged so far (M = -inf: nothing yet)
        const float f = M == -INFINITY ? 0.f : fast_exp2(M - m_u);
        den *= f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] *= f;
        M = m_u;
      }
      const float w = m_u == -INFINITY ? 0.f : fast_exp2(m_u - M);
      den += w * ml[u].y;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[c] += w * ov[u][c];
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat16* dst = p.o + row * D + lane * CPL;
#pragma unroll
  for (int c = 0; c < CPL; c += 2)
    *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
  if (p.lse && lane == 0)
    p.lse[row] = den > 0.f ? 0.6931471805599453f * (M + __log2f(den)) : -INFINITY;
}

// Degenerate cache (cap == 0): every output is zero, every log-sum-exp -inf.
__global__ void decode_zero_kernel(__nv_bfloat16* o, size_t n, float* lse, size_t nl) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    o[i] = __float2bfloat16_rn(0.f);
  if (lse)
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nl;
         i += (size_t)gridDim.x * blockDim.x)
      lse[i] = -INFINITY;
}

static int decode_nsplit(int B, int Hq, int Hkv, int cap, int Sq, int tt) {
  const int G = Hq / Hkv;
  const int n_hb = (Sq * G + dec::HB - 1) / dec::HB;
  const long units = (long)B * Hkv * n_hb;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  long ns = sms / (units > 0 ? units : 1);
  const long max_tiles = ((long)cap + tt - 1) / tt;
  if (ns > max_tiles) ns = max_tiles;
  if (ns > kMaxSplits) ns = kMaxSplits;  // the combine's one-pass limit
  if (ns < 1) ns = 1;
  return (int)ns;
}

// Balanced splits for a paged batch: only when its units fit in fewer CTAs
// than the SMs (the lengths can then differ per sequence and the grid can
// still cover every SM); the CTA count is the SM count.
static bool decode_balanced(int B, int Hq, int Hkv, int Sq, bool paged) {
  if (!paged) return false;
  const int G = Hq / Hkv;
  const int n_hb = (Sq * G + dec::HB - 1) / dec::HB;
  const long units = (long)B * Hkv * n_hb;
  const int sms = sm_count() > 0 ? sm_count() : 148;
  return units < sms && sms <= kMaxSplits && B <= dec::THREADS;
}

size_t decode_scratch_floats(int B, int Hq, int Hkv, int cap, int D, int Sq, bool paged) {
  if (decode_balanced(B, Hq, Hkv, Sq, paged)) {
    const size_t sms = (size_t)(sm_count() > 0 ? sm_count() : 148);
    const size_t units = (size_t)B * Hkv * ((Sq * (Hq / Hkv) + dec::HB - 1) / dec::HB);
    return sms * dec::HB * ((size_t)D + 2) + 2 * units + 2;  // + the unit map (int2, aligned)
  }
  // Paged caches may take 32-token tiles: the most splits either tile allows.
  const size_t ns = (size_t)decode_nsplit(B, Hq, Hkv, cap, Sq, paged ? dec::TT : 64);
  return (size_t)B * Sq * Hq * ns * ((size_t)D + 2);
}

template <int D>
static int launch_decode_t(const void* q, const void* kc, const void* vc, const DecodeLayout& ly,
                           void* o, float* lse, int B, int Hq, int Hkv, float scale,
                           float* scratch, cudaStream_t stream) {
  using CC = dec::Cfg<D, false, 64>;  // contiguous caches
  using CP = dec::Cfg<D, true, 32>;   // paged caches, pages of 32-token multiples
  using CP64 = dec::Cfg<D, true, 64>; // paged caches, pages of 64-token multiples
  const bool paged = ly.page_table != nullptr;
  const int cap = paged ? ly.max_pages * ly.page_size : ly.cap;
  const int Sq = paged ? ly.Sq : 1;
  const bool bal = decode_balanced(B, Hq, Hkv, Sq, paged);
  // 64-token tiles for pages of 64-token multiples (in balanced mode the
  // split planner takes one thread per sequence, so also B <= its threads).
  const bool big = paged && ly.page_size % 64 == 0 && (!bal || B <= CP64::THREADS);
  CUtensorMap tk, tv;
  if (paged) {
    const int tt = big ? CP64::TT : CP::TT;
    if (encode_tmap_rows(&tk, kc, D, Hkv, ly.page_size, ly.num_pages, tt))
      return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tv, vc, D, Hkv, ly.page_size, ly.num_pages, tt))
      return cudaErrorInvalidValue;
  } else {
    if (encode_tmap_rows(&tk, kc, D, Hkv, cap, B, CC::TT)) return cudaErrorInvalidValue;
    if (encode_tmap_rows(&tv, vc, D, Hkv, cap, B, CC::TT)) return cudaErrorInvalidValue;
  }
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    const void* kernels[6] = {(const void*)decode_split_kernel<D, false, 1, 64>,
                              (const void*)decode_split_kernel<D, false, 2, 64>,
                              (const void*)decode_split_kernel<D, true, 1, 32>,
                              (const void*)decode_split_kernel<D, true, 2, 32>,
                              (const void*)decode_split_kernel<D, true, 1, 64>,
                              (const void*)decode_split_kernel<D, true, 2, 64>};
    const int smem[6] = {CC::SMEM_TOTAL, CC::SMEM_TOTAL, CP::SMEM_TOTAL, CP::SMEM_TOTAL,
                         CP64::SMEM_TOTAL, CP64::SMEM_TOTAL};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 6; ++i) {
      e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
      if (e != cudaSuccess) return e;
    }
    // Same shared-memory carveout as the split kernel, so that combine CTAs
    // can become resident beside split CTAs and wait there.
    for (const void* k : {(const void*)decode_combine_kernel<D>,
                          (const void*)decode_combine_rows_kernel<D>}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = 1;
  }
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.valid_len = ly.valid_len;
  p.len_stride = ly.len_stride;
  p.page_table = ly.page_table;
  p.page_size = ly.page_size;
  p.max_pages = ly.max_pages;
  p.num_pages = ly.num_pages;
  const int ns = bal ? (sm_count() > 0 ? sm_count() : 148)
                     : decode_nsplit(B, Hq, Hkv, cap, Sq, paged && !big ? CP::TT : 64);
  p.part_o = scratch;
  p.part_ml = scratch + (bal ? (size_t)ns * dec::HB * D : (size_t)B * Sq * Hq * ns * D);
  p.balanced = bal ? 1 : 0;
  {  // the unit map follows the partials, 8-byte aligned
    const size_t off = (size_t)ns * dec::HB * (D + 2);
    p.unit_map = bal ? reinterpret_cast<int2*>(scratch + off + (off & 1)) : nullptr;
  }
  p.Sq = Sq;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.cap = cap;
  p.G = Hq / Hkv;
  p.nsplit = ns;
  p.n_hb = (Sq * p.G + dec::HB - 1) / dec::HB;
  p.c = scale * 1.4426950408889634f;

  // Both kernels are programmatic dependents of the grid before them: each
  // runs only its prologue before griddepcontrol.wait.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t sc = {};
  sc.gridDim = bal ? dim3(ns, 1, 1) : dim3(ns, Hkv * p.n_hb, B);
  sc.blockDim = dim3(!paged ? CC::THREADS : (big ? CP64::THREADS : CP::THREADS), 1, 1);
  sc.dynamicSmemBytes = !paged ? CC::SMEM_TOTAL : (big ? CP64::SMEM_TOTAL : CP::SMEM_TOTAL);
  sc.stream = stream;
  sc.attrs = attr;
  sc.numAttrs = 1;
  // One block of 8 query rows per CTA when the kv head has at most 8 rows.
  const bool nb1 = Sq * p.G <= 8;
  cudaError_t e;
  if (paged && big)
    e = nb1 ? cudaLaunchKernelEx(&sc, decode_split_kernel<D, true, 1, 64>, tk, tv, p)
            : cudaLaunchKernelEx(&sc, decode_split_kernel<D, true, 2, 64>, tk, tv, p);
  else if (paged)
    e = nb1 ? cudaLaunchKernelEx(&sc, decode_split_kernel<D, true, 1, 32>, tk, tv, p)
            : cudaLaunchKernelEx(&sc, decode_split_kernel<D, true, 2, 32>, tk, tv, p);
  else
    e = nb1 ? cudaLaunchKernelEx(&sc, decode_split_kernel<D, false, 1, 64>, tk, tv, p)
            : cudaLaunchKernelEx(&sc, decode_split_kernel<D, false, 2, 64>, tk, tv, p);
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  const size_t n_rows = (size_t)B * Sq * Hq;
  cfg.gridDim = bal ? dim3((unsigned)((n_rows + kRowWarps - 1) / kRowWarps), 1, 1)
                    : dim3((D + 31) / 32, Sq * Hq, B);
  cfg.blockDim = dim3(bal ? kRowWarps * 32 : kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = bal ? cudaLaunchKernelEx(&cfg, decode_combine_rows_kernel<D>, p)
          : cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p);
  return e;
}

int launch_decode_layout(const void* q, const void* kc, const void* vc, const DecodeLayout& ly,
                         void* o, float* lse, int B, int Hq, int Hkv, int D, float scale,
                         float* scratch, size_t scratch_floats, cudaStream_t stream) {
  if (B == 0 || Hq == 0) return cudaSuccess;
  const int cap = ly.page_table ? ly.max_pages * ly.page_size : ly.cap;
  if (cap == 0) {
    const size_t rows = (size_t)B * (ly.page_table ? ly.Sq : 1) * Hq, n = rows * D;
    decode_zero_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0,
                         stream>>>(static_cast<__nv_bfloat16*>(o), n, lse, rows);
    return cudaGetLastError();
  }
  const int Sq = ly.page_table ? ly.Sq : 1;
  if (scratch_floats < decode_scratch_floats(B, Hq, Hkv, cap, D, Sq, ly.page_table != nullptr))
    return cudaErrorInvalidValue;
  if (D == 64)
    return launch_decode_t<64>(q, kc, vc, ly, o, lse, B, Hq, Hkv, scale, scratch, stream);
  return launch_decode_t<128>(q, kc, vc, ly, o, lse, B, Hq, Hkv, scale, scratch, stream);
}

int launch_decode(const void* q, const void* kc, const void* vc, const int32_t* valid_len,
                  void* o, float* lse, int B, int Hq, int Hkv, int cap, int D, float scale,
                  float* scratch, size_t scratch_floats, cudaStream_t stream) {
  DecodeLayout ly;
  ly.valid_len = valid_len;
  ly.len_stride = 0;
  ly.cap = cap;
  return launch_decode_layout(q, kc, vc, ly, o, lse, B, Hq, Hkv, D, scale, scratch,
                              scratch_floats, stream);
}

int set_decode_wait_limit(unsigned long long ns) { return set_wait_limit_this_unit(ns); }

int read_decode_error(unsigned int* out, int reset) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (reset && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_decode_err, &z, sizeof(z));
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace fa
