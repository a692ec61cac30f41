// fa_api.cu -- the C ABI (include/fa.h): argument validation, tensor-map
// encoding, stream-ordered scratch for the decode partials, status mapping.
// Every step of the attention itself runs in the kernels of fa_prefill.cu and
// fa_decode.cu; this file only validates, marshals and enqueues.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int encode_tmap_rows(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint64_t d3, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return 1;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  const cuuint32_t box[4] = {64, 1, box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 1;
}

int sm_count() {
  static int cache[64];
  static std::once_flag once;
  std::call_once(once, [] {
    for (int i = 0; i < 64; ++i) cache[i] = 0;
  });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace fa

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Raw CUDA error and call site of the most recent FA_ERR_CUDA in this thread.
static thread_local int t_last_cuda_error = 0;
static thread_local const char* t_last_site = "";

int fa::record_cuda_status(int e, const char* site) {
  if (e == 0) return FA_OK;
  t_last_cuda_error = e;
  t_last_site = site;
  cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return FA_ERR_CUDA;
}

static int cuda_status(int e, const char* site) { return fa::record_cuda_status(e, site); }

static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static int prefill_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                        bool want_lse, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                        float scale, int causal, int dtype, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0 || Sq == 0) return FA_OK;  // empty problem: nothing to write
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!q || !o || !aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (want_lse && (!lse || !aligned4(lse))) return FA_ERR_INVALID_ARG;
  if (Sk > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return FA_ERR_INVALID_ARG;
  // Work items (B * Hq * ceil(Sq/256)) and element counts must fit the kernel's
  // 32-bit item index and the tensor maps' 40-bit byte strides.
  const int64_t items = (int64_t)B * Hq * ((Sq + 255) / 256);
  if (items > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)Sq * Hq * D * 2 >= (1ll << 40) || (int64_t)Sk * Hkv * D * 2 >= (1ll << 40))
    return FA_ERR_INVALID_ARG;
  return cuda_status(fa::launch_prefill(q, k, v, o, want_lse ? lse : nullptr, B, Hq, Hkv, Sq, Sk,
                                        D, scale, causal, dtype == FA_BF16, stream),
                     "prefill launch");
}

extern "C" int fa_prefill_fwd(const void* q, const void* k, const void* v, void* o, int B,
                              int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                              int dtype, cudaStream_t stream) {
  return prefill_impl(q, k, v, o, nullptr, false, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype,
                      stream);
}

extern "C" int fa_prefill_fwd_lse(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                                  float scale, int causal, int dtype, cudaStream_t stream) {
  return prefill_impl(q, k, v, o, lse, true, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype,
                      stream);
}

extern "C" int fa_prefill_varlen_fwd(const void* q, const void* k, const void* v, void* o,
                                     float* lse, const int32_t* cu_seqlens_q,
                                     const int32_t* cu_seqlens_k, int B, int Hq, int Hkv,
                                     int total_q, int total_k, int max_seqlen_q, int D,
                                     float scale, int causal, int dtype, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0)
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0 || total_q == 0) return FA_OK;  // no query row: nothing to write
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (max_seqlen_q > total_q) return FA_ERR_INVALID_ARG;
  if (!q || !o || !aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && !aligned4(lse)) return FA_ERR_INVALID_ARG;
  if (!cu_seqlens_q || !cu_seqlens_k || !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k))
    return FA_ERR_INVALID_ARG;
  if (total_k > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return FA_ERR_INVALID_ARG;
  const int64_t items = (int64_t)B * Hq * ((max_seqlen_q + 255) / 256);
  if (items > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)total_q * Hq * D * 2 >= (1ll << 40) || (int64_t)total_k * Hkv * D * 2 >= (1ll << 40))
    return FA_ERR_INVALID_ARG;
  return cuda_status(fa::launch_prefill_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq,
                                               Hkv, total_q, total_k, max_seqlen_q, D, scale,
                                               causal, dtype == FA_BF16, stream),
                     "prefill varlen launch");
}

extern "C" int fa_backward(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale,
                           int causal, int dtype, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (Sq > 0 && (!q || !o || !dout || !dq || !lse || !aligned16(q) || !aligned16(o) ||
                 !aligned16(dout) || !aligned16(dq) || !aligned4(lse)))
    return FA_ERR_INVALID_ARG;
  if (Sk > 0 && (!k || !v || !dk || !dv || !aligned16(k) || !aligned16(v) || !aligned16(dk) ||
                 !aligned16(dv)))
    return FA_ERR_INVALID_ARG;
  const int64_t items_q = (int64_t)B * Hq * ((Sq + 127) / 128);
  const int64_t items_k = (int64_t)B * Hkv * ((Sk + 127) / 128);
  if (items_q > INT32_MAX || items_k > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)Sq * Hq * D * 2 >= (1ll << 40) || (int64_t)Sk * Hkv * D * 2 >= (1ll << 40))
    return FA_ERR_INVALID_ARG;
  // No key: dQ = 0 (and no dK, dV rows).  No query row: dK = dV = 0.
  if (Sq == 0 || Sk == 0) {
    cudaError_t e = cudaSuccess;
    if (Sk == 0 && Sq > 0) e = cudaMemsetAsync(dq, 0, (size_t)B * Sq * Hq * D * 2, stream);
    if (e == cudaSuccess && Sq == 0 && Sk > 0) {
      e = cudaMemsetAsync(dk, 0, (size_t)B * Sk * Hkv * D * 2, stream);
      if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, (size_t)B * Sk * Hkv * D * 2, stream);
    }
    return cuda_status(e, "backward zero-fill");
  }
  void* delta = nullptr;
  // Delta [B, Hq, Sq], then the two work counters of the dq and dkdv kernels.
  cudaError_t e = cudaMallocAsync(&delta, ((size_t)B * Hq * Sq + 2) * sizeof(float), stream);
  if (e != cudaSuccess) return cuda_status(e, "backward cudaMallocAsync");
  int r = fa::launch_backward(q, k, v, o, dout, lse, dq, dk, dv, static_cast<float*>(delta), B,
                              Hq, Hkv, Sq, Sk, D, scale, causal, dtype == FA_BF16, stream);
  cudaError_t ef = cudaFreeAsync(delta, stream);
  if (r != 0) return cuda_status(r, "backward launch");
  return cuda_status(ef, "backward cudaFreeAsync");
}

static int decode_impl(const void* q, const void* kcache, const void* vcache,
                       const int32_t* valid_len_dev, void* o, float* lse, bool want_lse, int B,
                       int Hq, int Hkv, int cap, int D, float scale, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || cap < 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535 || (int64_t)Hkv * ((Hq / Hkv + 15) / 16) > 65535)
    return FA_ERR_INVALID_ARG;
  if (!q || !o || !aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (want_lse && (!lse || !aligned4(lse))) return FA_ERR_INVALID_ARG;
  if (!want_lse) lse = nullptr;
  if (cap > 0 && (!kcache || !vcache || !valid_len_dev || !aligned16(kcache) ||
                  !aligned16(vcache) || (reinterpret_cast<uintptr_t>(valid_len_dev) & 3u)))
    return FA_ERR_INVALID_ARG;
  if ((int64_t)cap * Hkv * D * 2 >= (1ll << 40)) return FA_ERR_INVALID_ARG;
  if (cap == 0)
    return cuda_status(fa::launch_decode(q, kcache, vcache, valid_len_dev, o, lse, B, Hq, Hkv, 0,
                                         D, scale, nullptr, 0, stream),
                       "decode zero-fill launch");
  const size_t nf = fa::decode_scratch_floats(B, Hq, Hkv, cap, D);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, nf * sizeof(float), stream);
  if (e != cudaSuccess) return cuda_status(e, "decode cudaMallocAsync");
  int r = fa::launch_decode(q, kcache, vcache, valid_len_dev, o, lse, B, Hq, Hkv, cap, D, scale,
                            static_cast<float*>(scratch), nf, stream);
  cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (r != 0) return cuda_status(r, "decode launch");
  return cuda_status(ef, "decode cudaFreeAsync");
}

extern "C" int fa_decode_paged_fwd(const void* q, const void* kpages, const void* vpages,
                                   const int32_t* page_table, const int32_t* seqlens, void* o,
                                   float* lse, int B, int Sq, int Hq, int Hkv, int num_pages,
                                   int page_size, int max_pages, int D, float scale,
                                   cudaStream_t stream) {
  if (B < 0 || Sq < 0 || Hq < 0 || Hkv < 0 || num_pages < 0 || max_pages < 0)
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (page_size < 32 || page_size % 32 != 0) return FA_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0 || Hq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (B > 65535 || (int64_t)Sq * Hq > 65535 ||
      (int64_t)Hkv * (((int64_t)Sq * (Hq / Hkv) + 15) / 16) > 65535)
    return FA_ERR_INVALID_ARG;
  if ((int64_t)max_pages * page_size > INT32_MAX) return FA_ERR_INVALID_ARG;
  if (!q || !o || !aligned16(q) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && !aligned4(lse)) return FA_ERR_INVALID_ARG;
  if (max_pages > 0 &&
      (num_pages < 1 || !kpages || !vpages || !aligned16(kpages) || !aligned16(vpages) ||
       !page_table || !seqlens || !aligned4(page_table) || !aligned4(seqlens)))
    return FA_ERR_INVALID_ARG;
  if ((int64_t)num_pages * page_size * Hkv * D * 2 >= (1ll << 40)) return FA_ERR_INVALID_ARG;
  fa::DecodeLayout ly;
  ly.valid_len = seqlens;
  ly.len_stride = 1;
  ly.page_table = page_table;
  ly.page_size = page_size;
  ly.max_pages = max_pages;
  ly.num_pages = num_pages;
  ly.Sq = Sq;
  const int cap = max_pages * page_size;
  if (cap == 0)
    return cuda_status(fa::launch_decode_layout(q, kpages, vpages, ly, o, lse, B, Hq, Hkv, D,
                                                scale, nullptr, 0, stream),
                       "paged decode zero-fill launch");
  const size_t nf = fa::decode_scratch_floats(B, Hq, Hkv, cap, D, Sq, true);
  void* scratch = nullptr;
  cudaError_t e = cudaMallocAsync(&scratch, nf * sizeof(float), stream);
  if (e != cudaSuccess) return cuda_status(e, "paged decode cudaMallocAsync");
  int r = fa::launch_decode_layout(q, kpages, vpages, ly, o, lse, B, Hq, Hkv, D, scale,
                                   static_cast<float*>(scratch), nf, stream);
  cudaError_t ef = cudaFreeAsync(scratch, stream);
  if (r != 0) return cuda_status(r, "paged decode launch");
  return cuda_status(ef, "paged decode cudaFreeAsync");
}

extern "C" int fa_decode_fwd(const void* q, const void* kcache, const void* vcache,
                             const int32_t* valid_len_dev, void* o, int B, int Hq, int Hkv,
                             int cap, int D, float scale, cudaStream_t stream) {
  return decode_impl(q, kcache, vcache, valid_len_dev, o, nullptr, false, B, Hq, Hkv, cap, D,
                     scale, stream);
}

extern "C" int fa_decode_fwd_lse(const void* q, const void* kcache, const void* vcache,
                                 const int32_t* valid_len_dev, void* o, float* lse, int B,
                                 int Hq, int Hkv, int cap, int D, float scale,
                                 cudaStream_t stream) {
  return decode_impl(q, kcache, vcache, valid_len_dev, o, lse, true, B, Hq, Hkv, cap, D, scale,
                     stream);
}

extern "C" const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported configuration";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device pipeline wait hit its time limit";
    case FA_ERR_TOO_LARGE:
      return "FA_ERR_TOO_LARGE: request needs more scratch than "
             "fa_decode_fwd_noalloc's fixed array";
    case FA_ERR_BOUNDS:
      return "FA_ERR_BOUNDS: a device-side bounds check skipped an access "
             "(offsets or page ids out of range)";
    default: return "unknown status";
  }
}

extern "C" int fa_device_error(int reset, unsigned int* detail) {
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  unsigned int a = 0, b = 0, c = 0;
  if (fa::read_prefill_error(&a, reset) != 0) return FA_ERR_CUDA;
  if (fa::read_decode_error(&b, reset) != 0) return FA_ERR_CUDA;
  if (fa::read_backward_error(&c, reset) != 0) return FA_ERR_CUDA;
  a |= c;  // the backward kernels report in the prefill half
  if (detail) *detail = (a & 0xFFFFu) | (b << 16);
  if ((a | b) & 1u) return FA_ERR_TIMEOUT;
  return (a | b) ? FA_ERR_BOUNDS : FA_OK;
}

extern "C" int fa_num_sms(void) { return fa::sm_count(); }

extern "C" int fa_prefill_rescale_count(int reset, unsigned long long* count) {
  if (!count) return FA_ERR_INVALID_ARG;
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "rescale count synchronize");
  return cuda_status(fa::read_prefill_rescales(count, reset), "rescale count read");
}

extern "C" int fa_set_wait_limit_ns(unsigned long long ns) {
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "wait limit synchronize");
  int r = fa::set_prefill_wait_limit(ns);
  if (r == 0) r = fa::set_decode_wait_limit(ns);
  if (r == 0) r = fa::set_backward_wait_limit(ns);
  return cuda_status(r, "wait limit set");
}

extern "C" int fa_last_cuda_error(const char** site) {
  if (site) *site = t_last_site;
  return t_last_cuda_error;
}

extern "C" int fa_prefill_work_item(int w, int B, int Hq, int Hkv, int Sq, int Sk, int causal,
                                    int* b, int* hq, int* qblock) {
  (void)Sk;
  (void)causal;
  if (B < 0 || Hq < 0 || Hkv <= 0 || Sq < 0 || (Hq % Hkv) != 0) return -1;
  const int64_t n_qb = (Sq + 255) / 256;
  const int64_t n = (int64_t)B * Hq * n_qb;
  if (n > INT32_MAX) return -1;
  if (w >= 0 && w < n) {
    int bb, hh, qq;
    fa::prefill_item_host(w, B, Hq, Hkv, (int)n_qb, &bb, &hh, &qq);
    if (b) *b = bb;
    if (hq) *hq = hh;
    if (qblock) *qblock = qq;
  }
  return (int)n;
}
