// fa_internal.h -- host-side declarations shared by the C-ABI layer and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Tensor map over a contiguous [d3][d2][d1][d0] tensor of 16-bit elements,
// 128-byte swizzle, zero fill outside the tensor, box (64, 1, box_rows, 1).
// Returns 0 on success.
int encode_tmap_rows(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint64_t d3, uint32_t box_rows);

// SM count of the current device (cached per device), or -1.
int sm_count();

// Enqueue the prefill kernel; lse ([B, Hq, Sq] fp32) may be null.  Returns a
// cudaError_t (0 = success).
int launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal, bool bf16,
                   cudaStream_t stream);

// Enqueue the prefill kernel over packed sequences: q/o [total_q, Hq, D],
// k/v [total_k, Hkv, D], cu_q / cu_k device prefix sums [B + 1], lse
// ([Hq, total_q] fp32) may be null.  Returns a cudaError_t.
int launch_prefill_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* cu_q, const int32_t* cu_k, int B, int Hq, int Hkv,
                          int total_q, int total_k, int max_seqlen_q, int D, float scale,
                          int causal, bool bf16, cudaStream_t stream);

// Enqueue split + combine decode kernels with the given fp32 scratch
// (partials); lse ([B, Hq] fp32) may be null.  scratch_floats is the scratch
// size in floats.  Returns a cudaError_t.
int launch_decode(const void* q, const void* kc, const void* vc, const int32_t* valid_len,
                  void* o, float* lse, int B, int Hq, int Hkv, int cap, int D, float scale,
                  float* scratch, size_t scratch_floats, cudaStream_t stream);

// Where the decode's K/V live and how long each sequence is.
//   contiguous caches [B, cap, Hkv, D]: page_table == nullptr, cap = capacity;
//   paged caches [num_pages, page_size, Hkv, D] with page_table [B, max_pages]
//   (device; page_size a multiple of 32): capacity max_pages * page_size.
//   valid_len: device int32, L of batch entry b at valid_len[b * len_stride].
struct DecodeLayout {
  const int32_t* valid_len = nullptr;
  int len_stride = 0;
  int cap = 0;
  const int32_t* page_table = nullptr;
  int page_size = 0, max_pages = 0, num_pages = 0;
  int Sq = 1;  // new query tokens per sequence (paged layout only)
};

int launch_decode_layout(const void* q, const void* kc, const void* vc, const DecodeLayout& ly,
                         void* o, float* lse, int B, int Hq, int Hkv, int D, float scale,
                         float* scratch, size_t scratch_floats, cudaStream_t stream);

// Scratch floats the decode needs for these sizes (Sq new tokens per sequence).
size_t decode_scratch_floats(int B, int Hq, int Hkv, int cap, int D, int Sq = 1,
                             bool paged = false);

// Enqueue the backward pass: Delta into `delta` ([B, Hq, Sq] fp32 scratch, then
// two uint32 work counters),
// then dq [B, Sq, Hq, D] and dk, dv [B, Sk, Hkv, D] from q, k, v, the forward
// output o, dout and the forward's lse ([B, Hq, Sq]).  Sq, Sk > 0.
int launch_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, float* delta, int B, int Hq,
                    int Hkv, int Sq, int Sk, int D, float scale, int causal, bool bf16,
                    cudaStream_t stream);
int read_backward_error(unsigned int* out, int reset);

// Device error words of the kernel translation units (read + optionally clear).
int read_prefill_error(unsigned int* out, int reset);
int read_decode_error(unsigned int* out, int reset);

// Rows whose prefill lazy rescale fired since the last reset (read + optionally
// clear).  Returns a cudaError_t.
int read_prefill_rescales(unsigned long long* out, int reset);

// Time limit of the pipeline waits of each kernel translation unit on the
// current device (0 = the 2 s default).  Synchronous; return a cudaError_t.
int set_prefill_wait_limit(unsigned long long ns);
int set_decode_wait_limit(unsigned long long ns);
int set_backward_wait_limit(unsigned long long ns);

// Status of a CUDA call for the C ABI: FA_OK for 0, else FA_ERR_CUDA after
// recording the raw error and the failing call (a static string) for
// fa_last_cuda_error() in the calling thread.
int record_cuda_status(int cuda_error, const char* site);

// Work-item decode of the persistent prefill scheduler (host copy).
void prefill_item_host(int w, int B, int Hq, int Hkv, int n_qb, int* b, int* hq, int* qb);

}  // namespace fa
