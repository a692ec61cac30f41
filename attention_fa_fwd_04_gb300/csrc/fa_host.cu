// fa_host.cu -- prefill from host memory to host memory (fa_prefill_fwd_host):
// the uploads of Q, K, V and the download of O overlapped with the prefill
// kernels, all behind the C ABI.
//
// Why pieces: the query rows of one sequence split into independent pieces.
// Rows [s0, s1) need only the keys they can see, and that piece is again an
// ordinary prefill -- with causal masking a bottom-right aligned one over the
// key prefix [0, s1 + Sk - Sq) -- so it runs through the prefill kernel
// unchanged ("Dense flash-attention prefill (gfx950 / MI355X)", opening
// paragraph: causal prefill with Sq != Sk handled by the same kernel).  K and
// V go up first, then Q piece by piece, heaviest piece first; each piece's
// kernel starts as soon as its rows have landed, and its O goes back on a
// second copy stream.  Uploads, kernels and downloads of different pieces run
// at the same time.
//
// This file only orders copies and launches; every attention step runs in the
// prefill kernel.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kUnit = 256;  // rows of the prefill kernel's work unit

struct Piece {
  int b, s0, s1, sk;
};

// Row pieces of one sequence: at most n_pieces, boundaries on multiples of
// kUnit rows (except the end); sk = the key prefix the piece's rows can see.
void row_pieces(int Sq, int Sk, int causal, int n_pieces, std::vector<Piece>* out, int b) {
  if (Sq <= 0) return;
  const int64_t n_units = (Sq + kUnit - 1) / kUnit;
  const int64_t n = std::max<int64_t>(1, std::min<int64_t>(n_pieces, n_units));
  for (int64_t c = 0; c < n; ++c) {
    const int s0 = (int)std::min<int64_t>(Sq, (c * n_units / n) * kUnit);
    const int s1 = (int)std::min<int64_t>(Sq, ((c + 1) * n_units / n) * kUnit);
    if (s1 <= s0) continue;
    int sk = Sk;
    if (causal) sk = (int)std::min<int64_t>(Sk, std::max<int64_t>(0, (int64_t)s1 + Sk - Sq));
    out->push_back({b, s0, s1, sk});
  }
}

// The batch's pieces, heaviest (rows x visible keys) first: the kernels then
// have long pieces to work on while short ones upload, and the last download
// is a short one.
std::vector<Piece> plan(int B, int Sq, int Sk, int causal, int n_pieces) {
  std::vector<Piece> ps;
  for (int b = 0; b < B; ++b) row_pieces(Sq, Sk, causal, n_pieces, &ps, b);
  std::stable_sort(ps.begin(), ps.end(), [](const Piece& x, const Piece& y) {
    return (int64_t)(x.s1 - x.s0) * x.sk > (int64_t)(y.s1 - y.s0) * y.sk;
  });
  return ps;
}

// Per device: the copy and compute streams and the events that order them,
// created on first use and kept for the life of the process.  Calls on one
// device enqueue under a lock (they share the streams and events).  The
// pieces' kernels alternate between two compute streams: a piece is a few
// waves of work items, and the next piece's CTAs then take the SMs that the
// current piece's last wave leaves idle.
constexpr int kCompStreams = 2;
struct Pipe {
  cudaStream_t up = nullptr, down = nullptr;
  cudaStream_t comp[kCompStreams] = {nullptr, nullptr};
  cudaEvent_t start = nullptr, kv = nullptr, done = nullptr;
  std::vector<cudaEvent_t> ev_q, ev_o;
  std::mutex mu;
};

int make_event(cudaEvent_t* e) { return (int)cudaEventCreateWithFlags(e, cudaEventDisableTiming); }

int pipe_for_device(Pipe** out) {
  static std::mutex mu;
  static Pipe* pipes[kMaxDevices] = {nullptr};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!pipes[dev]) {
    Pipe* p = new Pipe();
    int r = (int)cudaStreamCreateWithFlags(&p->up, cudaStreamNonBlocking);
    for (int c = 0; c < kCompStreams && !r; ++c)
      r = (int)cudaStreamCreateWithFlags(&p->comp[c], cudaStreamNonBlocking);
    if (!r) r = (int)cudaStreamCreateWithFlags(&p->down, cudaStreamNonBlocking);
    if (!r) r = make_event(&p->start);
    if (!r) r = make_event(&p->kv);
    if (!r) r = make_event(&p->done);
    if (r) {  // the call fails: release what was created
      for (cudaStream_t s : {p->up, p->comp[0], p->comp[1], p->down})
        if (s) cudaStreamDestroy(s);
      for (cudaEvent_t ev : {p->start, p->kv, p->done})
        if (ev) cudaEventDestroy(ev);
      delete p;
      return r;
    }
    pipes[dev] = p;
  }
  *out = pipes[dev];
  return 0;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" int fa_prefill_host_pieces(int B, int Sq, int Sk, int causal, int n_pieces,
                                      int* b, int* s0, int* s1, int* sk, int max_pieces) {
  if (B < 0 || Sq < 0 || Sk < 0 || n_pieces < 1 || max_pieces < 0) return -1;
  const std::vector<Piece> ps = plan(B, Sq, Sk, causal, n_pieces);
  const int n = (int)ps.size();
  for (int i = 0; i < n && i < max_pieces; ++i) {
    if (b) b[i] = ps[i].b;
    if (s0) s0[i] = ps[i].s0;
    if (s1) s1[i] = ps[i].s1;
    if (sk) sk[i] = ps[i].sk;
  }
  return n;
}

extern "C" int fa_prefill_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                                   void* o_host, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                                   float scale, int causal, int dtype, int n_pieces,
                                   cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_INVALID_ARG;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (n_pieces < 1) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0 || Sq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!q_host || !o_host || (Sk > 0 && (!k_host || !v_host))) return FA_ERR_INVALID_ARG;
  const int64_t items = (int64_t)B * Hq * ((Sq + 255) / 256);
  if (items > INT32_MAX) return FA_ERR_INVALID_ARG;
  if ((int64_t)Sq * Hq * D * 2 >= (1ll << 40) || (int64_t)Sk * Hkv * D * 2 >= (1ll << 40))
    return FA_ERR_INVALID_ARG;

  const size_t row_q = (size_t)Hq * D * 2, row_k = (size_t)Hkv * D * 2;
  const size_t bq = (size_t)B * Sq * row_q, bk = (size_t)B * Sk * row_k;
  const std::vector<Piece> ps = plan(B, Sq, Sk, causal, n_pieces);
  const bool bf16 = dtype == FA_BF16;

  Pipe* pp = nullptr;
  int r = pipe_for_device(&pp);
  if (r) return fa::record_cuda_status(r, "host prefill stream set-up");
  std::lock_guard<std::mutex> lock(pp->mu);
  while (pp->ev_q.size() < ps.size()) {
    cudaEvent_t a = nullptr, c = nullptr;
    r = make_event(&a);
    if (!r) r = make_event(&c);
    if (r) {
      if (a) cudaEventDestroy(a);
      return fa::record_cuda_status(r, "host prefill event set-up");
    }
    pp->ev_q.push_back(a);
    pp->ev_o.push_back(c);
  }

  // Device copies of q, o, k, v: stream-ordered on the caller's stream, freed
  // on it after the last download.
  void* buf = nullptr;
  const size_t off_o = round256(bq), off_k = off_o + round256(bq), off_v = off_k + round256(bk);
  cudaError_t e = cudaMallocAsync(&buf, off_v + round256(bk), stream);
  if (e != cudaSuccess) return fa::record_cuda_status(e, "host prefill cudaMallocAsync");
  uint8_t* dq = static_cast<uint8_t*>(buf);
  uint8_t* dout = dq + off_o;
  uint8_t* dk = dq + off_k;
  uint8_t* dv = dq + off_v;
  const char* site = "host prefill enqueue";
  auto H2D = cudaMemcpyHostToDevice;
  // Fork: the three pipeline streams start after the work already on the
  // caller's stream (including the allocation).
  e = cudaEventRecord(pp->start, stream);
  if (!e) e = cudaStreamWaitEvent(pp->up, pp->start, 0);
  for (int c = 0; c < kCompStreams && !e; ++c) e = cudaStreamWaitEvent(pp->comp[c], pp->start, 0);
  if (!e) e = cudaStreamWaitEvent(pp->down, pp->start, 0);
  // K and V first, then Q piece by piece.
  if (!e && bk) e = cudaMemcpyAsync(dk, k_host, bk, H2D, pp->up);
  if (!e && bk) e = cudaMemcpyAsync(dv, v_host, bk, H2D, pp->up);
  if (!e) e = cudaEventRecord(pp->kv, pp->up);
  for (size_t i = 0; i < ps.size() && !e; ++i) {
    const size_t off = ((size_t)ps[i].b * Sq + ps[i].s0) * row_q;
    e = cudaMemcpyAsync(dq + off, static_cast<const uint8_t*>(q_host) + off,
                        (size_t)(ps[i].s1 - ps[i].s0) * row_q, H2D, pp->up);
    if (!e) e = cudaEventRecord(pp->ev_q[i], pp->up);
  }
  // One prefill per piece, each as soon as its Q rows have landed, on the
  // compute streams in turn.
  for (int c = 0; c < kCompStreams && !e; ++c) e = cudaStreamWaitEvent(pp->comp[c], pp->kv, 0);
  for (size_t i = 0; i < ps.size() && !e; ++i) {
    const Piece& c = ps[i];
    cudaStream_t cs = pp->comp[i % kCompStreams];
    const size_t qo = ((size_t)c.b * Sq + c.s0) * row_q, kv = (size_t)c.b * Sk * row_k;
    e = cudaStreamWaitEvent(cs, pp->ev_q[i], 0);
    if (!e) {
      const int lr = fa::launch_prefill(dq + qo, dk + kv, dv + kv, dout + qo, nullptr, 1, Hq, Hkv,
                                        c.s1 - c.s0, c.sk, D, scale, causal, bf16, cs);
      if (lr) {
        e = (cudaError_t)lr;
        site = "host prefill launch";
      }
    }
    if (!e) e = cudaEventRecord(pp->ev_o[i], cs);
  }
  // O back piece by piece; the caller's stream joins the last download.
  for (size_t i = 0; i < ps.size() && !e; ++i) {
    const size_t off = ((size_t)ps[i].b * Sq + ps[i].s0) * row_q;
    e = cudaStreamWaitEvent(pp->down, pp->ev_o[i], 0);
    if (!e)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(o_host) + off, dout + off,
                          (size_t)(ps[i].s1 - ps[i].s0) * row_q, cudaMemcpyDeviceToHost, pp->down);
  }
  // The down stream has waited for every piece's kernel (and the compute
  // streams for every upload), so its last event orders all of the call's
  // work.
  if (!e) e = cudaEventRecord(pp->done, pp->down);
  if (!e) e = cudaStreamWaitEvent(stream, pp->done, 0);
  if (e) {
    // Something failed part-way: let what was enqueued finish before the
    // buffer is released (the host waits here; failures only).
    cudaStreamSynchronize(pp->up);
    for (int c = 0; c < kCompStreams; ++c) cudaStreamSynchronize(pp->comp[c]);
    cudaStreamSynchronize(pp->down);
    const int st = fa::record_cuda_status((int)e, site);
    cudaFreeAsync(buf, stream);
    return st;
  }
  return fa::record_cuda_status(cudaFreeAsync(buf, stream), "host prefill cudaFreeAsync");
}
