/*
 * fa.h -- C ABI of the GB300 (sm_103a) flash-attention forward library
 *         (libfa_gb300.so).
 *
 * Two operations:
 *
 *   fa_prefill_fwd  dense attention forward, O = softmax(scale * Q K^T + mask) V,
 *                   for bf16/fp16, head_dim 64 or 128, MHA or GQA, causal or
 *                   not, Sq != Sk allowed.
 *                   Defined by: "Dense flash-attention prefill (gfx950 / MI355X)"
 *                   (opening paragraph: forward-only, bf16/fp16, head_dim
 *                   64/128, MHA or GQA, causal) and tessera #90
 *                   "compiler-generated flash_attn fwd+bwd" (flash_attn forward
 *                   commit note: S = scale*Q@K^T, causal/ragged mask, online
 *                   softmax, O += P@V; Sq/Sk/scale/causal are runtime values).
 *
 *   fa_decode_fwd   single-token attention over a KV cache whose valid length
 *                   lives in device memory, split over the sequence and merged
 *                   with a log-sum-exp combine.
 *                   Defined by: rocm-libraries #13108 "minimal single-token
 *                   attention decode" (interface description: Sq=1, contiguous
 *                   token-major K/V cache, device INT32 valid length, O only;
 *                   review finding: unused cache capacity may hold NaN and must
 *                   not reach the output; split-KV named as the next step).
 *
 *   fa_prefill_fwd_lse, fa_decode_fwd_lse
 *                   the same operations, also writing each row's log-sum-exp
 *                   lse = log sum_j exp(scale * <q, k_j>) over its visible keys
 *                   (fp32, natural log; -inf for a row with no visible key).
 *                   It is the per-row statistic a backward pass recomputes P
 *                   from (tessera #90, flash-attention backward commit note:
 *                   the "_pre" kernel's logsumexp) and the one partial results
 *                   over key ranges are merged by; rocm-libraries #13108 lists
 *                   the LSE output among what its first decode milestone
 *                   leaves out.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are contiguous, row-major, in device memory (or memory the device
 *   can address), 16-byte aligned:
 *       q, o   : [B, Sq, Hq,  D]     (decode: Sq = 1)
 *       k, v   : [B, Sk, Hkv, D]     (decode: [B, cap, Hkv, D], token-major)
 *   Query head h reads K/V head h / (Hq / Hkv) (contiguous GQA groups).
 * - The caller owns and allocates every tensor, including o.  The library
 *   keeps no pointer after the call returns.
 * - Work is enqueued on `stream`; no call synchronises the host.  A status of
 *   FA_OK means the work was validated and enqueued; device-side failures
 *   (a pipeline wait that exceeded its time limit) are reported by
 *   fa_device_error().
 * - Arguments are validated before anything touches the GPU; invalid
 *   arguments return FA_ERR_INVALID_ARG and enqueue nothing.
 * - Empty problems (B == 0, Sq == 0 or Hq == 0) are valid and enqueue nothing.
 *   Rows with no visible key (Sk == 0, or causal rows i with i + Sk - Sq < 0)
 *   produce O = 0.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* bad pointer, size, head config or dtype         */
  FA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement     */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed     */
  FA_ERR_TIMEOUT = 4,      /* a device-side pipeline wait hit its time limit  */
  FA_ERR_TOO_LARGE = 5,    /* request exceeds fa_decode_fwd_noalloc's scratch */
  FA_ERR_BOUNDS = 6        /* a device-side bounds check skipped an access     */
} fa_status_t;

/*
 * fa_prefill_fwd -- attention forward for a batch of full sequences.
 *
 *   q      [B, Sq, Hq, D]   bf16 or fp16 (dtype), read only
 *   k, v   [B, Sk, Hkv, D]  same dtype, read only
 *   o      [B, Sq, Hq, D]   same dtype, written (every element of every row)
 *   Hq % Hkv == 0; D in {64, 128}; Sq, Sk >= 0; B, Hq, Hkv >= 0.
 *   scale  multiplies Q K^T (any finite value, applied as passed).
 *   causal nonzero: row i sees keys j <= i + (Sk - Sq) (bottom-right aligned;
 *          equals the usual top-left mask when Sq == Sk).
 *   dtype  FA_BF16 or FA_FP16.
 *
 * Arithmetic: Q K^T and P V on the tensor cores with fp32 accumulation;
 * softmax in fp32 (exp2 domain); P rounded to the input dtype before P V;
 * O = (P V) / l rounded once to the output dtype (round to nearest even).
 *
 * Returns FA_OK, FA_ERR_INVALID_ARG (null/misaligned pointer, negative size,
 * Hq % Hkv != 0, D not 64/128, unknown dtype, non-finite scale),
 * or FA_ERR_CUDA (tensor-map encode, attribute or launch failure).
 */
int fa_prefill_fwd(const void* q, const void* k, const void* v, void* o,
                   int B, int Hq, int Hkv, int Sq, int Sk, int D,
                   float scale, int causal, int dtype, cudaStream_t stream);

/*
 * fa_prefill_fwd_lse -- fa_prefill_fwd that also writes
 *
 *   lse    [B, Hq, Sq]  fp32, 4-byte aligned, written:
 *          lse[b,h,i] = log sum_j exp(scale * <q[b,i,h], k[b,j,h/G]>) over the
 *          keys row i sees; -inf for a row that sees none.
 *
 * Everything else as fa_prefill_fwd; lse == NULL is FA_ERR_INVALID_ARG.
 */
int fa_prefill_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int Sq, int Sk, int D,
                       float scale, int causal, int dtype, cudaStream_t stream);

/*
 * fa_prefill_varlen_fwd -- fa_prefill_fwd over a batch of packed sequences of
 * different lengths (the gfx950 prefill README's TODO list names this
 * follow-up: packed varlen with per-sequence persistent scheduling).
 *
 *   q, o           [total_q, Hq, D]   sequences packed back to back
 *   k, v           [total_k, Hkv, D]
 *   cu_seqlens_q   [B + 1] int32 in device memory: sequence b's query rows are
 *   cu_seqlens_k   [cu_seqlens_q[b], cu_seqlens_q[b+1]), its keys likewise.
 *                  Read by the kernel only.
 *   max_seqlen_q   >= every query length (bounds the work plan)
 *   lse            NULL, or [Hq, total_q] fp32 written with each row's
 *                  log-sum-exp (-inf for a row with no visible key)
 *
 * Causal masking is bottom-right per sequence: row i of sequence b sees keys
 * j <= i + (Sk_b - Sq_b).  Keys of the neighbouring packed sequence that share
 * a tile are masked like keys past Sk.
 *
 * Scheduling: a one-CTA planning kernel reads the offsets on the device and
 * lists each sequence's 256-row query blocks, largest K/V tile count first;
 * the persistent prefill CTAs then claim (block, query head) items from that
 * list as they become free, so short and long sequences of a batch share the
 * grid instead of serialising.  The plan and the work counter live in
 * stream-ordered scratch (B * ceil(max_seqlen_q / 256) * 32 + 16 bytes).
 * Offsets that are not
 * 0 <= cu[b] <= cu[b+1] <= total, or a query length above max_seqlen_q, make
 * that sequence's rows unwritten and set the bounds bit reported by
 * fa_device_error().  Other rules as fa_prefill_fwd.
 */
int fa_prefill_varlen_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int B, int Hq, int Hkv, int total_q, int total_k, int max_seqlen_q,
                          int D, float scale, int causal, int dtype, cudaStream_t stream);

/*
 * fa_decode_fwd -- one new query token per sequence against a KV cache.
 *
 *   q              [B, 1, Hq, D]      bf16, read only
 *   kcache, vcache [B, cap, Hkv, D]   bf16, token-major, read only
 *   valid_len_dev  one int32 in device memory: the number of valid tokens L,
 *                  shared by the batch.  It is read by the kernels only (never
 *                  by the host), so the call never synchronises.  L is
 *                  clamped to [0, cap]; L == 0 gives O = 0.
 *   o              [B, 1, Hq, D]      bf16, written
 *   Hq % Hkv == 0; D in {64, 128}; cap >= 0.
 *
 * Cache entries at token positions >= L may hold anything, NaN and Inf
 * included: they are never used in arithmetic (zeroed in shared memory before
 * any MMA and given probability zero).
 *
 * Scratch: the split partials (fp32) are allocated stream-ordered on `stream`
 * (cudaMallocAsync / cudaFreeAsync), so calls on different streams never share
 * scratch.  Two kernels are enqueued: the split kernel and the combine, each
 * launched as a programmatic dependent of the grid before it on the stream:
 * before its griddepcontrol.wait a kernel only initialises shared-memory
 * barriers and prefetches its tensor maps, so it reads nothing an earlier
 * kernel may still be writing.
 *
 * Returns FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (dtype other than
 * bf16), or FA_ERR_CUDA.
 */
int fa_decode_fwd(const void* q, const void* kcache, const void* vcache,
                  const int32_t* valid_len_dev, void* o,
                  int B, int Hq, int Hkv, int cap, int D, float scale,
                  cudaStream_t stream);

/*
 * fa_decode_paged_fwd -- decode of Sq new tokens per sequence (Sq = 1: the
 * single-token step; Sq > 1: tokens proposed by speculative decoding) for a
 * batch of sequences with their own lengths, over a paged KV cache (the
 * decode PR's deferred items: batched shapes, several query tokens, and
 * non-contiguous KV storage).
 *
 *   q              [B, Sq, Hq, D]                   bf16, read only
 *   kpages, vpages [num_pages, page_size, Hkv, D]   bf16, read only
 *   page_table     [B, max_pages] int32, device: sequence b's tokens
 *                  [p*page_size, (p+1)*page_size) live in physical page
 *                  page_table[b][p]
 *   seqlens        [B] int32, device: sequence b's valid length L (including
 *                  its Sq new tokens, whose K/V are already in the cache),
 *                  clamped to [0, max_pages * page_size]
 *   o              [B, Sq, Hq, D]                   bf16, written
 *   lse            NULL, or [B, Sq, Hq] fp32 written with each row's
 *                  log-sum-exp
 *
 * New token s (0-based) sits at position L - Sq + s and sees the keys
 * [0, L - Sq + s] (bottom-right causal); rows that see no key give O = 0 and
 * lse = -inf.
 *   page_size      a positive multiple of 32
 *
 * Only the pages that hold a sequence's first seqlens[b] tokens are read; page
 * ids of a valid page must lie in [0, num_pages).  A page id outside that
 * range masks that page's tokens and sets the bounds bit reported by
 * fa_device_error().  Entries of pages past a sequence's length, and token
 * slots past its length in its last page, may hold anything (NaN included).
 * A contiguous cache with per-sequence lengths is the case page_size = cap,
 * max_pages = 1, page_table[b] = b.  Other rules as fa_decode_fwd.
 *
 * Scheduling: while the batch has fewer (sequence, kv head) units than SMs,
 * the kernels read the lengths on the device and give each sequence a number
 * of splits in proportion to its length (one CTA per SM), so a batch of very
 * different lengths keeps every SM streaming; otherwise each unit's share of
 * the SMs is sized from the capacity.  Either way the lengths are never read
 * on the host.
 */
int fa_decode_paged_fwd(const void* q, const void* kpages, const void* vpages,
                        const int32_t* page_table, const int32_t* seqlens, void* o, float* lse,
                        int B, int Sq, int Hq, int Hkv, int num_pages, int page_size,
                        int max_pages, int D, float scale, cudaStream_t stream);

/*
 * fa_decode_fwd_lse -- fa_decode_fwd that also writes
 *
 *   lse    [B, Hq]  fp32, 4-byte aligned, written: the log-sum-exp of each
 *          head's scores over the L valid tokens; -inf when L == 0.
 *
 * Everything else as fa_decode_fwd; lse == NULL is FA_ERR_INVALID_ARG.
 */
int fa_decode_fwd_lse(const void* q, const void* kcache, const void* vcache,
                      const int32_t* valid_len_dev, void* o, float* lse,
                      int B, int Hq, int Hkv, int cap, int D, float scale,
                      cudaStream_t stream);

/*
 * fa_decode_fwd_noalloc -- fa_decode_fwd for callers that cannot allocate
 * device memory during the call.
 *
 * No counterpart in the source material: the pages describe no
 * allocation-free variant; this is a deployment convenience of this library.
 *
 * Same arguments, layouts, results and errors as fa_decode_fwd, but the split
 * partials live in one fixed device array inside the library (4 MiB of fp32,
 * held by every GPU that loads the library until the process exits) instead of
 * memory from cudaMallocAsync.  It calls no allocating routine.  Meant for
 * code that must not allocate while it runs: serving loops with memory reserved
 * once at start-up, code running under an allocator lock, runtimes that forbid
 * allocation after initialisation.
 *
 * - Requests whose partials need more than the array holds
 *   (B * Hq * nsplit * (D + 2) floats, nsplit <= SM count) return
 *   FA_ERR_TOO_LARGE and enqueue nothing.
 * - The array is shared by all calls on a device: calls whose kernels overlap
 *   on the GPU (different streams with no ordering) race on it; calls ordered
 *   on one stream are safe.  No contents need to start at zero.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current).  Make that first call
 *   before any stream capture on the device.
 */
int fa_decode_fwd_noalloc(const void* q, const void* kcache, const void* vcache,
                          const int32_t* valid_len_dev, void* o,
                          int B, int Hq, int Hkv, int cap, int D, float scale,
                          cudaStream_t stream);

/*
 * fa_backward -- gradients of the loss sum(O * dout) with respect to q, k and
 * v (the flash-attention backward of tessera #90's backward commit note:
 * a "_pre" pass Delta = rowsum(dout * O), then dQ and dK/dV passes that
 * recompute P from the forward's log-sum-exp).
 *
 *   q, o, dout [B, Sq, Hq, D]    the forward's inputs, output, and the
 *                                output gradient (dtype), read only
 *   k, v       [B, Sk, Hkv, D]   read only
 *   lse        [B, Hq, Sq] fp32  the forward's log-sum-exp
 *                                (fa_prefill_fwd_lse), read only
 *   dq         [B, Sq, Hq, D]    written
 *   dk, dv     [B, Sk, Hkv, D]   written; query heads of a GQA group add
 *                                into their kv head
 *   scale, causal                as in the forward call
 *
 * Delta lives in stream-ordered scratch (B * Hq * Sq fp32).  Three kernels
 * are enqueued.  Other rules as fa_prefill_fwd.
 */
int fa_backward(const void* q, const void* k, const void* v, const void* o,
                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                int dtype, cudaStream_t stream);

/*
 * fa_prefill_fwd_host -- fa_prefill_fwd from host memory to host memory, with
 * the copies overlapped with the kernels.
 *
 *   q_host, o_host  [B, Sq, Hq, D]   in host memory (read / written)
 *   k_host, v_host  [B, Sk, Hkv, D]  in host memory (read)
 *   n_pieces        >= 1: query-row pieces per sequence (16 suits long
 *                   sequences; 1 = copies and kernel one after the other)
 *   other arguments as fa_prefill_fwd.
 *
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister):
 * with pageable memory the result is the same but the copies do not overlap.
 * The query rows of each sequence are split into at most n_pieces pieces on
 * 256-row boundaries; rows [s0, s1) see the key prefix [0, sk), sk = Sk, or
 * with causal masking min(Sk, max(0, s1 + Sk - Sq)), and form an ordinary
 * bottom-right aligned prefill of s1 - s0 rows over sk keys -- the same rows
 * and keys as in the whole problem, so O is bit-identical to fa_prefill_fwd's.
 * K and V are uploaded first, then Q piece by piece (heaviest piece first);
 * each piece's kernel runs as soon as its rows have landed and its O rows go
 * back while later pieces compute.
 *
 * Device copies of q, k, v, o are allocated stream-ordered on `stream`
 * (2 * B * (Sq * Hq + Sk * Hkv) * D * 2 bytes, freed on `stream` after the
 * last download).  Two copy streams and two compute streams per device (the
 * pieces' kernels alternate between them, so each fills the SMs the other's
 * last wave leaves idle), created on first use and kept, fork from `stream`
 * and join it again: work already on
 * `stream` runs first, and `stream` waits for the last download, so o_host is
 * complete once `stream` reaches that point (the call itself does not
 * synchronise).  Calls on one device are enqueued one at a time.
 *
 * Returns FA_OK, FA_ERR_INVALID_ARG (as fa_prefill_fwd, null host pointer,
 * n_pieces < 1) or FA_ERR_CUDA.
 */
int fa_prefill_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                        void* o_host, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                        float scale, int causal, int dtype, int n_pieces, cudaStream_t stream);

/*
 * fa_prefill_host_pieces -- the piece plan of fa_prefill_fwd_host, for
 * inspection and tests: fills b, s0, s1, sk (each may be NULL) for the first
 * min(count, max_pieces) pieces in the order they are uploaded, and returns
 * count, or -1 on bad arguments.  No GPU access.
 */
int fa_prefill_host_pieces(int B, int Sq, int Sk, int causal, int n_pieces,
                           int* b, int* s0, int* s1, int* sk, int max_pieces);

/* Static, human-readable name of a status code (never NULL). */
const char* fa_status_string(int status);

/*
 * fa_device_error -- read (and if reset != 0, clear) the device-side error
 * words of the current device.  Synchronises the current device.  Returns
 * FA_OK if no kernel reported a failure, FA_ERR_TIMEOUT if a pipeline wait
 * hit its time limit, FA_ERR_BOUNDS if only bounds checks fired (packed
 * offsets or page ids out of range, or an index self-check), FA_ERR_CUDA if
 * the read itself failed.
 * If detail != NULL it receives the raw bits: the prefill (and backward) word
 * in bits 0-15, the decode word in bits 16-31; in each, bit 0 = a wait timed out (bits 8-15:
 * which wait), bit 1 = a bounds check fired.  Bounds bit with site 15: the
 * D = 128 backward dK/dV kernel found its dynamic shared memory too far from
 * a 1 KiB boundary to lay out its rings, and its CTAs left without work.
 */
int fa_device_error(int reset, unsigned int* detail);

/*
 * fa_last_cuda_error -- the raw cudaError_t behind the most recent
 * FA_ERR_CUDA returned to the calling thread (0 if none), and, if site is not
 * NULL, a static string naming the call that failed.
 */
int fa_last_cuda_error(const char** site);

/* Number of SMs the persistent prefill grid uses on the current device
 * (queried once per device), or a negative value on failure. */
int fa_num_sms(void);

/*
 * fa_prefill_rescale_count -- how often the prefill softmax took its lazy
 * rescale on the current device since the last reset: the number of
 * (query row, K/V tile) steps at which O and the row sum were rescaled to a
 * new running max and the tile's P recomputed.
 *
 * The lazy rescale is the "lazy" lever of "Dense flash-attention prefill
 * (gfx950 / MI355X)", *Measured*: the softmax exponentiates each K/V tile
 * against the row's running max without first taking the tile's own max, and
 * only when the tile's row sum of P exceeds 2^60 (bf16 P) or 2^15 (fp16 P),
 * or the row had no finite score before, does it find the new max, rescale
 * and recompute.  Scores of ordinary inputs never trigger it; a count that
 * grows on a workload says its scores jump by tens of units within rows.
 *
 *   reset  nonzero: clear the counter after reading it
 *   count  receives the value (non-NULL)
 *
 * Synchronises the current device.  Returns FA_OK, FA_ERR_INVALID_ARG
 * (count == NULL) or FA_ERR_CUDA.
 */
int fa_prefill_rescale_count(int reset, unsigned long long* count);

/*
 * fa_set_wait_limit_ns -- time limit of every device-side pipeline wait
 * (mbarrier waits of the prefill, decode and backward kernels) on the current
 * device; ns == 0 restores the default of 2 s.
 *
 * A wait that runs past the limit makes its CTA abort: every warp leaves its
 * loop, the loads and MMAs already in flight are waited for (each such
 * teardown wait keeps the fixed 2 s limit), tensor memory is freed, and the
 * timeout bit plus the wait's site are set in the error word read by
 * fa_device_error().  The outputs of an aborted call are undefined.  The
 * default is far above any wait of a healthy call; a short limit serves as a
 * watchdog, or in tests to make the timeout path run.
 *
 * Below 1 ms the limit is a watchdog: the decode kernels, and the dense
 * prefill (whose launches then use a polling instantiation of the kernel),
 * check it at every probe of every wait.  The packed-sequence prefill and the
 * backward kernels keep suspending probes of about 4 us each, so there a wait
 * trips the watchdog only once it has lasted about two of them.
 *
 * Synchronises the current device and applies to calls enqueued afterwards.
 * Returns FA_OK or FA_ERR_CUDA.
 */
int fa_set_wait_limit_ns(unsigned long long ns);

/*
 * fa_prefill_work_item -- host copy of the persistent scheduler's work-item
 * decode, for inspection and tests.  Work item w in [0, n_items) maps to
 * (b, hq, qblock); a qblock is 256 query rows.  Returns the number of items
 * n_items = B * Hq * ceil(Sq / 256), and fills *b, *hq, *qblock when
 * 0 <= w < n_items (the pointers may be NULL).  Returns -1 on bad arguments.
 *
 * Items are numbered kv-head-major, longest causal query blocks first.  In a
 * dense launch the persistent CTAs claim items in that order from a work
 * counter (the next free CTA takes the next item).  (Packed sequences,
 * fa_prefill_varlen_fwd, claim from a list planned on the device instead.)
 */
int fa_prefill_work_item(int w, int B, int Hq, int Hkv, int Sq, int Sk, int causal,
                         int* b, int* hq, int* qblock);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
