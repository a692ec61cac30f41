"""Python binding of libfa_gb300.so (the C ABI declared in include/fa.h).

Argument marshalling only: every step of the attention runs in the CUDA
kernels of the library.  PyTorch supplies device memory and streams.  There is
no fallback: if the library is missing or cannot be loaded, every call raises.

Raw entry points (same names and argument order as the C ABI; pointers are
integers, ``stream`` a ``cudaStream_t`` value):
    fa_prefill_fwd, fa_prefill_fwd_lse, fa_prefill_varlen_fwd, fa_decode_fwd, fa_decode_fwd_lse,
    fa_decode_paged_fwd, fa_backward,
    fa_decode_fwd_noalloc, fa_status_string, fa_device_error, fa_last_cuda_error,
    fa_num_sms, fa_prefill_work_item, fa_prefill_rescale_count, fa_set_wait_limit_ns,
    fa_prefill_fwd_host, fa_prefill_host_pieces
Tensor conveniences (contiguous CUDA tensors, caller-owned outputs):
    prefill(q, k, v, scale, causal, out=None, stream=None, lse=None)
    prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, scale, causal,
                   out=None, stream=None, lse=None)
    decode(q, kcache, vcache, valid_len, scale, out=None, stream=None, lse=None)
    decode_paged(q, kpages, vpages, page_table, seqlens, scale, out=None, stream=None,
                 lse=None)
    backward(q, k, v, o, dout, lse, scale, causal, stream=None) -> (dq, dk, dv)
    prefill_host(q, k, v, out, scale, causal, n_pieces=16, stream=None)
    (lse=True allocates the fp32 log-sum-exp output; a tensor is used as is.)
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_BF16, FA_FP16 = 0, 1
FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_ERR_TOO_LARGE = 5
FA_ERR_BOUNDS = 6

# Every symbol include/fa.h declares (checked by the tests against the header).
EXPORTS = ("fa_prefill_fwd", "fa_prefill_fwd_lse", "fa_prefill_varlen_fwd", "fa_decode_fwd",
           "fa_decode_fwd_lse", "fa_decode_paged_fwd", "fa_backward",
           "fa_decode_fwd_noalloc", "fa_status_string", "fa_device_error", "fa_last_cuda_error",
           "fa_num_sms", "fa_prefill_work_item", "fa_prefill_rescale_count",
           "fa_set_wait_limit_ns", "fa_prefill_fwd_host", "fa_prefill_host_pieces")

_lib = None


class FAError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        extra = ""
        if status == FA_ERR_CUDA:
            code, site = fa_last_cuda_error()
            extra = f"; cudaError {code} at {site}"
        super().__init__(f"{what}: {fa_status_string(status)} (status {status}{extra})")


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} not found: build it with `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_prefill_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp]
    lib.fa_prefill_fwd.restype = i32
    lib.fa_prefill_fwd_lse.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                       i32, vp]
    lib.fa_prefill_fwd_lse.restype = i32
    lib.fa_prefill_varlen_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                          i32, i32, f32, i32, i32, vp]
    lib.fa_prefill_varlen_fwd.restype = i32
    lib.fa_decode_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
    lib.fa_decode_fwd.restype = i32
    lib.fa_decode_fwd_lse.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
    lib.fa_decode_fwd_lse.restype = i32
    lib.fa_decode_paged_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                        i32, i32, f32, vp]
    lib.fa_decode_paged_fwd.restype = i32
    lib.fa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                f32, i32, i32, vp]
    lib.fa_backward.restype = i32
    lib.fa_decode_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp]
    lib.fa_decode_fwd_noalloc.restype = i32
    lib.fa_status_string.argtypes = [i32]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_device_error.argtypes = [i32, ctypes.POINTER(ctypes.c_uint)]
    lib.fa_device_error.restype = i32
    lib.fa_last_cuda_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
    lib.fa_last_cuda_error.restype = i32
    lib.fa_num_sms.argtypes = []
    lib.fa_num_sms.restype = i32
    ip = ctypes.POINTER(ctypes.c_int)
    lib.fa_prefill_work_item.argtypes = [i32, i32, i32, i32, i32, i32, i32, ip, ip, ip]
    lib.fa_prefill_work_item.restype = i32
    lib.fa_prefill_rescale_count.argtypes = [i32, ctypes.POINTER(ctypes.c_ulonglong)]
    lib.fa_prefill_rescale_count.restype = i32
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_wait_limit_ns.restype = i32
    lib.fa_prefill_fwd_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                        i32, i32, vp]
    lib.fa_prefill_fwd_host.restype = i32
    lib.fa_prefill_host_pieces.argtypes = [i32, i32, i32, i32, i32, ip, ip, ip, ip, i32]
    lib.fa_prefill_host_pieces.restype = i32
    _lib = lib
    return lib


# ----------------------------------------------------------------------------
# Raw C-ABI mirrors
# ----------------------------------------------------------------------------
def fa_prefill_fwd(q, k, v, o, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype, stream):
    return load().fa_prefill_fwd(q, k, v, o, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype, stream)


def fa_prefill_fwd_lse(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype, stream):
    return load().fa_prefill_fwd_lse(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype,
                                     stream)


def fa_prefill_varlen_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q,
                          total_k, max_seqlen_q, D, scale, causal, dtype, stream):
    return load().fa_prefill_varlen_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv,
                                        total_q, total_k, max_seqlen_q, D, scale, causal, dtype,
                                        stream)


def fa_prefill_fwd_host(q_host, k_host, v_host, o_host, B, Hq, Hkv, Sq, Sk, D, scale, causal,
                        dtype, n_pieces, stream):
    return load().fa_prefill_fwd_host(q_host, k_host, v_host, o_host, B, Hq, Hkv, Sq, Sk, D,
                                      scale, causal, dtype, n_pieces, stream)


def fa_prefill_host_pieces(B, Sq, Sk, causal, n_pieces):
    """The piece plan of fa_prefill_fwd_host: a list of (b, s0, s1, sk) in
    upload order (rows [s0, s1) of sequence b see keys [0, sk))."""
    lib = load()
    n = lib.fa_prefill_host_pieces(B, Sq, Sk, int(bool(causal)), n_pieces, None, None, None,
                                   None, 0)
    if n < 0:
        raise ValueError("bad arguments")
    arr = [(ctypes.c_int * max(n, 1))() for _ in range(4)]
    lib.fa_prefill_host_pieces(B, Sq, Sk, int(bool(causal)), n_pieces, *arr, n)
    return [tuple(a[i] for a in arr) for i in range(n)]


def fa_decode_fwd(q, kcache, vcache, valid_len_dev, o, B, Hq, Hkv, cap, D, scale, stream):
    return load().fa_decode_fwd(q, kcache, vcache, valid_len_dev, o, B, Hq, Hkv, cap, D, scale,
                                stream)


def fa_decode_paged_fwd(q, kpages, vpages, page_table, seqlens, o, lse, B, Sq, Hq, Hkv,
                        num_pages, page_size, max_pages, D, scale, stream):
    return load().fa_decode_paged_fwd(q, kpages, vpages, page_table, seqlens, o, lse, B, Sq, Hq,
                                      Hkv, num_pages, page_size, max_pages, D, scale, stream)


def fa_decode_fwd_lse(q, kcache, vcache, valid_len_dev, o, lse, B, Hq, Hkv, cap, D, scale,
                      stream):
    return load().fa_decode_fwd_lse(q, kcache, vcache, valid_len_dev, o, lse, B, Hq, Hkv, cap, D,
                                    scale, stream)


def fa_decode_fwd_noalloc(q, kcache, vcache, valid_len_dev, o, B, Hq, Hkv, cap, D, scale,
                          stream):
    """fa_decode_fwd without any device allocation: for callers that must not
    allocate while they run (memory reserved once at start-up, allocator locks
    held, runtimes that forbid allocation after initialisation).  Its partials
    live in a fixed 4 MiB array inside the library, shared by every call on the
    device; calls overlapping on the GPU race on it.  Make the first call on a
    device before any stream capture (it looks up the array's address).
    Returns FA_ERR_TOO_LARGE for requests whose partials do not fit."""
    return load().fa_decode_fwd_noalloc(q, kcache, vcache, valid_len_dev, o, B, Hq, Hkv, cap, D,
                                        scale, stream)


def fa_status_string(status) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_device_error(reset=1):
    """(status, detail bits) of the device-side error word; synchronises."""
    detail = ctypes.c_uint(0)
    st = load().fa_device_error(int(reset), ctypes.byref(detail))
    return st, detail.value


def fa_last_cuda_error():
    """(raw cudaError_t, failing call) of this thread's latest FA_ERR_CUDA."""
    site = ctypes.c_char_p()
    code = load().fa_last_cuda_error(ctypes.byref(site))
    return code, (site.value or b"").decode()


def fa_num_sms() -> int:
    return load().fa_num_sms()


def fa_prefill_work_item(w, B, Hq, Hkv, Sq, Sk=0, causal=1):
    """(n_items, b, hq, qblock) of the persistent scheduler's item w."""
    b, hq, qb = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    n = load().fa_prefill_work_item(w, B, Hq, Hkv, Sq, Sk, causal, ctypes.byref(b),
                                     ctypes.byref(hq), ctypes.byref(qb))
    return n, b.value, hq.value, qb.value


def fa_prefill_rescale_count(reset=0):
    """(status, count): prefill (row, K/V tile) steps that took the lazy
    rescale since the last reset; synchronises."""
    c = ctypes.c_ulonglong(0)
    st = load().fa_prefill_rescale_count(int(reset), ctypes.byref(c))
    return st, c.value


def fa_set_wait_limit_ns(ns):
    """Time limit of every device pipeline wait (0: the 2 s default);
    synchronises."""
    return load().fa_set_wait_limit_ns(int(ns))


# ----------------------------------------------------------------------------
# Tensor conveniences
# ----------------------------------------------------------------------------
def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp16)")


def _check(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _lse_tensor(lse, shape, like):
    import torch
    if lse is True:
        return torch.empty(shape, dtype=torch.float32, device=like.device)
    if lse.dtype != torch.float32 or tuple(lse.shape) != tuple(shape):
        raise ValueError(f"lse must be a float32 tensor of shape {tuple(shape)}")
    _check(lse, "lse")
    return lse


def prefill(q, k, v, scale, causal, out=None, stream=None, lse=None):
    """O = softmax(scale * Q K^T [+ causal mask]) V.

    q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D]: contiguous CUDA bf16/fp16 tensors.
    Returns ``out`` (allocated like q if None).  Enqueued on ``stream``
    (default: torch's current stream); no host synchronisation.
    lse: None, True (allocate) or a float32 [B,Hq,Sq] tensor; when given,
    returns (out, lse) with each row's log-sum-exp (-inf: no visible key).
    """
    import torch
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k, v")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out")
    if lse is not None and lse is not False:
        lse = _lse_tensor(lse, (B, Hq, Sq), q)
        st = fa_prefill_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, Hq, Hkv, Sq, Sk, D, float(scale),
                                int(bool(causal)), _dtype_code(q), _stream_handle(stream))
        if st != FA_OK:
            raise FAError(st, "fa_prefill_fwd_lse")
        return out, lse
    st = fa_prefill_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv,
                        Sq, Sk, D, float(scale), int(bool(causal)), _dtype_code(q),
                        _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_prefill_fwd")
    return out


def prefill_host(q, k, v, out, scale, causal, n_pieces=16, stream=None):
    """fa_prefill_fwd_host: O = softmax(scale * Q K^T [+ causal mask]) V from
    host tensors q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] into the host tensor ``out``
    (contiguous, bf16/fp16; pinned for the copies to overlap the kernels).
    Enqueued on ``stream`` (default: torch's current stream); ``out`` is
    complete once that stream reaches the point after this call."""
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, k, v, out")
    if k.dtype != q.dtype or v.dtype != q.dtype or out.dtype != q.dtype:
        raise TypeError("q, k, v, out must share a dtype")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    st = fa_prefill_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv,
                             Sq, Sk, D, float(scale), int(bool(causal)), _dtype_code(q),
                             int(n_pieces), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_prefill_fwd_host")
    return out


def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, scale, causal, out=None,
                   stream=None, lse=None):
    """Attention over packed sequences of different lengths.

    q [total_q,Hq,D], k/v [total_k,Hkv,D]: contiguous CUDA bf16/fp16 tensors;
    cu_seqlens_q / cu_seqlens_k: int32 CUDA tensors [B+1] (prefix sums of the
    lengths, read on the device only); max_seqlen_q >= every query length.
    Returns ``out`` ([total_q,Hq,D]), or (out, lse) with lse [Hq,total_q] fp32
    when lse is True or a tensor.
    """
    import torch
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    if Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch between q, k, v")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cu_seqlens_q, "cu_seqlens_q"),
                 (cu_seqlens_k, "cu_seqlens_k")):
        _check(t, n)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32 CUDA tensors")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B+1 entries")
    B = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out")
    lse_ptr = 0
    if lse is not None and lse is not False:
        lse = _lse_tensor(lse, (Hq, total_q), q)
        lse_ptr = lse.data_ptr()
    st = fa_prefill_varlen_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                               cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, Hq, Hkv,
                               total_q, total_k, int(max_seqlen_q), D, float(scale),
                               int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_prefill_varlen_fwd")
    return (out, lse) if lse_ptr else out


def decode(q, kcache, vcache, valid_len, scale, out=None, stream=None, lse=None):
    """Single-token decode over the first L tokens of the cache.

    q [B,1,Hq,D] (or [B,Hq,D]) bf16; kcache/vcache [B,cap,Hkv,D] bf16;
    valid_len: int32 CUDA tensor holding L (read on the device only).
    Returns ``out`` shaped like q; with lse (True or a float32 [B,Hq] tensor)
    returns (out, lse).
    """
    import torch
    B, cap, Hkv, D = kcache.shape
    Hq = q.shape[-2]
    if q.shape[0] != B or q.shape[-1] != D or q.numel() != B * Hq * D:
        raise ValueError("q must be [B,1,Hq,D] matching the cache")
    if tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("kcache and vcache shapes differ")
    for t, n in ((q, "q"), (kcache, "kcache"), (vcache, "vcache"), (valid_len, "valid_len")):
        _check(t, n)
    if valid_len.dtype != torch.int32:
        raise TypeError("valid_len must be an int32 CUDA tensor")
    if q.dtype != torch.bfloat16 or kcache.dtype != torch.bfloat16 or vcache.dtype != torch.bfloat16:
        raise TypeError("decode takes bf16 q/kcache/vcache")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out")
    if lse is not None and lse is not False:
        lse = _lse_tensor(lse, (B, Hq), q)
        st = fa_decode_fwd_lse(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                               valid_len.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
                               cap, D, float(scale), _stream_handle(stream))
        if st != FA_OK:
            raise FAError(st, "fa_decode_fwd_lse")
        return out, lse
    st = fa_decode_fwd(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), valid_len.data_ptr(),
                       out.data_ptr(), B, Hq, Hkv, cap, D, float(scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_decode_fwd")
    return out


def decode_paged(q, kpages, vpages, page_table, seqlens, scale, out=None, stream=None, lse=None):
    """Decode of Sq new tokens for each of B sequences over a paged cache.

    q [B,Sq,Hq,D] (or [B,Hq,D] for Sq = 1) bf16; kpages/vpages
    [num_pages,page_size,Hkv,D] bf16; page_table int32 CUDA [B,max_pages];
    seqlens int32 CUDA [B] (lengths including the new tokens).  Returns ``out``
    shaped like q, or (out, lse) with lse [B,Sq,Hq] fp32 when lse is True or a
    tensor.
    """
    import torch
    num_pages, page_size, Hkv, D = kpages.shape
    B, max_pages = page_table.shape
    Hq = q.shape[-2]
    Sq = q.shape[1] if q.dim() == 4 else 1
    if q.shape[0] != B or q.shape[-1] != D or q.numel() != B * Sq * Hq * D:
        raise ValueError("q must be [B,Sq,Hq,D] matching the page table and pages")
    if tuple(vpages.shape) != tuple(kpages.shape):
        raise ValueError("kpages and vpages shapes differ")
    for t, n in ((q, "q"), (kpages, "kpages"), (vpages, "vpages"), (page_table, "page_table"),
                 (seqlens, "seqlens")):
        _check(t, n)
    if page_table.dtype != torch.int32 or seqlens.dtype != torch.int32 or seqlens.numel() != B:
        raise TypeError("page_table and seqlens must be int32 CUDA tensors ([B,max_pages], [B])")
    if q.dtype != torch.bfloat16 or kpages.dtype != torch.bfloat16 or vpages.dtype != torch.bfloat16:
        raise TypeError("decode takes bf16 q and pages")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out")
    lse_ptr = 0
    if lse is not None and lse is not False:
        lse = _lse_tensor(lse, (B, Sq, Hq), q)
        lse_ptr = lse.data_ptr()
    st = fa_decode_paged_fwd(q.data_ptr(), kpages.data_ptr(), vpages.data_ptr(),
                             page_table.data_ptr(), seqlens.data_ptr(), out.data_ptr(), lse_ptr,
                             B, Sq, Hq, Hkv, num_pages, page_size, max_pages, D, float(scale),
                             _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_decode_paged_fwd")
    return (out, lse) if lse_ptr else out


def fa_backward(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, scale, causal, dtype,
                stream):
    return load().fa_backward(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, scale,
                              causal, dtype, stream)


def backward(q, k, v, o, dout, lse, scale, causal, stream=None):
    """Gradients (dq, dk, dv) of sum(o * dout) for the forward call that
    produced o and lse (fa_prefill_fwd_lse).  q/o/dout [B,Sq,Hq,D], k/v
    [B,Sk,Hkv,D] contiguous CUDA tensors of one dtype; lse float32
    [B,Hq,Sq]."""
    import torch
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout"), (lse, "lse")):
        _check(t, n)
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape) or \
            tuple(v.shape) != tuple(k.shape) or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("shape mismatch among q, k, v, o, dout, lse")
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                     lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq,
                     Sk, D, float(scale), int(bool(causal)), _dtype_code(q),
                     _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_backward")
    return dq, dk, dv
