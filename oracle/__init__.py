"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the cpu_baseline / reference leg
of ``bench.py`` may import this package.  The CUDA product path
(``attention_fa_fwd_04_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, one query row at a
time: explicit scores, max-subtracted exponentials, one division).  This module
only widens the caller's bf16/fp16 tensors to float64 (exact) and marshals
arguments.  See ``attn_oracle.c`` for the definition and its sources:

- tessera #90 "compiler-generated flash_attn fwd+bwd", flash_attn forward
  commit note (scale*Q@K^T, causal/ragged mask, softmax, P@V);
- "Dense flash-attention prefill (gfx950 / MI355X)", opening paragraph
  (forward, MHA or GQA, causal);
- rocm-libraries #13108 "minimal single-token attention decode", interface
  description (Sq=1, token-major cache, device valid length).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _bind(path):
    """Load the compiled oracle at ``path`` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_int64)
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_attention_rows.argtypes = [dp, dp, dp, dp, lp, i64, i32, i32,
                                          i32, i64, i64, i32, f64, i32, i32]
    lib.oracle_attention_rows.restype = i32
    lib.oracle_attention_rows_lse.argtypes = [dp, dp, dp, dp, dp, lp, i64, i32, i32,
                                              i32, i64, i64, i32, f64, i32, i32]
    lib.oracle_attention_rows_lse.restype = i32
    lib.oracle_attention_probs.argtypes = [dp, dp, dp, dp, dp, i32, i32, i64,
                                           i32, i32, i32, i64, i64, i32, f64, i32]
    lib.oracle_attention_probs.restype = i32
    lib.oracle_decode.argtypes = [dp, dp, dp, dp, i32, i32, i32, i64, i32, i64, f64]
    lib.oracle_decode.restype = i32
    lib.oracle_decode_lse.argtypes = [dp, dp, dp, dp, dp, i32, i32, i32, i64, i32, i64, f64]
    lib.oracle_decode_lse.restype = i32
    lib.oracle_attention_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i32, i32, i32, i64,
                                         i64, i32, f64, i32, i32]
    lib.oracle_attention_bwd.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(_build.build())
    return _lib


def _f64(t) -> np.ndarray:
    """Exact widening of a torch tensor (bf16/fp16/fp32/fp64) or array to a
    C-contiguous float64 numpy array."""
    if hasattr(t, "detach"):
        import torch
        return np.ascontiguousarray(t.detach().to("cpu", torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _ptr(a: np.ndarray, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def attention(q, k, v, scale: float, causal: bool, rows=None, nthreads=None,
              return_lse=False):
    """O for q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D].

    rows=None: full output, float64 [B,Sq,Hq,D].
    rows=int array [n,3] of (b, h, i): float64 [n, D], row r = O[b,i,h,:].
    return_lse: also return the log-sum-exp of each row's scores (-inf for a
    row with no visible key): [B,Hq,Sq] for rows=None, else [n].
    """
    lib = _load()
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    assert Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape)
    kd, vd = _f64(k), _f64(v)
    if rows is None:
        b, i, h = np.meshgrid(np.arange(B), np.arange(Sq), np.arange(Hq), indexing="ij")
        rows_arr = np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int64)
        q_rows = _f64(q).reshape(-1, D)  # [B*Sq*Hq, D] in (b, i, h) order
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        qt = q[rows_arr[:, 0], rows_arr[:, 2], rows_arr[:, 1], :] if len(rows_arr) else q.reshape(0, D)
        q_rows = _f64(qt).reshape(-1, D)
    q_rows = np.ascontiguousarray(q_rows)
    n = rows_arr.shape[0]
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    if n:
        rc = lib.oracle_attention_rows_lse(
            _ptr(q_rows), _ptr(kd), _ptr(vd), _ptr(out), _ptr(lse),
            _ptr(rows_arr, ctypes.c_int64), n, B, Hq, Hkv, Sq, Sk, D, float(scale),
            int(bool(causal)), int(nthreads or default_threads()))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_rows failed with status {rc}")
    if rows is None:
        out = out.reshape(B, Sq, Hq, D)
        lse = np.ascontiguousarray(lse.reshape(B, Sq, Hq).transpose(0, 2, 1))
    return (out, lse) if return_lse else out


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool,
                     return_lse=False, nthreads=None):
    """Packed sequences: q [total_q,Hq,D], k/v [total_k,Hkv,D], cu_seqlens_* host
    sequences of B+1 prefix sums.  Sequence b is the dense problem on rows
    [cu_q[b], cu_q[b+1]) and keys [cu_k[b], cu_k[b+1]) (bottom-right causal
    within it), computed by the dense oracle above.  Returns float64
    [total_q,Hq,D] (and lse [Hq,total_q] when return_lse)."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    total_q, Hq, D = q.shape
    out = np.zeros((total_q, Hq, D), dtype=np.float64)
    lse = np.full((Hq, total_q), -np.inf, dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        o_b, l_b = attention(q[q0:q1].unsqueeze(0), k[k0:k1].unsqueeze(0),
                             v[k0:k1].unsqueeze(0), scale, causal, nthreads=nthreads,
                             return_lse=True)
        out[q0:q1] = o_b[0]
        lse[:, q0:q1] = l_b[0]
    return (out, lse) if return_lse else out


def decode_paged(q, kpages, vpages, page_table, seqlens, scale: float, return_lse=False):
    """Decode of Sq new tokens per sequence over a paged cache: sequence b's
    token t lives in page page_table[b][t // page_size], slot t % page_size.
    Each sequence's first L = seqlens[b] tokens (clamped to the table's
    capacity) are gathered into a contiguous cache; its Sq new query tokens
    are the last Sq positions, so the dense oracle with bottom-right causal
    masking (Sq rows against L keys) gives the result.
    q [B,Sq,Hq,D] (or [B,Hq,D] for Sq = 1); pages [num_pages,page_size,Hkv,D];
    page_table, seqlens host int sequences.  Returns float64 [B,Sq,Hq,D] (and
    lse [B,Sq,Hq])."""
    import torch
    num_pages, page_size, Hkv, D = kpages.shape
    table = [[int(x) for x in row] for row in page_table]
    B = len(table)
    qd = q.reshape(B, -1, q.shape[-2], D)
    Sq, Hq = qd.shape[1], qd.shape[2]
    out = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    lse = np.full((B, Sq, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        L = max(0, min(int(seqlens[b]), len(table[b]) * page_size))
        n_pages = -(-L // page_size)
        pages = torch.tensor(table[b][:n_pages], dtype=torch.long)
        kc = kpages[pages].reshape(1, n_pages * page_size, Hkv, D)[:, :L]
        vc = vpages[pages].reshape(1, n_pages * page_size, Hkv, D)[:, :L]
        o_b, l_b = attention(qd[b:b + 1], kc, vc, scale, True, return_lse=True)
        out[b], lse[b] = o_b[0], l_b[0].T
    return (out, lse) if return_lse else out


def attention_bwd(q, k, v, dout, scale: float, causal: bool, nthreads=None):
    """Gradients (dq [B,Sq,Hq,D], dk, dv [B,Sk,Hkv,D], float64) of the loss
    sum(O * dout) for the forward pass above (same masking and GQA map)."""
    lib = _load()
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    qd, kd, vd, dd = _f64(q), _f64(k), _f64(v), _f64(dout)
    dq = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    dk = np.zeros((B, Sk, Hkv, D), dtype=np.float64)
    dv = np.zeros((B, Sk, Hkv, D), dtype=np.float64)
    rc = lib.oracle_attention_bwd(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(dd), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, Hq, Hkv, Sq, Sk, D, float(scale),
                                  int(bool(causal)), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_bwd failed with status {rc}")
    return dq, dk, dv


def probs(q, k, v, scale: float, causal: bool, b: int, h: int, i: int):
    """(p [Sk], o [D]) of one query row: p over all Sk keys, 0 where masked."""
    lib = _load()
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    kd, vd = _f64(k), _f64(v)
    qrow = np.ascontiguousarray(_f64(q[b, i, h]))
    p = np.zeros(max(Sk, 1), dtype=np.float64)
    o = np.zeros(D, dtype=np.float64)
    rc = lib.oracle_attention_probs(_ptr(qrow), _ptr(kd), _ptr(vd), _ptr(p), _ptr(o),
                                    b, h, i, B, Hq, Hkv, Sq, Sk, D, float(scale),
                                    int(bool(causal)))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_probs failed with status {rc}")
    return p[:Sk], o


def decode(q, kcache, vcache, L: int, scale: float, return_lse=False):
    """Single-token decode. q [B,1,Hq,D] or [B,Hq,D]; caches [B,cap,Hkv,D];
    L = valid length (host int), clamped to [0, cap].  Returns float64 [B,Hq,D]
    (and the log-sum-exp [B,Hq] when return_lse)."""
    lib = _load()
    qd = _f64(q)
    B, cap, Hkv, D = kcache.shape
    qd = np.ascontiguousarray(qd.reshape(B, -1, D))
    Hq = qd.shape[1]
    kd, vd = _f64(kcache), _f64(vcache)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    rc = lib.oracle_decode_lse(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(out), _ptr(lse), B, Hq, Hkv,
                               cap, D, int(L), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed with status {rc}")
    return (out, lse) if return_lse else out
