"""Prefill from pinned host buffers with the copies overlapped with the kernels.

A caller whose Q, K, V live in host memory pays for moving them to the device
and for moving O back.  Done one after the other, those copies (570 MB at the
B1 Hq128 Hkv8 S8192 D128 shape) take longer than the kernel.  The query rows
of one sequence split into independent pieces: rows [s0, s1) need only the
keys they can see, and that piece is again an ordinary prefill (with causal
masking, a bottom-right aligned one), so it runs through fa_prefill_fwd
unchanged.  HostPrefill sends K and V first, then Q piece by piece (heaviest
piece first) on one copy stream.  Each piece's kernel starts as soon as its
rows have landed, and its O goes back on a second copy stream.  Uploads,
kernels and downloads of different pieces overlap.

Host orchestration only: every attention step runs in the library's kernels.
"""
import torch

from . import FA_OK, FAError, _dtype_code, fa_prefill_fwd


def prefill_row_chunks(Sq, Sk, causal, n_chunks, unit=256):
    """Split the Sq query rows of one sequence into at most n_chunks pieces.

    Returns a list of (s0, s1, sk): query rows [s0, s1) and the key prefix
    [0, sk) that any of them can see.  Piece boundaries fall on multiples of
    `unit` rows (the prefill kernel's work unit), except the end.  Without
    causal masking every piece sees all Sk keys.  With bottom-right causal
    masking (row i sees keys j <= i + Sk - Sq), sk = s1 + Sk - Sq clamped to
    [0, Sk].  The piece, taken as a prefill of Sq' = s1 - s0 rows over sk keys
    with the same bottom-right alignment, gives its row r exactly the keys
    that row s0 + r sees in the whole problem.
    """
    if Sq <= 0:
        return []
    n_units = (Sq + unit - 1) // unit
    n = max(1, min(int(n_chunks), n_units))
    pieces = []
    for c in range(n):
        s0 = min(Sq, (c * n_units // n) * unit)
        s1 = min(Sq, ((c + 1) * n_units // n) * unit)
        if s1 <= s0:
            continue
        sk = min(Sk, max(0, s1 + Sk - Sq)) if causal else Sk
        pieces.append((s0, s1, sk))
    return pieces


class HostPrefill:
    """O = softmax(scale * Q K^T [+ causal mask]) V from pinned host tensors.

    Shapes: q, out [B, Sq, Hq, D]; k, v [B, Sk, Hkv, D] (bf16 or fp16), all
    in pinned host memory.  The object owns its device buffers, two copy
    streams, a compute stream and the events that order them.  Reuse it for
    calls of the same shape.

    A call is ordered after the work already on the caller's stream, and the
    caller's stream waits for its last download.  Events recorded on that
    stream around the call therefore time the whole host-to-host operation.
    """

    def __init__(self, B, Hq, Hkv, Sq, Sk, D, dtype, causal, n_chunks=8, device=None):
        self.B, self.Hq, self.Hkv, self.Sq, self.Sk, self.D = B, Hq, Hkv, Sq, Sk, D
        self.dtype, self.causal = dtype, bool(causal)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.q = torch.empty(B, Sq, Hq, D, dtype=dtype, device=dev)
        self.k = torch.empty(B, Sk, Hkv, D, dtype=dtype, device=dev)
        self.v = torch.empty(B, Sk, Hkv, D, dtype=dtype, device=dev)
        self.o = torch.empty(B, Sq, Hq, D, dtype=dtype, device=dev)
        self.up = torch.cuda.Stream(device=dev)
        self.comp = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        # (b, s0, s1, sk) for every piece of every sequence of the batch, the
        # heaviest first (with causal masking the later rows see more keys):
        # the kernels then have the long pieces to work on while the short
        # ones are still uploading, and the last download is a short one.
        pieces = [(b,) + p for b in range(B)
                  for p in prefill_row_chunks(Sq, Sk, causal, n_chunks)]
        self.pieces = sorted(pieces, key=lambda t: -(t[2] - t[1]) * t[3])
        self.ev_start = torch.cuda.Event()
        self.ev_kv = torch.cuda.Event()
        self.ev_q = [torch.cuda.Event() for _ in self.pieces]
        self.ev_o = [torch.cuda.Event() for _ in self.pieces]
        self.ev_done = torch.cuda.Event()

    def __call__(self, q_h, k_h, v_h, out_h, scale, stream=None):
        caller = torch.cuda.current_stream() if stream is None else stream
        for t, n, shp in ((q_h, "q", self.q.shape), (k_h, "k", self.k.shape),
                          (v_h, "v", self.v.shape), (out_h, "out", self.o.shape)):
            if tuple(t.shape) != tuple(shp) or t.dtype != self.dtype or t.is_cuda:
                raise ValueError(f"{n}: expected a host tensor {tuple(shp)} {self.dtype}")
            if not t.is_pinned() or not t.is_contiguous():
                raise ValueError(f"{n} must be contiguous pinned host memory")
        self.ev_start.record(caller)
        for s in (self.up, self.comp, self.down):
            s.wait_event(self.ev_start)
        # K and V first, then Q piece by piece.
        with torch.cuda.stream(self.up):
            self.k.copy_(k_h, non_blocking=True)
            self.v.copy_(v_h, non_blocking=True)
            self.ev_kv.record(self.up)
            for (b, s0, s1, _), ev in zip(self.pieces, self.ev_q):
                self.q[b, s0:s1].copy_(q_h[b, s0:s1], non_blocking=True)
                ev.record(self.up)
        # One prefill per piece, each as soon as its Q rows have landed.
        self.comp.wait_event(self.ev_kv)
        row_q, row_k = self.Hq * self.D * self.q.element_size(), \
            self.Hkv * self.D * self.k.element_size()
        code, sh = _dtype_code(self.q), self.comp.cuda_stream
        for (b, s0, s1, sk), ev_q, ev_o in zip(self.pieces, self.ev_q, self.ev_o):
            self.comp.wait_event(ev_q)
            qo_off = (b * self.Sq + s0) * row_q
            kv_off = b * self.Sk * row_k
            st = fa_prefill_fwd(self.q.data_ptr() + qo_off, self.k.data_ptr() + kv_off,
                                self.v.data_ptr() + kv_off, self.o.data_ptr() + qo_off, 1,
                                self.Hq, self.Hkv, s1 - s0, sk, self.D, float(scale),
                                int(self.causal), code, sh)
            if st != FA_OK:
                raise FAError(st, "fa_prefill_fwd")
            ev_o.record(self.comp)
        # O back piece by piece.
        with torch.cuda.stream(self.down):
            for (b, s0, s1, _), ev in zip(self.pieces, self.ev_o):
                self.down.wait_event(ev)
                out_h[b, s0:s1].copy_(self.o[b, s0:s1], non_blocking=True)
            self.ev_done.record(self.down)
        caller.wait_event(self.ev_done)
        return out_h
