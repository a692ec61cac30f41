"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds the workload shapes and the random-number recipe only: it
does no attention arithmetic.  Both the CUDA path and the fp64 oracle consume
the tensors it returns, so the two sides see identical bits.

Recipe: ``torch.Generator().manual_seed(seed)``; every tensor is drawn as
float32 ``randn`` (i.i.d. N(0, 1)) and rounded to the storage dtype.  The
draw order is fixed (decode: L, q, k-cache, v-cache; prefill: q, k, v).
"""
import itertools
import math
from dataclasses import dataclass, field

import torch

BF16_QNAN_BITS = 0x7FC0  # bf16 quiet NaN used to poison unused cache capacity


@dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    dtype: torch.dtype
    scale: float

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*Hq*Sq*Sk*D (two matmuls of 2*Sq*Sk*D each per
        head), halved when causal (the 2*B*Hq*Sq*Sk*D causal convention)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    Hq: int
    Hkv: int
    cap: int
    D: int
    scale: float
    dtype: torch.dtype = field(default=torch.bfloat16)


# The five workloads: four prefill shapes and one single-token decode.
TINY_CAUSAL_GQA = PrefillShape("tiny_causal_gqa_prefill_b1_hq2_hkv1_s128_d64_bf16",
                               1, 2, 1, 128, 128, 64, True, torch.bfloat16, 1.0 / math.sqrt(64))
RAGGED_NONCAUSAL = PrefillShape("ragged_noncausal_prefill_b2_h8_sq1000_sk1536_d64_fp16",
                                2, 8, 8, 1000, 1536, 64, False, torch.float16, 1.0 / 8.0)
MHA_CAUSAL = PrefillShape("mha_causal_prefill_b4_h16_s4096_d128_bf16",
                          4, 16, 16, 4096, 4096, 128, True, torch.bfloat16, 1.0 / math.sqrt(128))
GQA_CAUSAL_8K = PrefillShape("gqa_causal_prefill_b1_hq128_hkv8_s8192_d128_bf16",
                             1, 128, 8, 8192, 8192, 128, True, torch.bfloat16, 1.0 / math.sqrt(128))
DECODE_1TOK = DecodeShape("single_token_decode_b1_hq8_hkv2_d128_cap65536_bf16",
                          1, 8, 2, 65536, 128, 1.0 / math.sqrt(128))

PREFILL_SHAPES = [TINY_CAUSAL_GQA, RAGGED_NONCAUSAL, MHA_CAUSAL, GQA_CAUSAL_8K]


def _randn(g: torch.Generator, shape, dtype) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dtype=torch.bfloat16, seed=0):
    """q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] on the CPU, i.i.d. N(0,1) rounded to dtype."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (B, Sq, Hq, D), dtype)
    k = _randn(g, (B, Sk, Hkv, D), dtype)
    v = _randn(g, (B, Sk, Hkv, D), dtype)
    return q, k, v


def sparse_q_prefill_inputs(rows, Hkv, Sk, D, B=1, dtype=torch.bfloat16, seed=0):
    """For a query tensor too large to draw on the host: only the listed query
    rows get values, every other row of q is left zero by the caller.

    rows: int64 [n, 3] of (b, h, i).  Returns q_rows [n, D] (the rows' values,
    in the order of ``rows``) and k/v [B, Sk, Hkv, D], i.i.d. N(0, 1) rounded
    to dtype, drawn in that order from the seed."""
    g = torch.Generator().manual_seed(seed)
    q_rows = _randn(g, (len(rows), D), dtype)
    k = _randn(g, (B, Sk, Hkv, D), dtype)
    v = _randn(g, (B, Sk, Hkv, D), dtype)
    return q_rows, k, v


def prefill_inputs_for(shape: PrefillShape, seed=0):
    return prefill_inputs(shape.B, shape.Hq, shape.Hkv, shape.Sq, shape.Sk, shape.D,
                          shape.dtype, seed)


def tile_gain_inputs(B, Hq, Hkv, Sq, Sk, D, dtype, gains, seed=0, tile=128):
    """prefill_inputs with the keys of key tile t (rows [t*tile, (t+1)*tile)
    of k) multiplied by gains[t] before rounding to dtype (tiles past the list
    keep gain 1; q and v are unchanged).

    A row's scores against tile t then spread gains[t] times wider, so a row
    that has seen only ordinary scores meets, in a later tile, scores larger
    by tens of units: the running max of an online softmax jumps there.  The
    draw order and the unscaled values are those of prefill_inputs."""
    g = torch.Generator().manual_seed(seed)
    q = _randn(g, (B, Sq, Hq, D), dtype)
    k32 = torch.randn(B, Sk, Hkv, D, generator=g, dtype=torch.float32)
    v = _randn(g, (B, Sk, Hkv, D), dtype)
    for t, gain in enumerate(gains):
        k32[:, t * tile:(t + 1) * tile] *= float(gain)
    return q, k32.to(dtype), v


def first_tile_overflow_inputs(B, Hq, Hkv, Sq, Sk, D, seed=0, tile=128):
    """bf16 inputs whose scores against key tile 0 are -2^112 * D in raw
    units for every row, while every later key scores of order 2^-14 * sqrt(D).

    q is 1 everywhere; the keys of tile 0 are -2^112 in every element (both
    exact in bf16); later keys are 2^-14 * N(0, 1); v is N(0, 1).  With a
    softmax scale near 2^12 / log2(e), the first tile's scaled scores leave
    the fp32 range (below -2^128) although the raw scores fit it, and the
    later tiles' scaled scores are of order one."""
    g = torch.Generator().manual_seed(seed)
    q = torch.ones(B, Sq, Hq, D, dtype=torch.float32).to(torch.bfloat16)
    k32 = torch.randn(B, Sk, Hkv, D, generator=g, dtype=torch.float32) * 2.0 ** -14
    k32[:, :tile] = -(2.0 ** 112)
    v = _randn(g, (B, Sk, Hkv, D), torch.bfloat16)
    return q, k32.to(torch.bfloat16), v


def draw_valid_length(cap: int, seed=0) -> int:
    """The seeded valid length in [1, cap] (the first draw of the decode recipe)."""
    g = torch.Generator().manual_seed(seed)
    return 1 + int(torch.randint(0, cap, (1,), generator=g).item())


def varlen_lengths(n=16, max_len=4096, seed=0):
    """Seeded sequence lengths in [1, max_len] for a packed (varlen) batch."""
    g = torch.Generator().manual_seed(seed)
    return [1 + int(x) for x in torch.randint(0, max_len, (n,), generator=g).tolist()]


def varlen_inputs(lens_q, lens_k, Hq, Hkv, D, dtype=torch.bfloat16, seed=0):
    """Packed q [sum lens_q, Hq, D], k/v [sum lens_k, Hkv, D] (seeded N(0,1) in
    dtype) and the int32 prefix sums cu_q, cu_k ([B+1], host tensors)."""
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lens_q), sum(lens_k)
    q = _randn(g, (tq, Hq, D), dtype)
    k = _randn(g, (tk, Hkv, D), dtype)
    v = _randn(g, (tk, Hkv, D), dtype)
    cu_q = torch.tensor([0] + list(itertools.accumulate(lens_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(lens_k)), dtype=torch.int32)
    return q, k, v, cu_q, cu_k


def decode_inputs(B, Hq, Hkv, cap, D, dtype=torch.bfloat16, seed=0, L=None,
                  poison_k=True, poison_v=True):
    """Single-token decode inputs on the CPU.

    Returns (q [B,1,Hq,D], kcache [B,cap,Hkv,D], vcache [B,cap,Hkv,D], L).
    L is drawn from the seed in [1, cap] unless given.  Entries at token
    positions >= L are overwritten with the bf16 quiet NaN 0x7FC0 (V always
    poisoned, K as well unless poison_k=False), as in the unused-capacity
    reproduction of rocm-libraries #13108's review.
    """
    g = torch.Generator().manual_seed(seed)
    L_seeded = 1 + int(torch.randint(0, max(cap, 1), (1,), generator=g).item())
    if L is None:
        L = L_seeded
    q = _randn(g, (B, 1, Hq, D), dtype)
    kc = _randn(g, (B, cap, Hkv, D), dtype)
    vc = _randn(g, (B, cap, Hkv, D), dtype)
    lo = max(0, min(int(L), cap))
    if lo < cap:
        nan = poison_value(dtype)
        if poison_k:
            kc[:, lo:] = nan
        if poison_v:
            vc[:, lo:] = nan
    return q, kc, vc, int(L)


def decode_inputs_for(shape: DecodeShape, seed=0, L=None):
    return decode_inputs(shape.B, shape.Hq, shape.Hkv, shape.cap, shape.D, shape.dtype,
                         seed, L)


def paged_decode_batch(lens, Sq, Hq, Hkv, D, page_size, seed=0, device="cuda", spare_pages=8):
    """A batch of sequences in a paged bf16 KV cache, drawn on ``device`` (the
    pages are large; torch's generator of that device, seeded).

    Sequence b holds lens[b] tokens (its Sq new ones included) in
    ceil(lens[b] / page_size) pages taken in a seeded random physical order;
    every slot past a length and every spare page is the bf16 NaN 0x7FC0.
    Returns q [B, Sq, Hq, D], kpages, vpages [num_pages, page_size, Hkv, D],
    page_table int32 [B, max_pages] (unused entries 0) and seqlens int32 [B]."""
    B = len(lens)
    n_pages = [(L + page_size - 1) // page_size for L in lens]
    num_pages, max_pages = sum(n_pages) + spare_pages, max(1, max(n_pages))
    g_host = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g_host)
    table = torch.zeros(B, max_pages, dtype=torch.int32)
    used = 0
    for b, n in enumerate(n_pages):
        table[b, :n] = perm[used:used + n].to(torch.int32)
        used += n
    g = torch.Generator(device=device).manual_seed(seed)
    kp = torch.randn(num_pages, page_size, Hkv, D, generator=g, device=device).to(torch.bfloat16)
    vp = torch.randn(num_pages, page_size, Hkv, D, generator=g, device=device).to(torch.bfloat16)
    q = torch.randn(B, Sq, Hq, D, generator=g, device=device).to(torch.bfloat16)
    nan = poison_value(torch.bfloat16).to(device)
    for b, L in enumerate(lens):
        if L % page_size:
            last = int(table[b, n_pages[b] - 1])
            kp[last, L % page_size:] = nan
            vp[last, L % page_size:] = nan
    spare = perm[used:].to(device)
    kp[spare] = nan
    vp[spare] = nan
    return q, kp, vp, table.to(device), torch.tensor(lens, dtype=torch.int32, device=device)


def poison_value(dtype) -> torch.Tensor:
    """A scalar NaN of the given dtype; for bf16 exactly the bit pattern 0x7FC0."""
    if dtype == torch.bfloat16:
        return torch.tensor([BF16_QNAN_BITS], dtype=torch.int16).view(torch.bfloat16)[0]
    return torch.tensor(float("nan"), dtype=dtype)


def sample_rows(B, Hq, Hkv, Sq, n=4096, seed=0):
    """Seeded sample of query rows (b, h, i), int64 [m, 3], m <= n + specials.

    Always contains the rows i in {0, 1, 127, 128, 255, 256, Sq-1} (clipped to
    [0, Sq)) for the first and last query head of every GQA group and for
    b in {0, B-1}; the rest is uniform from the seed.
    """
    G = Hq // Hkv
    heads = sorted({h for kv in range(Hkv) for h in (kv * G, kv * G + G - 1)})
    rows_i = sorted({i for i in (0, 1, 127, 128, 255, 256, Sq - 1) if 0 <= i < Sq})
    bs = sorted({0, B - 1})
    special = [(b, h, i) for b in bs for h in heads for i in rows_i]
    g = torch.Generator().manual_seed(seed + 1)
    m = max(0, n - len(special))
    rb = torch.randint(0, B, (m,), generator=g)
    rh = torch.randint(0, Hq, (m,), generator=g)
    ri = torch.randint(0, Sq, (m,), generator=g)
    rand = list(zip(rb.tolist(), rh.tolist(), ri.tolist()))
    seen, out = set(), []
    for t in special + rand:
        if t not in seen:
            seen.add(t)
            out.append(t)
    return torch.tensor(out, dtype=torch.int64).reshape(-1, 3)
