"""Batched single-token decode over a paged KV cache on the GPU
(fa_decode_paged_fwd) against the fp64 oracle: each sequence's pages are
gathered through its page table and decoded over its own valid length
(rocm-libraries #13108 defers batched shapes and non-contiguous KV storage;
its review finding on NaN in unused capacity applies to every unused slot)."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare
from tests.test_lse_gpu import lse_compare

pytestmark = pytest.mark.gpu


def paged_inputs(B, Hq, Hkv, D, page_size, max_pages, lens, seed, spare_pages=5):
    """Random pages in a shuffled physical order; every slot not holding a
    valid token (pages past a length, slots past it, spare pages) is NaN."""
    g = torch.Generator().manual_seed(seed)
    num_pages = B * max_pages + spare_pages
    nan = fa_inputs.poison_value(torch.bfloat16)
    kp = torch.full((num_pages, page_size, Hkv, D), float("nan")).to(torch.bfloat16)
    vp = kp.clone()
    kp[:] = nan
    vp[:] = nan
    perm = torch.randperm(num_pages, generator=g)
    table = perm[:B * max_pages].reshape(B, max_pages).to(torch.int32)
    for b in range(B):
        for t0 in range(0, min(lens[b], max_pages * page_size), page_size):
            n = min(page_size, lens[b] - t0)
            pid = int(table[b, t0 // page_size])
            kp[pid, :n] = torch.randn(n, Hkv, D, generator=g).to(torch.bfloat16)
            vp[pid, :n] = torch.randn(n, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(B, 1, Hq, D, generator=g).to(torch.bfloat16)
    return q, kp, vp, table, torch.tensor(lens, dtype=torch.int32)


def run_paged(fa, q, kp, vp, table, lens, scale, lse=True):
    dev = torch.device("cuda", 0)
    out, l = fa.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lens.to(dev),
                             scale, lse=lse)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    return out.float().cpu().numpy().reshape(q.shape), l.cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,D,page_size,max_pages,lens", [
    (1, 8, 2, 128, 64, 1024, [2733]),                 # the single-token workload, paged
    (4, 8, 2, 128, 32, 40, [0, 1, 1000, 1280]),       # per-sequence lengths, page edge
    (3, 16, 4, 64, 128, 20, [129, 2560, 777]),
    (2, 32, 2, 128, 256, 8, [2048, 300]),             # two 16-head blocks per kv head
])
def test_paged_decode_against_oracle(fa, B, Hq, Hkv, D, page_size, max_pages, lens):
    q, kp, vp, table, L = paged_inputs(B, Hq, Hkv, D, page_size, max_pages, lens, seed=B + D)
    scale = 1 / math.sqrt(D)
    o, l = run_paged(fa, q, kp, vp, table, L, scale)
    ref, ref_l = oracle.decode_paged(q, kp, vp, table.tolist(), L.tolist(), scale,
                                     return_lse=True)
    compare(o, ref)
    lse_compare(l, ref_l)


def test_paged_with_one_page_per_sequence_matches_contiguous_decode(fa):
    """page_size = cap, page_table[b] = b: the paged path reads the same tiles
    as fa_decode_fwd.  The two merge their splits in a different order (the
    paged rows online, one warp per row), so the outputs agree to the last
    rounding: within 2 bf16 ulps of the largest output, and both match the
    oracle.  A tile read from the wrong place moves an output by O(1)."""
    B, Hq, Hkv, cap, D = 2, 8, 2, 4096, 128
    q, kc, vc, L = fa_inputs.decode_inputs(B, Hq, Hkv, cap, D, seed=31, L=3000)
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), kc.to(dev), vc.to(dev)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    ref = fa.decode(qd, kd, vd, vl, 0.088)
    table = torch.arange(B, dtype=torch.int32, device=dev).reshape(B, 1)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    got = fa.decode_paged(qd, kd, vd, table, lens, 0.088)
    torch.cuda.synchronize()
    g, r = got.float().cpu(), ref.float().cpu()
    assert (g - r).abs().max().item() <= 2 * 2.0 ** -8 * r.abs().max().item()
    want = oracle.decode(q, kc, vc, L, 0.088)
    compare(g.numpy().reshape(want.shape), want)


def test_paged_bad_page_id_is_masked_and_reported(fa):
    """A page id outside [0, num_pages) is never read: its tokens are masked
    (the result equals decoding without that page) and the bounds bit of the
    device error word is set."""
    B, Hq, Hkv, D, ps, P = 1, 8, 2, 128, 64, 4
    q, kp, vp, table, L = paged_inputs(B, Hq, Hkv, D, ps, P, [4 * ps], seed=41)
    bad = table.clone()
    bad[0, 2] = 10_000
    o, _ = None, None
    dev = torch.device("cuda", 0)
    out = fa.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), bad.to(dev), L.to(dev), 0.088)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_ERR_BOUNDS and (detail >> 16) & 2   # decode word, bounds bit
    # reference: the same sequence without page 2's tokens (their keys masked)
    kc = kp[table[0].long()].reshape(1, P * ps, Hkv, D)
    vc = vp[table[0].long()].reshape(1, P * ps, Hkv, D)
    keep = torch.cat([kc[:, :2 * ps], kc[:, 3 * ps:]], dim=1)
    keepv = torch.cat([vc[:, :2 * ps], vc[:, 3 * ps:]], dim=1)
    ref = oracle.decode(q, keep, keepv, 3 * ps, 0.088)
    compare(out.float().cpu().numpy().reshape(1, Hq, D), ref)


@pytest.mark.parametrize("B,Sq,Hq,Hkv,D,page_size,max_pages,lens", [
    (2, 4, 8, 2, 128, 64, 16, [700, 3]),        # 4 tokens x 4 heads = 16 MMA rows; L < Sq
    (3, 2, 32, 4, 64, 32, 30, [1, 960, 513]),   # 2 x 8 rows per kv head
    (1, 5, 8, 1, 128, 128, 8, [1000]),          # 5 x 8 = 40 rows: three 16-row blocks
    (2, 2, 8, 2, 128, 64, 16, [500, 64]),       # 2 x 4 = 8 rows: one 8-row block
])
def test_paged_decode_several_new_tokens(fa, B, Sq, Hq, Hkv, D, page_size, max_pages, lens):
    """Sq new tokens per sequence (speculative decoding): bottom-right causal
    among the new tokens, each row with its own visible length."""
    q1, kp, vp, table, L = paged_inputs(B, Hq, Hkv, D, page_size, max_pages, lens, seed=Sq + D)
    g = torch.Generator().manual_seed(Sq)
    q = torch.randn(B, Sq, Hq, D, generator=g).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    o, l = run_paged(fa, q, kp, vp, table, L, scale)
    ref, ref_l = oracle.decode_paged(q, kp, vp, table.tolist(), L.tolist(), scale,
                                     return_lse=True)
    compare(o, ref)
    lse_compare(l, ref_l)


@pytest.mark.parametrize("B,Hq,Hkv,D", [
    (75, 4, 2, 64),    # 150 (sequence, kv head) units: balanced splits, scan over 3 warps
    (76, 4, 2, 64),    # 152 units, as many as SMs on GB300: splits sized from the capacity
    (150, 4, 1, 128),  # the largest batch with balanced splits on 152 SMs: 5 warps of sequences
])
def test_paged_decode_large_ragged_batches(fa, B, Hq, Hkv, D):
    """Many sequences of different lengths (some empty) on 32-token pages:
    with fewer units than SMs the kernels size each sequence's splits from the
    lengths on the device; with more, from the capacity.  Both must match the
    oracle for every sequence, and every output must be finite."""
    g = torch.Generator().manual_seed(B + Hkv)
    lens = [0 if x < 40 else int(x) for x in torch.randint(0, 700, (B,), generator=g).tolist()]
    page_size, max_pages = 32, 22
    q, kp, vp, table, L = paged_inputs(B, Hq, Hkv, D, page_size, max_pages, lens, seed=B * 7,
                                       spare_pages=3)
    scale = 1 / math.sqrt(D)
    got, lse = run_paged(fa, q, kp, vp, table, L, scale)
    assert np.isfinite(got).all()
    want, want_lse = oracle.decode_paged(q, kp, vp, table.tolist(), L.tolist(), scale,
                                         return_lse=True)
    compare(got, want)
    lse_compare(lse, want_lse)
