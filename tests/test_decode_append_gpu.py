"""A serving-style decode loop on the GPU: tokens are appended to a cache that
starts out entirely NaN, the valid length advances on the device, and a
decode follows every append.  Each step's output is compared with the fp64
oracle over the cache as it stood at that step.  Between two decodes runs a
torch kernel (the append and the length update), so every decode's launch
follows a kernel that is not its own; the rocm-libraries #13108 page
describes the same integration check (two sequences of 128 appends over
NaN-poisoned storage, "Validation and limits")."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


def test_contiguous_decode_after_each_append(fa):
    B, Hq, Hkv, cap, D, steps = 2, 8, 2, 256, 128, 128
    scale = 1 / math.sqrt(D)
    dev = torch.device("cuda", 0)
    nan = fa_inputs.poison_value(torch.bfloat16).to(dev)
    kc = torch.empty(B, cap, Hkv, D, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kc[:] = nan
    vc[:] = nan
    g = torch.Generator().manual_seed(11)
    new_k = torch.randn(steps, B, Hkv, D, generator=g).to(torch.bfloat16)
    new_v = torch.randn(steps, B, Hkv, D, generator=g).to(torch.bfloat16)
    qs = torch.randn(steps, B, 1, Hq, D, generator=g).to(torch.bfloat16)
    nk, nv, qd = new_k.to(dev), new_v.to(dev), qs.to(dev)
    vl = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for t in range(steps):
        kc[:, t] = nk[t]  # append token t (device copies on the current stream)
        vc[:, t] = nv[t]
        vl.fill_(t + 1)   # the valid length advances on the device
        outs.append(fa.decode(qd[t], kc, vc, vl, scale))
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, hex(detail)
    k_all, v_all = kc.cpu(), vc.cpu()
    for t in range(steps):
        got = outs[t].float().cpu().numpy().reshape(B, Hq, D)
        assert np.isfinite(got).all(), t
        compare(got, oracle.decode(qs[t], k_all, v_all, t + 1, scale))


def test_paged_decode_after_each_append_per_sequence_lengths(fa):
    """Sequence 0 appends a token every step, sequence 1 every other step; both
    live on 32-token pages in a shuffled physical order, spare pages NaN."""
    B, Hq, Hkv, D, page, steps = 2, 8, 2, 128, 32, 128
    scale = 1 / math.sqrt(D)
    dev = torch.device("cuda", 0)
    max_pages = steps // page
    num_pages = B * max_pages + 3
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(12))
    table = perm[:B * max_pages].reshape(B, max_pages).to(torch.int32)
    nan = fa_inputs.poison_value(torch.bfloat16).to(dev)
    kp = torch.empty(num_pages, page, Hkv, D, dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    kp[:] = nan
    vp[:] = nan
    g = torch.Generator().manual_seed(13)
    new_k = torch.randn(steps, B, Hkv, D, generator=g).to(torch.bfloat16)
    new_v = torch.randn(steps, B, Hkv, D, generator=g).to(torch.bfloat16)
    qs = torch.randn(steps, B, 1, Hq, D, generator=g).to(torch.bfloat16)
    nk, nv, qd, tabd = new_k.to(dev), new_v.to(dev), qs.to(dev), table.to(dev)
    sl = torch.zeros(B, dtype=torch.int32, device=dev)
    lens = [0, 0]
    outs, seen = [], []
    for t in range(steps):
        for b in range(B):
            if b == 0 or t % 2 == 0:  # sequence 1 appends every other step
                pos = lens[b]
                pid = int(table[b, pos // page])
                kp[pid, pos % page] = nk[t, b]
                vp[pid, pos % page] = nv[t, b]
                lens[b] += 1
        sl.copy_(torch.tensor(lens, dtype=torch.int32), non_blocking=False)
        outs.append(fa.decode_paged(qd[t], kp, vp, tabd, sl, scale))
        seen.append(list(lens))
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, hex(detail)
    k_all, v_all = kp.cpu(), vp.cpu()
    for t in range(steps):
        got = outs[t].float().cpu().numpy()
        assert np.isfinite(got).all(), t
        # Tokens appended after step t are NaN-free data the step did not see;
        # the oracle reads only each sequence's first seen[t][b] tokens.
        compare(got, oracle.decode_paged(qs[t], k_all, v_all, table.tolist(), seen[t], scale))
