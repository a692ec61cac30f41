"""Prefill (dense and packed), decode (contiguous and paged) and backward
recorded in a CUDA graph and replayed.

The calls allocate nothing on the host's behalf that could go stale under a
graph: decode and backward scratch is stream-ordered (allocation nodes in the
graph), and the dense prefill's work counter is either the stream's own slot
(zero between launches, because the last CTA of every launch zeroes it) or,
for a capturing stream that has no slot yet, a captured allocation and
memset.  The packed prefill's plan and counter, and the paged decode's
partials and unit map, are stream-ordered scratch too.  Every replay must give
the oracle's result.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


def test_replayed_graph_matches_oracle(fa):
    dev = torch.device("cuda", 0)
    # Prefill: causal GQA with a ragged 256-row tail.
    q, k, v = fa_inputs.prefill_inputs(1, 8, 2, 700, 700, 128, torch.bfloat16, 31)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ref_p = oracle.attention(q, k, v, 0.1, True)
    # Decode: NaN-poisoned tail past L.
    dq, kc, vc, L = fa_inputs.decode_inputs(1, 8, 2, 4096, 128, seed=7, L=3000)
    dqd, kcd, vcd = dq.to(dev), kc.to(dev), vc.to(dev)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    scale_d = 1 / math.sqrt(128)
    ref_d = oracle.decode(dq, kc, vc, L, scale_d)
    # Backward of a tiny causal prefill.
    bq, bk, bv = fa_inputs.prefill_inputs(1, 4, 2, 300, 300, 64, torch.bfloat16, 5)
    bdo = torch.randn(bq.shape, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    bqd, bkd, bvd, bdod = bq.to(dev), bk.to(dev), bv.to(dev), bdo.to(dev)
    ref_g = oracle.attention_bwd(bq, bk, bv, bdo, 0.125, True)
    # Packed prefill: whole and partial warps of rows (TMA and thread stores).
    lens = [300, 33, 256, 97]
    vq, vk, vv, cq, ck = fa_inputs.varlen_inputs(lens, lens, 8, 2, 128, seed=8)
    vqd, vkd, vvd, cqd, ckd = (t.to(dev) for t in (vq, vk, vv, cq, ck))
    ref_v = oracle.attention_varlen(vq, vk, vv, cq.tolist(), ck.tolist(), 0.1, True)
    # Paged decode: ragged lengths over shuffled 32-token pages, NaN elsewhere.
    from tests.test_paged_decode_gpu import paged_inputs
    pq, kp, vp, table, plen = paged_inputs(4, 8, 2, 128, 32, 40, [0, 1, 1000, 1280], seed=9)
    pqd, kpd, vpd, tabd, plend = (t.to(dev) for t in (pq, kp, vp, table, plen))
    ref_pd = oracle.decode_paged(pq, kp, vp, table.tolist(), plen.tolist(), scale_d)

    def step():
        out_p = fa.prefill(qd, kd, vd, 0.1, True)
        out_d = fa.decode(dqd, kcd, vcd, vl, scale_d)
        o, lse = fa.prefill(bqd, bkd, bvd, 0.125, True, lse=True)
        grads = fa.backward(bqd, bkd, bvd, o, bdod, lse, 0.125, True)
        out_v = fa.prefill_varlen(vqd, vkd, vvd, cqd, ckd, max(lens), 0.1, True)
        out_pd = fa.decode_paged(pqd, kpd, vpd, tabd, plend, scale_d)
        return out_p, out_d, grads, out_v, out_pd

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out_p, out_d, grads, out_v, out_pd = step()
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        compare(out_p.float().cpu().numpy(), ref_p)
        compare(out_d.float().cpu().numpy().reshape(1, 8, 128), ref_d)
        for g, r in zip(grads, ref_g):
            g = g.float().cpu().numpy().astype(np.float64)
            assert np.isfinite(g).all()
            assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-2
        compare(out_v.float().cpu().numpy(), ref_v)
        compare(out_pd.float().cpu().numpy(), ref_pd)
    assert fa.fa_device_error()[0] == fa.FA_OK
