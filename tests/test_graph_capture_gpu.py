"""Prefill, decode and backward recorded in a CUDA graph and replayed.

The calls allocate nothing on the host's behalf that could go stale under a
graph: decode and backward scratch is stream-ordered (allocation nodes in the
graph), and the dense prefill's work counter is either the stream's own slot
(zero between launches, because the last CTA of every launch zeroes it) or,
for a capturing stream that has no slot yet, a captured allocation and
memset.  Every replay must give the oracle's result.
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

    def step():
        out_p = fa.prefill(qd, kd, vd, 0.1, True)
        out_d = fa.decode(dqd, kcd, vcd, vl, scale_d)
        o, lse = fa.prefill(bqd, bkd, bvd, 0.125, True, lse=True)
        grads = fa.backward(bqd, bkd, bvd, o, bdod, lse, 0.125, True)
        return out_p, out_d, grads

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out_p, out_d, grads = step()
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        compare(out_p.float().cpu().numpy(), ref_p)
        compare(out_d.float().cpu().numpy().reshape(1, 8, 128), ref_d)
        for g, r in zip(grads, ref_g):
            g = g.float().cpu().numpy().astype(np.float64)
            assert np.isfinite(g).all()
            assert np.linalg.norm(g - r) / np.linalg.norm(r) <= 1e-2
    assert fa.fa_device_error()[0] == fa.FA_OK
