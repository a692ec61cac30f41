"""A prefill whose Q and O hold 2^31 elements each (4 GiB of bf16): row
offsets past the int32 range.

Shape: B1 Hq64 Hkv1, Sq 262144, Sk 4096, D 128, bf16, not causal.  Q is zero
except for a seeded sample of rows (b, h, i) that includes the first and last
rows and heads; K and V are i.i.d. N(0, 1).  With one kv head and no mask, row
(b, h, i) of O depends only on its own query row and on K, V: the oracle
computes the sampled rows as a batch of independent rows ([1, n, 1, D]), and
every zero query row must equal the mean of V (uniform scores).  A row written
to the wrong place, or not written, fails one of the two checks; every element
of O must be finite.
"""
import math

import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


def test_prefill_rows_past_2_31_elements(fa):
    B, Hq, Hkv, Sq, Sk, D = 1, 64, 1, 1 << 18, 4096, 128
    assert B * Sq * Hq * D == 1 << 31
    dev = torch.device("cuda", 0)
    free, _ = torch.cuda.mem_get_info(dev)
    if free < 12 * (1 << 30):
        pytest.skip("needs about 11 GiB of free device memory")
    scale = 1 / math.sqrt(D)
    rows = fa_inputs.sample_rows(B, Hq, Hkv, Sq, n=256, seed=3)
    rows = torch.unique(rows, dim=0)
    q_rows, k, v = fa_inputs.sparse_q_prefill_inputs(rows, Hkv, Sk, D, B=B, seed=3)
    q = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16, device=dev)
    r = rows.to(dev)
    q[r[:, 0], r[:, 2], r[:, 1], :] = q_rows.to(dev)
    out = fa.prefill(q, k.to(dev), v.to(dev), scale, False)
    torch.cuda.synchronize()
    assert fa.fa_device_error()[0] == fa.FA_OK
    assert torch.isfinite(out).all().item()

    got = out[r[:, 0], r[:, 2], r[:, 1], :].float().cpu().numpy()
    ref = oracle.attention(q_rows.reshape(1, -1, 1, D), k, v, scale, False).reshape(-1, D)
    compare(got, ref)

    # Zero query rows, last ones included: uniform scores give the mean of V.
    zrows = torch.tensor([[0, 1, Sq - 1], [0, Hq - 2, Sq - 2], [0, Hq // 2 + 1, Sq // 2 + 7]])
    sampled = {tuple(x) for x in rows.tolist()}
    zrows = torch.stack([z for z in zrows if tuple(z.tolist()) not in sampled])
    zr = zrows.to(dev)
    gz = out[zr[:, 0], zr[:, 2], zr[:, 1], :].float().cpu().numpy()
    zero_q = torch.zeros(1, len(zrows), 1, D, dtype=torch.bfloat16)
    compare(gz, oracle.attention(zero_q, k, v, scale, False).reshape(-1, D))
