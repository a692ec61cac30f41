"""Failure detection on the device without a fault: a pipeline wait that runs
past its time limit makes the kernel abort and report, and the context stays
usable.

fa_set_wait_limit_ns(1) is a watchdog limit: the dense prefill (through its
polling instantiation) and the decode check the clock at every probe of every
wait, so a wait that is not satisfied at once gives up.  The CTA leaves its
loops, waits (with the fixed 2 s teardown limit) for the loads and MMAs
already in flight, frees its tensor memory and sets the timeout bit and the
wait's site in the error word.  Nothing waits
without a bound, and no kernel is altered for the test.  The tests check that
a prefill, a 65536-token decode, a backward call (D = 128 and 64), a paged
decode and a packed-sequence prefill report FA_ERR_TIMEOUT with a site, then
restore the default limit and check that the next calls match the oracle.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


def test_wait_limit_aborts_report_timeout_and_the_next_calls_are_correct(fa):
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, S, D = 1, 8, 2, 1024, 128
    scale = 1 / math.sqrt(D)
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=5)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sd = fa_inputs.DECODE_1TOK
    dq, kc, vc, L = fa_inputs.decode_inputs_for(sd, seed=5, L=sd.cap)
    dqd, kcd, vcd = dq.to(dev), kc.to(dev), vc.to(dev)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    assert fa.fa_device_error(reset=1)[0] == fa.FA_OK

    try:
        assert fa.fa_set_wait_limit_ns(1) == fa.FA_OK
        fa.prefill(qd, kd, vd, scale, True)
        st, detail = fa.fa_device_error(reset=1)
        assert st == fa.FA_ERR_TIMEOUT, (st, hex(detail))
        assert detail & 1 and (detail >> 8) & 0xFF, hex(detail)  # prefill word: bit 0 + site
        fa.decode(dqd, kcd, vcd, vl, sd.scale)
        st, detail = fa.fa_device_error(reset=1)
        assert st == fa.FA_ERR_TIMEOUT, (st, hex(detail))
        assert (detail >> 16) & 1 and (detail >> 24) & 0xFF, hex(detail)  # decode word
    finally:
        assert fa.fa_set_wait_limit_ns(0) == fa.FA_OK

    out = fa.prefill(qd, kd, vd, scale, True)
    od = fa.decode(dqd, kcd, vcd, vl, sd.scale)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error(reset=1)
    assert st == fa.FA_OK, hex(detail)
    compare(out.float().cpu().numpy(), oracle.attention(q, k, v, scale, True))
    got = od.float().cpu().numpy().reshape(sd.B, sd.Hq, sd.D)
    compare(got, oracle.decode(dq, kc, vc, L, sd.scale))
    assert np.isfinite(got).all()


def test_watchdog_limit_that_no_wait_reaches_gives_correct_results(fa):
    """Under a watchdog limit (below 1 ms) the dense prefill runs its polling
    instantiation and the decode polls its waits.  A limit of 500 us is far
    above any wait of these calls, so nothing times out and the outputs must
    match the oracle, for the dense and the packed prefill and the decode."""
    dev = torch.device("cuda", 0)
    q, k, v = fa_inputs.prefill_inputs(2, 8, 2, 700, 900, 128, torch.bfloat16, seed=9)
    sd = fa_inputs.DECODE_1TOK
    dq, kc, vc, L = fa_inputs.decode_inputs_for(sd, seed=9)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    lens = [300, 0, 257, 129]  # 686 rows: within the 700 query and 900 key rows drawn
    qp, kp, vp = (t[0, :sum(lens)].contiguous() for t in (q, k, v))
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    assert fa.fa_device_error(reset=1)[0] == fa.FA_OK
    try:
        assert fa.fa_set_wait_limit_ns(500_000) == fa.FA_OK
        out = fa.prefill(q.to(dev), k.to(dev), v.to(dev), 0.088, True)
        outp = fa.prefill_varlen(qp.to(dev), kp.to(dev), vp.to(dev), cu.to(dev), cu.to(dev),
                                 max(lens), 0.088, True)
        od = fa.decode(dq.to(dev), kc.to(dev), vc.to(dev), vl, sd.scale)
        torch.cuda.synchronize()
        st, detail = fa.fa_device_error(reset=1)
    finally:
        assert fa.fa_set_wait_limit_ns(0) == fa.FA_OK
    assert st == fa.FA_OK, hex(detail)
    compare(out.float().cpu().numpy(), oracle.attention(q, k, v, 0.088, True))
    compare(outp.float().cpu().numpy(),
            oracle.attention_varlen(qp, kp, vp, cu.tolist(), cu.tolist(), 0.088, True))
    compare(od.float().cpu().numpy().reshape(sd.B, sd.Hq, sd.D),
            oracle.decode(dq, kc, vc, L, sd.scale))


@pytest.mark.parametrize("D", [128, 64])
def test_backward_wait_limit_aborts_report_timeout_and_the_next_call_is_correct(fa, D):
    """The backward kernels under a 1 ns limit.  Their waits keep suspending
    probes of about 4 us, so a wait gives up once it has lasted about two of
    them; the first key tile of a 2048-token causal GQA call takes hundreds
    of microseconds, so its epilogue wait (and others) give up.  Each aborted
    CTA tears down as the forward's do; then, at the default limit, a small
    backward call matches the oracle's gradients."""
    from tests.test_backward_gpu import grad_compare, run_backward
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, S = 1, 16, 1, 2048
    scale = 1 / math.sqrt(D)
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=21)
    dout = torch.randn(B, S, Hq, D, generator=torch.Generator().manual_seed(22)).to(torch.bfloat16)
    qd, kd, vd, dd = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    o, lse = fa.prefill(qd, kd, vd, scale, True, lse=True)
    torch.cuda.synchronize()
    assert fa.fa_device_error(reset=1)[0] == fa.FA_OK
    try:
        assert fa.fa_set_wait_limit_ns(1) == fa.FA_OK
        fa.backward(qd, kd, vd, o, dd, lse, scale, True)
        st, detail = fa.fa_device_error(reset=1)
        assert st == fa.FA_ERR_TIMEOUT, (st, hex(detail))
        assert detail & 1 and (detail >> 8) & 0xFF, hex(detail)  # backward word: bit 0 + site
    finally:
        assert fa.fa_set_wait_limit_ns(0) == fa.FA_OK

    q2, k2, v2 = fa_inputs.prefill_inputs(1, 4, 2, 300, 300, D, torch.bfloat16, seed=23)
    do2 = torch.randn(1, 300, 4, D, generator=torch.Generator().manual_seed(24)).to(torch.bfloat16)
    got = run_backward(fa, q2, k2, v2, do2, scale, True)
    ref = oracle.attention_bwd(q2, k2, v2, do2, scale, True)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        grad_compare(g, r, name)


def test_paged_decode_and_packed_prefill_wait_limit_abort_and_recover(fa):
    """A paged decode (balanced splits, row combine) and a packed-sequence
    prefill under a 1 ns limit report FA_ERR_TIMEOUT; then small calls of both
    at the default limit match the oracle.  The paged decode polls, so its
    first unsatisfied wait gives up.  The packed prefill suspends (about 4 us
    a probe); with items of up to 32 K/V tiles its producer waits for a whole
    item before loading the next item's Q, so that wait gives up."""
    from tests.test_paged_decode_gpu import paged_inputs, run_paged
    dev = torch.device("cuda", 0)
    lens = [16384, 8000, 12000, 3000, 16000, 9000, 15000, 11000]
    qd, kpd, vpd, tabd, sld = fa_inputs.paged_decode_batch(lens, 1, 8, 2, 128, 256, seed=3,
                                                           device=dev)
    vl = [4096, 3000, 2048]
    qv, kv, vv, cq, ck = fa_inputs.varlen_inputs(vl, vl, 16, 2, 128, seed=4)
    qv, kv, vv, cq, ck = (t.to(dev) for t in (qv, kv, vv, cq, ck))
    torch.cuda.synchronize()
    assert fa.fa_device_error(reset=1)[0] == fa.FA_OK
    try:
        assert fa.fa_set_wait_limit_ns(1) == fa.FA_OK
        fa.decode_paged(qd, kpd, vpd, tabd, sld, 1 / math.sqrt(128))
        st, detail = fa.fa_device_error(reset=1)
        assert st == fa.FA_ERR_TIMEOUT, (st, hex(detail))
        assert (detail >> 16) & 1 and (detail >> 24) & 0xFF, hex(detail)  # decode word
        fa.prefill_varlen(qv, kv, vv, cq, ck, max(vl), 1 / math.sqrt(128), True)
        st, detail = fa.fa_device_error(reset=1)
        assert st == fa.FA_ERR_TIMEOUT, (st, hex(detail))
        assert detail & 1 and (detail >> 8) & 0xFF, hex(detail)  # prefill word
    finally:
        assert fa.fa_set_wait_limit_ns(0) == fa.FA_OK

    q, kp, vp, table, L = paged_inputs(4, 8, 2, 128, 32, 40, [0, 1, 1000, 1280], seed=5)
    o, _ = run_paged(fa, q, kp, vp, table, L, 1 / math.sqrt(128))
    compare(o, oracle.decode_paged(q, kp, vp, table.tolist(), L.tolist(), 1 / math.sqrt(128)))
    small = [300, 0, 257, 129]
    qs, ks, vs, cqs, cks = fa_inputs.varlen_inputs(small, small, 8, 2, 128, seed=6)
    out = fa.prefill_varlen(qs.to(dev), ks.to(dev), vs.to(dev), cqs.to(dev), cks.to(dev),
                            max(small), 0.088, True)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error(reset=1)
    assert st == fa.FA_OK, hex(detail)
    compare(out.float().cpu().numpy(),
            oracle.attention_varlen(qs, ks, vs, cqs.tolist(), cks.tolist(), 0.088, True))
