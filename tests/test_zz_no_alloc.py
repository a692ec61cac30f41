"""fa_decode_fwd_noalloc: the decode entry point for callers that cannot
allocate device memory while they run -- a serving loop whose memory is
reserved once at start-up, code that runs while an allocator lock is held, a
runtime that forbids allocation after initialisation.  Its split partials live
in one fixed array inside the library instead of memory from cudaMallocAsync,
and every call on the device shares that array.

The test makes two calls in a row: first a long request (L = 50001), then the
seeded short one (L = 2733) with the same shape, so the short call's splits
sit on the partials the long call left behind.  Each output must be
bit-identical to fa_decode_fwd's on the same inputs (both run the same
kernels with the same split count) and match the fp64 oracle; the caches'
unused capacity holds NaN.

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


def _upload(inputs, dev):
    q, kc, vc, L = inputs
    return (q.to(dev), kc.to(dev), vc.to(dev),
            torch.tensor([L], dtype=torch.int32, device=dev))


def _call(entry, t, shape, out, stream):
    q, kc, vc, vl = t
    return entry(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), vl.data_ptr(), out.data_ptr(),
                 shape.B, shape.Hq, shape.Hkv, shape.cap, shape.D, shape.scale, stream)


def test_noalloc_decode_on_two_calls_in_a_row_matches_decode_and_oracle(fa):
    dev = torch.device("cuda", 0)
    shape = fa_inputs.DECODE_1TOK
    stream = torch.cuda.current_stream(dev).cuda_stream
    host = [fa_inputs.decode_inputs_for(shape, seed=7, L=50001),   # long request first
            fa_inputs.decode_inputs_for(shape, seed=0)]            # then the seeded L
    assert host[1][3] < host[0][3]
    runs = [_upload(h, dev) for h in host]
    refs = [torch.empty_like(r[0]) for r in runs]
    outs = [torch.empty_like(r[0]) for r in runs]
    for t, ref in zip(runs, refs):
        assert _call(fa.fa_decode_fwd, t, shape, ref, stream) == fa.FA_OK
    torch.cuda.synchronize()
    for t, out in zip(runs, outs):  # two no-allocation calls back to back
        assert _call(fa.fa_decode_fwd_noalloc, t, shape, out, stream) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_error()[0] == fa.FA_OK
    for (q, kc, vc, L), out, ref in zip(host, outs, refs):
        assert torch.equal(out, ref)
        got = out.float().cpu().numpy().reshape(shape.B, shape.Hq, shape.D)
        compare(got, oracle.decode(q, kc, vc, L, shape.scale))


def test_noalloc_decode_rejects_requests_larger_than_its_scratch(fa):
    dev = torch.device("cuda", 0)
    q = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    vl = torch.zeros(1, dtype=torch.int32, device=dev)
    # 60000 sequences x 64 heads of D=128 partials need far more than 4 MiB.
    st = fa.fa_decode_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), vl.data_ptr(),
                                  q.data_ptr(), 60000, 64, 8, 4096, 128, 0.1, 0)
    assert st == fa.FA_ERR_TOO_LARGE
    assert "FA_ERR_TOO_LARGE" in fa.fa_status_string(st)
