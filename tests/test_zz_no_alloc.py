"""fa_decode_fwd_noalloc: the decode entry point for callers that cannot
allocate device memory while they run (memory reserved once at start-up,
allocator locks held, runtimes that forbid allocation after initialisation).
Its split partials live in a fixed array inside the library instead of memory
from cudaMallocAsync.  Its output must match fa_decode_fwd's on the same inputs,
over two calls in a row that share that array.

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import pytest
import torch

import fa_inputs
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


def test_noalloc_decode_matches_allocating_decode_on_two_calls_in_a_row(fa):
    dev = torch.device("cuda", 0)
    shape = fa_inputs.DECODE_1TOK
    stream = torch.cuda.current_stream(dev).cuda_stream
    # Two different requests: the seeded valid length and a longer one, so a
    # call reading the previous call's partials would show.
    runs = [_upload(fa_inputs.decode_inputs_for(shape, seed=0), dev),
            _upload(fa_inputs.decode_inputs_for(shape, seed=7, L=50001), dev)]
    refs = [torch.empty_like(r[0]) for r in runs]
    outs = [torch.empty_like(r[0]) for r in runs]
    for t, ref in zip(runs, refs):
        assert _call(fa.fa_decode_fwd, t, shape, ref, stream) == fa.FA_OK
    torch.cuda.synchronize()
    for t, out in zip(runs, outs):  # two no-allocation calls back to back
        assert _call(fa.fa_decode_fwd_noalloc, t, shape, out, stream) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_error()[0] == fa.FA_OK
    for out, ref in zip(outs, refs):
        compare(out.float().cpu().numpy(), ref.float().cpu().numpy())


def test_noalloc_decode_rejects_requests_larger_than_its_scratch(fa):
    dev = torch.device("cuda", 0)
    q = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    vl = torch.zeros(1, dtype=torch.int32, device=dev)
    # 60000 sequences x 64 heads of D=128 partials need far more than 4 MiB.
    st = fa.fa_decode_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), vl.data_ptr(),
                                  q.data_ptr(), 60000, 64, 8, 4096, 128, 0.1, 0)
    assert st == fa.FA_ERR_TOO_LARGE
    assert "FA_ERR_TOO_LARGE" in fa.fa_status_string(st)
