"""The seeded input recipe: deterministic, right shapes/dtypes, NaN tails."""
import torch

import fa_inputs


def test_prefill_inputs_deterministic():
    a = fa_inputs.prefill_inputs(1, 4, 2, 33, 40, 64, torch.bfloat16, seed=3)
    b = fa_inputs.prefill_inputs(1, 4, 2, 33, 40, 64, torch.bfloat16, seed=3)
    c = fa_inputs.prefill_inputs(1, 4, 2, 33, 40, 64, torch.bfloat16, seed=4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    q, k, v = a
    assert q.shape == (1, 33, 4, 64) and k.shape == (1, 40, 2, 64) and v.dtype == torch.bfloat16


def test_decode_inputs_poison_tail_and_seeded_length():
    q, kc, vc, L = fa_inputs.decode_inputs(1, 8, 2, 1000, 128, seed=0)
    assert L == fa_inputs.draw_valid_length(1000, seed=0)
    assert 1 <= L <= 1000
    assert torch.isfinite(kc[:, :L].float()).all() and torch.isfinite(vc[:, :L].float()).all()
    if L < 1000:
        assert (vc[:, L:].view(torch.int16) == fa_inputs.BF16_QNAN_BITS).all()
        assert (kc[:, L:].view(torch.int16) == fa_inputs.BF16_QNAN_BITS).all()


def test_headline_decode_length_in_range():
    L = fa_inputs.draw_valid_length(fa_inputs.DECODE_1TOK.cap, seed=0)
    assert 1 <= L <= 65536


def test_sample_rows_contains_specials():
    rows = fa_inputs.sample_rows(2, 16, 4, 4096, n=512, seed=0)
    s = {tuple(r) for r in rows.tolist()}
    for i in (0, 1, 127, 128, 255, 256, 4095):
        for h in (0, 3, 4, 7, 12, 15):
            for b in (0, 1):
                assert (b, h, i) in s
    assert len(s) == len(rows)


def test_flop_convention():
    s = fa_inputs.GQA_CAUSAL_8K
    assert s.flops == 2 * 1 * 128 * 8192 * 8192 * 128
    assert fa_inputs.RAGGED_NONCAUSAL.flops == 4 * 2 * 8 * 1000 * 1536 * 64


def test_paged_decode_batch_layout():
    """Valid tokens are finite and sit in their sequence's pages in order;
    every slot past a length and every spare page is the bf16 NaN 0x7FC0."""
    lens = [1, 33, 64, 100]
    q, kp, vp, table, sl = fa_inputs.paged_decode_batch(lens, 2, 8, 2, 64, 32, seed=0,
                                                        device="cpu")
    assert q.shape == (4, 2, 8, 64) and sl.tolist() == lens
    used = set()
    for b, L in enumerate(lens):
        for t in range(-(-L // 32) * 32):
            pid = int(table[b, t // 32])
            used.add(pid)
            finite = bool(torch.isfinite(kp[pid, t % 32].float()).all()) and \
                bool(torch.isfinite(vp[pid, t % 32].float()).all())
            assert finite == (t < L), (b, t)
    spare = [p for p in range(kp.shape[0]) if p not in used]
    assert len(spare) == 8
    for p in spare:
        assert bool((kp[p].view(torch.int16) == 0x7FC0).all())
        assert bool((vp[p].view(torch.int16) == 0x7FC0).all())
