"""The prefill softmax's lazy rescale, driven on the GPU and compared with the
fp64 oracle element by element.

The lazy rescale is the "lazy" lever of "Dense flash-attention prefill (gfx950 /
MI355X)", *Measured*.  Here each K/V tile after a row's first is exponentiated
against the row's running max without taking the tile's own max; only when
the tile's row sum of P passes 2^60 (bf16 P) or 2^15 (fp16 P), or the row had
no finite score before, does the slow path find the new max, rescale O (in
tensor memory) and the row sum by 2^(m_old - m_new), and recompute P.

Seeded N(0, 1) inputs never reach that path.  The inputs here do:
``fa_inputs.tile_gain_inputs`` multiplies the keys of chosen key tiles, so a
row's scores jump by tens of units in a later tile.  With gains (1, 1, g2, 1,
g4) the first jump (tile 2) sits near the threshold, so some rows of a warp
rescale and their neighbours do not; the second (tile 4) is larger, so rows
rescale a second time, some with P past the fp32 range before the rescale.
Under causal masking, query tile t meets the jump of key tile t inside its
diagonal (masked) tile.  A plausible mistake in the slow path (O or l not
rescaled, the factor inverted, P left against the old max) moves O by far
more than the bar: the old contributions are 2^60 (bf16) or 2^15 (fp16)
times too large, or P overflows.

The library's rescale counter (fa_prefill_rescale_count) shows the path ran;
on N(0, 1) inputs and on jumps below the threshold it stays at zero.

Bar: softmax weights this peaked put most of a row's weight on a few keys, so
the arithmetic bar of tests/parity.py applies (one rounding of P, relative
2^-8 for bf16 and 2^-11 for fp16, times max|V|, plus half an ulp of O),
together with relative L2 <= 5e-3; lse within 1e-3 where finite.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare, rounding_bound

pytestmark = pytest.mark.gpu

# Gains per key tile.  bf16: the tile-2 jump, 16 x N(0,1) scores (max ~40
# natural-log units, ~58 in log2 units over an ordinary row max), straddles
# the 2^60 threshold; tile 4 (40x) passes it, and fp32 for some rows.  fp16:
# the same at its 2^15 threshold.
GAINS = {torch.bfloat16: (1, 1, 16, 1, 40), torch.float16: (1, 1, 5, 1, 12)}
BITS = {torch.bfloat16: 8, torch.float16: 11}


def rescales(fa, reset=1):
    st, n = fa.fa_prefill_rescale_count(reset)
    assert st == fa.FA_OK
    return n


def run_and_compare(fa, q, k, v, scale, causal, dtype, bar=None):
    dev = torch.device("cuda", 0)
    out, lse = fa.prefill(q.to(dev), k.to(dev), v.to(dev), scale, causal, lse=True)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    ref, ref_lse = oracle.attention(q, k, v, scale, causal, return_lse=True)
    got = out.float().cpu().numpy()
    if bar is None:
        bar = rounding_bound(ref, v.abs().max().item(), BITS[dtype])
    compare(got, ref, max_abs=bar)
    g_lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(g_lse), fin)
    assert np.abs(g_lse[fin] - ref_lse[fin]).max() <= 1e-3
    return got


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_jumps_in_later_tiles_rescale_and_match_the_oracle(fa, dtype, D, causal):
    q, k, v = fa_inputs.tile_gain_inputs(1, 4, 2, 700, 700, D, dtype, GAINS[dtype], seed=D)
    rescales(fa)
    run_and_compare(fa, q, k, v, 1 / math.sqrt(D), causal, dtype)
    assert rescales(fa) > 0, "the lazy-rescale path did not run"


@pytest.mark.parametrize("Sq,Sk", [(600, 900), (900, 600)])
def test_ragged_causal_jumps(fa, Sq, Sk):
    """Bottom-right causal with Sq != Sk: rows that see few keys (or none,
    for Sq > Sk) share warps with rows that rescale, so lanes with nothing to
    rescale run the warp's slow path with factor 1."""
    dtype = torch.bfloat16
    q, k, v = fa_inputs.tile_gain_inputs(2, 4, 1, Sq, Sk, 128, dtype, GAINS[dtype], seed=Sq)
    rescales(fa)
    run_and_compare(fa, q, k, v, 1 / math.sqrt(128), True, dtype)
    assert rescales(fa) > 0


def test_first_tile_scores_overflowing_to_minus_inf(fa):
    """The slow path's other trigger: a row whose running max is -inf after
    its first tile although a later tile has finite scores.  With a prefix of
    visible keys (causal or not) a row that sees any key sees key 0, so this
    happens only when every scaled score of the first tile leaves the fp32
    range: raw scores -2^118 (D = 64) times scale * log2(e) = 2^12.  Those
    keys carry weight exp(-10^38) = 0 in the oracle; the kernel must drop
    them, restart the row from the later tiles, and match."""
    D = 64
    q, k, v = fa_inputs.first_tile_overflow_inputs(1, 2, 1, 300, 500, D)
    scale = 2.0 ** 12 / math.log2(math.e)
    rescales(fa)
    run_and_compare(fa, q, k, v, scale, False, torch.bfloat16)
    assert rescales(fa) > 0


def test_ordinary_and_below_threshold_inputs_do_not_rescale(fa):
    """N(0, 1) inputs, and jumps that stay below the threshold (bf16 gain 6:
    scores up to ~25 log2 units above the running max, so P up to ~2^25 is
    kept unrescaled), leave the counter at zero and still match the oracle."""
    rescales(fa)
    q, k, v = fa_inputs.prefill_inputs(1, 4, 2, 700, 700, 128, torch.bfloat16, seed=3)
    run_and_compare(fa, q, k, v, 1 / math.sqrt(128), True, torch.bfloat16)
    assert rescales(fa) == 0
    q, k, v = fa_inputs.tile_gain_inputs(1, 4, 2, 700, 700, 128, torch.bfloat16, (1, 1, 6),
                                         seed=4)
    run_and_compare(fa, q, k, v, 1 / math.sqrt(128), False, torch.bfloat16)
    assert rescales(fa) == 0
