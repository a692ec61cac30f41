"""Pins for the fp64 oracle: things the pages and the mathematics fix, chosen so
that a plausible mistake in the oracle (a dropped term, a wrong sign or index,
a transposed operand, a wrong mask edge, a wrong GQA map) fails one of them.

Sources for what the oracle computes: tessera #90 (flash_attn forward commit
note: scale*Q@K^T, causal/ragged mask, softmax, P@V); "Dense flash-attention
prefill (gfx950 / MI355X)" (MHA or GQA, causal; parity checked against
torch.nn.functional.scaled_dot_product_attention in its Measured section);
rocm-libraries #13108 (decode over the first L tokens of a token-major cache;
the unused-capacity NaN reproduction).
"""
import math
import os

import numpy as np
import pytest
import torch

import fa_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f64(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# 1. Brute force on tiny shapes: whole-matrix numpy formulation
#    (S = scale*Q K^T over all (i, j) at once, additive -inf mask, softmax
#    along keys, P V), a different computation order from the oracle's
#    per-row loop.
# ---------------------------------------------------------------------------
def brute_force(q, k, v, scale, causal):
    q, k, v = f64(q), f64(k), f64(v)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    G = Hq // Hkv
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            Q = q[b, :, h, :]                       # [Sq, D]
            K = k[b, :, h // G, :]                  # [Sk, D]
            V = v[b, :, h // G, :]
            S = scale * (Q @ K.T)                   # [Sq, Sk]
            if causal:
                ii = np.arange(Sq)[:, None]
                jj = np.arange(Sk)[None, :]
                S = np.where(jj <= ii + (Sk - Sq), S, -np.inf)
            for i in range(Sq):
                row = S[i]
                if np.all(np.isneginf(row)):
                    continue                        # no visible key: 0
                e = np.exp(row - row.max())
                out[b, i, h] = (e / e.sum()) @ V
    return out


TINY = [
    # B, Hq, Hkv, Sq, Sk, D, causal, dtype, scale
    (1, 2, 1, 7, 7, 8, True, torch.bfloat16, 0.3),
    (2, 4, 2, 5, 11, 16, True, torch.bfloat16, 0.25),
    (2, 4, 4, 9, 4, 8, True, torch.float16, 0.5),     # Sq > Sk: fully masked rows
    (1, 3, 1, 6, 13, 4, False, torch.float16, 1.0),
    (2, 4, 2, 16, 16, 8, False, torch.bfloat16, 0.125),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt,scale", TINY)
def test_brute_force_tiny(B, Hq, Hkv, Sq, Sk, D, causal, dt, scale):
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=3)
    o = oracle.attention(q, k, v, scale, causal)
    ref = brute_force(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# 2. Library routine: torch fp64 scaled_dot_product_attention on the CPU (the
#    routine the gfx950 prefill README measures its parity against).  GQA via
#    repeat_interleave of K/V heads; bottom-right causal via an explicit mask.
# ---------------------------------------------------------------------------
def sdpa_ref(q, k, v, scale, causal):
    G = q.shape[2] // k.shape[2]
    qt = q.to(torch.float64).permute(0, 2, 1, 3)                        # [B,Hq,Sq,D]
    kt = k.to(torch.float64).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    vt = v.to(torch.float64).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    Sq, Sk = q.shape[1], k.shape[1]
    mask = None
    if causal:
        ii = torch.arange(Sq)[:, None]
        jj = torch.arange(Sk)[None, :]
        mask = jj <= ii + (Sk - Sq)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                         scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("shape", [fa_inputs.TINY_CAUSAL_GQA, fa_inputs.RAGGED_NONCAUSAL],
                         ids=lambda s: s.name)
def test_matches_torch_sdpa_fp64(shape):
    q, k, v = fa_inputs.prefill_inputs_for(shape, seed=0)
    o = oracle.attention(q, k, v, shape.scale, shape.causal)
    ref = sdpa_ref(q, k, v, shape.scale, shape.causal)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-11)


def test_matches_torch_sdpa_sq_lt_sk_causal():
    q, k, v = fa_inputs.prefill_inputs(2, 6, 3, 37, 70, 16, torch.bfloat16, seed=5)
    o = oracle.attention(q, k, v, 0.2, True)
    np.testing.assert_allclose(o, sdpa_ref(q, k, v, 0.2, True), rtol=0, atol=1e-11)


def test_sampled_rows_equal_full_output():
    q, k, v = fa_inputs.prefill_inputs(2, 4, 2, 33, 33, 16, torch.bfloat16, seed=9)
    full = oracle.attention(q, k, v, 0.25, True)
    rows = fa_inputs.sample_rows(2, 4, 2, 33, n=40, seed=1)
    part = oracle.attention(q, k, v, 0.25, True, rows=rows)
    r = rows.numpy()
    np.testing.assert_array_equal(part, full[r[:, 0], r[:, 2], r[:, 1]])


# ---------------------------------------------------------------------------
# 3. Softmax rows sum to one; masked keys get exactly zero weight.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
def test_probabilities_sum_to_one(causal):
    q, k, v = fa_inputs.prefill_inputs(1, 4, 2, 12, 20, 8, torch.bfloat16, seed=2)
    for h in range(4):
        for i in (0, 5, 11):
            p, o = oracle.probs(q, k, v, 0.4, causal, 0, h, i)
            assert abs(p.sum() - 1.0) < 1e-14
            assert np.all(p >= 0)
            if causal:
                last = i + (20 - 12)
                assert np.all(p[last + 1:] == 0.0) and p[last] > 0
            # O is the p-weighted sum of the head's V rows
            np.testing.assert_allclose(o, p @ f64(v)[0, :, h // 2, :], atol=1e-13)


# ---------------------------------------------------------------------------
# 4. Uniform scores (Q = 0): O row i is the mean of V over its visible keys.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
def test_zero_query_gives_mean_of_visible_values(causal):
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 10, 14, 8
    _, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=4)
    q = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16)
    o = oracle.attention(q, k, v, 0.7, causal)
    vv = f64(v)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                n = min(Sk, i + (Sk - Sq) + 1) if causal else Sk
                np.testing.assert_allclose(o[b, i, h], vv[b, :n, h // 2].mean(axis=0),
                                           atol=1e-14)


# ---------------------------------------------------------------------------
# 5. One visible key returns that key's V exactly: causal row 0 (Sq == Sk) and
#    decode with valid length 1.
# ---------------------------------------------------------------------------
def test_causal_row0_is_first_value_exactly():
    q, k, v = fa_inputs.prefill_inputs(2, 4, 2, 9, 9, 16, torch.bfloat16, seed=6)
    o = oracle.attention(q, k, v, 0.3, True)
    vv = f64(v)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(o[b, 0, h], vv[b, 0, h // 2])


def test_decode_valid_length_one_is_first_value_exactly():
    q, kc, vc, L = fa_inputs.decode_inputs(1, 8, 2, 16, 128, seed=1, L=1)
    o = oracle.decode(q, kc, vc, L, 1 / math.sqrt(128))
    vv = f64(vc)
    for h in range(8):
        assert np.array_equal(o[0, h], vv[0, 0, h // 4])


# ---------------------------------------------------------------------------
# 6. GQA equals MHA with K/V heads repeated G times (contiguous groups).
# ---------------------------------------------------------------------------
def test_gqa_equals_mha_with_repeated_kv():
    B, Hq, Hkv, Sq, Sk, D = 2, 8, 2, 11, 17, 16
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=8)
    G = Hq // Hkv
    o_gqa = oracle.attention(q, k, v, 0.25, True)
    o_mha = oracle.attention(q, k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2),
                             0.25, True)
    assert np.array_equal(o_gqa, o_mha)
    # and NOT the interleaved (h % Hkv) map: the two differ on this input
    o_wrong = oracle.attention(q, k.repeat(1, 1, G, 1), v.repeat(1, 1, G, 1), 0.25, True)
    assert np.max(np.abs(o_gqa - o_wrong)) > 1e-3


# ---------------------------------------------------------------------------
# 7. Unused cache capacity: NaN tails give the same output as zero tails, and
#    the worked example of rocm-libraries #13108's review (capacity 128, valid
#    length 1, V tail = bf16 0x7fc0 -> output equals the first V token).
# ---------------------------------------------------------------------------
def test_decode_nan_tail_equals_zero_tail():
    q, kc, vc, L = fa_inputs.decode_inputs(2, 8, 2, 300, 64, seed=3, L=123)
    assert torch.isnan(vc[:, L:].float()).all() and torch.isnan(kc[:, L:].float()).all()
    kz, vz = kc.clone(), vc.clone()
    kz[:, L:] = 0
    vz[:, L:] = 0
    a = oracle.decode(q, kc, vc, L, 0.125)
    b = oracle.decode(q, kz, vz, L, 0.125)
    assert np.isfinite(a).all()
    assert np.array_equal(a, b)


def read_fixture(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split(None, 1)
                kv[key] = val
    return kv


def test_golden_nan_tail_worked_example():
    fx = read_fixture("nan_tail_decode.txt")
    B, Hq, Hkv, D, cap = (int(fx[k]) for k in ("B", "Hq", "Hkv", "D", "cap"))
    L = int(fx["valid_length"])
    assert cap * Hkv * D == int(fx["v_buffer_elements"])
    q, kc, vc, _ = fa_inputs.decode_inputs(B, Hq, Hkv, cap, D, seed=0, L=L, poison_k=False)
    assert (vc[:, L:].view(torch.int16) == int(fx["v_tail_bits"], 16)).all()
    o = oracle.decode(q, kc, vc, L, 1 / math.sqrt(D))
    first_v = f64(vc)[0, 0]
    G = Hq // Hkv
    for h in range(Hq):
        ref = first_v[h // G]
        tol = float(fx["tolerance_abs"]) + float(fx["tolerance_rel"]) * np.abs(ref)
        assert np.all(np.abs(o[0, h] - ref) <= tol)
        assert np.array_equal(o[0, h], ref)  # one visible key: exact


# ---------------------------------------------------------------------------
# 8. Decode equals non-causal prefill with Sq=1 over the first L tokens; the
#    valid length is clamped to [0, cap].
# ---------------------------------------------------------------------------
def test_decode_equals_prefill_over_valid_prefix():
    q, kc, vc, L = fa_inputs.decode_inputs(2, 8, 2, 64, 32, seed=2, L=41)
    o_dec = oracle.decode(q, kc, vc, L, 0.2)
    o_pre = oracle.attention(q, kc[:, :L], vc[:, :L], 0.2, False)
    np.testing.assert_allclose(o_dec, o_pre[:, 0], rtol=0, atol=0)


def test_decode_clamps_valid_length():
    q, kc, vc, _ = fa_inputs.decode_inputs(1, 4, 1, 20, 16, seed=4, L=20)
    assert np.array_equal(oracle.decode(q, kc, vc, 0, 0.3), np.zeros((1, 4, 16)))
    assert np.array_equal(oracle.decode(q, kc, vc, -5, 0.3), np.zeros((1, 4, 16)))
    assert np.array_equal(oracle.decode(q, kc, vc, 25, 0.3), oracle.decode(q, kc, vc, 20, 0.3))
    # L = cap: every cached token is visible, i.e. non-causal prefill over the cache
    full = oracle.attention(q, kc, vc, 0.3, False)[:, 0]
    np.testing.assert_allclose(oracle.decode(q, kc, vc, 20, 0.3), full, rtol=0, atol=0)


# ---------------------------------------------------------------------------
# 9. Index and operand checks.
# ---------------------------------------------------------------------------
def test_dominant_key_selects_its_value_row():
    """A key aligned with the query and a large scale takes all the weight: the
    output must be that key's V row (catches K/V index mix-ups and a
    transposed Q K^T)."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 4, 6, 8
    _, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.float16, seed=12)
    q = torch.zeros(B, Sq, Hq, D, dtype=torch.float16)
    target = [3, 0, 5, 2]                       # key picked by row i
    k[0, :, 0, :] = 0
    for j in range(Sk):
        k[0, j, 0, j % D] = 1.0                 # key j = unit vector e_j
    for i, j in enumerate(target):
        q[0, i, :, j % D] = 1.0
    o = oracle.attention(q, k, v, 200.0, False)
    vv = f64(v)
    for i, j in enumerate(target):
        for h in range(Hq):
            np.testing.assert_allclose(o[0, i, h], vv[0, j, 0], atol=1e-12)


def test_causal_mask_edge_bottom_right():
    """Row i sees key i + (Sk - Sq) and not key i + (Sk - Sq) + 1."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 6, 10, 8
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=13)
    base = oracle.attention(q, k, v, 0.3, True)
    i = 2
    last = i + Sk - Sq
    v2 = v.clone()
    v2[0, last + 1] += 1.0
    o2 = oracle.attention(q, k, v2, 0.3, True)
    assert np.array_equal(o2[0, : i + 1], base[0, : i + 1])
    v3 = v.clone()
    v3[0, last] += 1.0
    o3 = oracle.attention(q, k, v3, 0.3, True)
    assert np.max(np.abs(o3[0, i] - base[0, i])) > 1e-6
    assert np.array_equal(o3[0, :i], base[0, :i])


def test_fully_masked_rows_are_zero():
    q, k, v = fa_inputs.prefill_inputs(1, 2, 1, 8, 3, 8, torch.bfloat16, seed=14)
    o = oracle.attention(q, k, v, 0.5, True)
    # Sq - Sk = 5 leading rows see no key (bottom-right alignment)
    assert np.array_equal(o[0, :5], np.zeros((5, 2, 8)))
    assert np.all(np.abs(o[0, 5:]) > 0)


def test_noncausal_key_permutation_invariance():
    q, k, v = fa_inputs.prefill_inputs(1, 2, 2, 5, 12, 8, torch.bfloat16, seed=15)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(0))
    a = oracle.attention(q, k, v, 0.4, False)
    b = oracle.attention(q, k[:, perm], v[:, perm], 0.4, False)
    np.testing.assert_allclose(a, b, atol=1e-14)


def test_scale_multiplies_scores():
    q, k, v = fa_inputs.prefill_inputs(1, 2, 1, 5, 5, 8, torch.float32, seed=16)
    a = oracle.attention(q * 2, k, v, 0.25, True)
    b = oracle.attention(q, k, v, 0.5, True)
    np.testing.assert_allclose(a, b, atol=1e-13)


def test_softmax_shift_invariance_against_closed_form_two_keys():
    """Two keys: O = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1."""
    q = torch.tensor([[[[1.0, 2.0]]]], dtype=torch.float64)            # [1,1,1,2]
    k = torch.tensor([[[[0.5, -1.0]], [[2.0, 0.25]]]], dtype=torch.float64)  # [1,2,1,2]
    v = torch.tensor([[[[3.0, -2.0]], [[-1.0, 4.0]]]], dtype=torch.float64)
    scale = 0.7
    s0 = scale * (1.0 * 0.5 + 2.0 * -1.0)
    s1 = scale * (1.0 * 2.0 + 2.0 * 0.25)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    ref = w0 * np.array([3.0, -2.0]) + (1 - w0) * np.array([-1.0, 4.0])
    o = oracle.attention(q, k, v, scale, False)
    np.testing.assert_allclose(o[0, 0, 0], ref, atol=1e-15)


@pytest.mark.parametrize("scale", [500.0, -500.0])
def test_scores_far_outside_exp_range_closed_form(scale):
    """Softmax is shift invariant, so scores of +-1000 (exp overflows or
    underflows in fp64) still have the closed form of the two-key case:
    w0 = 1 / (1 + exp(s1 - s0)).  Here |s1 - s0| = 2000, so all the weight
    goes to the larger score and O is that key's V row exactly."""
    q = torch.tensor([[[[1.0, 2.0]]]], dtype=torch.float64)
    k = torch.tensor([[[[0.5, -1.0]], [[2.0, 0.25]]]], dtype=torch.float64)
    v = torch.tensor([[[[3.0, -2.0]], [[-1.0, 4.0]]]], dtype=torch.float64)
    o = oracle.attention(q, k, v, scale, False)
    want = [-1.0, 4.0] if scale > 0 else [3.0, -2.0]   # s0 = -1.5*scale, s1 = 2.5*scale
    np.testing.assert_array_equal(o[0, 0, 0], want)
    # same shift on both keys (s0 = s1 = -1000 or +1000): the plain mean
    k_eq = torch.tensor([[[[2.0, 0.0]], [[0.0, 1.0]]]], dtype=torch.float64)
    o_eq = oracle.attention(q, k_eq, v, scale, False)
    np.testing.assert_array_equal(o_eq[0, 0, 0], [1.0, 1.0])


# ---------------------------------------------------------------------------
# 10. Log-sum-exp output: log sum_j exp(s_j) over the visible keys of a row.
# ---------------------------------------------------------------------------
def brute_force_lse(q, k, v, scale, causal):
    """[B, Hq, Sq]: numpy logaddexp.reduce over the explicit masked score
    matrix (a different formulation from the oracle's max + log(sum))."""
    q, k = f64(q), f64(k)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    G = Hq // Hkv
    out = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            S = scale * (q[b, :, h, :] @ k[b, :, h // G, :].T)
            for i in range(Sq):
                vis = np.arange(Sk) <= i + (Sk - Sq) if causal else np.ones(Sk, bool)
                if vis.any():
                    out[b, h, i] = np.logaddexp.reduce(S[i, vis])
    return out


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt,scale", TINY)
def test_lse_brute_force_tiny(B, Hq, Hkv, Sq, Sk, D, causal, dt, scale):
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=3)
    _, lse = oracle.attention(q, k, v, scale, causal, return_lse=True)
    ref = brute_force_lse(q, k, v, scale, causal)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(lse[fin], ref[fin], rtol=0, atol=1e-12)


def test_lse_matches_torch_logsumexp_ragged():
    shape = fa_inputs.RAGGED_NONCAUSAL
    q, k, v = fa_inputs.prefill_inputs_for(shape, seed=0)
    _, lse = oracle.attention(q, k, v, shape.scale, False, return_lse=True)
    G = shape.Hq // shape.Hkv
    qt = q.to(torch.float64).permute(0, 2, 1, 3)
    kt = k.to(torch.float64).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
    ref = torch.logsumexp(shape.scale * (qt @ kt.transpose(-1, -2)), dim=-1).numpy()
    np.testing.assert_allclose(lse, ref, rtol=0, atol=1e-11)


def test_lse_zero_query_is_log_of_visible_count():
    """All scores 0: lse = log(number of visible keys); -inf with none."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 9, 6, 8
    _, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=4)
    q = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16)
    _, lse = oracle.attention(q, k, v, 0.7, True, return_lse=True)
    for i in range(Sq):
        n = max(0, min(Sk, i + (Sk - Sq) + 1))
        want = math.log(n) if n else -math.inf
        for h in range(Hq):
            assert lse[0, h, i] == pytest.approx(want, abs=1e-15) if n else lse[0, h, i] == want


def test_lse_single_visible_key_is_that_score():
    """Causal row 0 (Sq = Sk) sees key 0 only: lse = scale * <q_0, k_0>."""
    q, k, v = fa_inputs.prefill_inputs(1, 3, 1, 5, 5, 16, torch.float32, seed=6)
    _, lse = oracle.attention(q, k, v, 0.3, True, return_lse=True)
    for h in range(3):
        want = 0.3 * float(np.dot(f64(q)[0, 0, h], f64(k)[0, 0, 0]))
        assert lse[0, h, 0] == pytest.approx(want, abs=1e-13)


def test_lse_two_keys_closed_form_and_far_range():
    """Two keys: lse = max(s0, s1) + log(1 + exp(-|s0 - s1|)); with |s| ~ 1000
    (exp overflows in fp64) the same closed form gives the larger score."""
    q = torch.tensor([[[[1.0, 2.0]]]], dtype=torch.float64)
    k = torch.tensor([[[[0.5, -1.0]], [[2.0, 0.25]]]], dtype=torch.float64)
    v = torch.zeros(1, 2, 1, 2, dtype=torch.float64)
    for scale in (0.7, 500.0, -500.0):
        s0, s1 = scale * -1.5, scale * 2.5
        want = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
        _, lse = oracle.attention(q, k, v, scale, False, return_lse=True)
        assert lse[0, 0, 0] == pytest.approx(want, rel=1e-15, abs=1e-15)


def test_lse_normalises_the_probabilities():
    """exp(s_j - lse) are the softmax probabilities: they sum to one and equal
    the oracle's P row."""
    q, k, v = fa_inputs.prefill_inputs(1, 2, 1, 7, 11, 8, torch.bfloat16, seed=8)
    _, lse = oracle.attention(q, k, v, 0.4, True, return_lse=True)
    qd, kd = f64(q), f64(k)
    for h in range(2):
        for i in (0, 3, 6):
            p, _ = oracle.probs(q, k, v, 0.4, True, b=0, h=h, i=i)
            s = 0.4 * (kd[0, :, 0, :] @ qd[0, i, h])
            vis = p > 0
            np.testing.assert_allclose(np.exp(s[vis] - lse[0, h, i]), p[vis], rtol=1e-13)
            assert np.exp(s[vis] - lse[0, h, i]).sum() == pytest.approx(1.0, abs=1e-14)


def test_decode_lse_equals_prefill_lse_and_ignores_nan_tail():
    q, kc, vc, L = fa_inputs.decode_inputs(2, 8, 2, 64, 32, seed=2, L=41)
    _, lse_dec = oracle.decode(q, kc, vc, L, 0.2, return_lse=True)
    _, lse_pre = oracle.attention(q, kc[:, :L], vc[:, :L], 0.2, False, return_lse=True)
    np.testing.assert_array_equal(lse_dec, lse_pre[:, :, 0])
    assert np.all(np.isfinite(lse_dec))
    _, lse0 = oracle.decode(q, kc, vc, 0, 0.2, return_lse=True)
    assert np.all(np.isneginf(lse0))


# ---------------------------------------------------------------------------
# 11. Packed (variable-length) sequences: each sequence is its own dense
#     problem; a packed batch of equal lengths is the dense batch.
# ---------------------------------------------------------------------------
def test_varlen_equal_lengths_equal_dense_batch():
    B, Hq, Hkv, Sq, Sk, D = 3, 4, 2, 9, 13, 8
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=21)
    cq = [b * Sq for b in range(B + 1)]
    ck = [b * Sk for b in range(B + 1)]
    for causal in (True, False):
        o_d, l_d = oracle.attention(q, k, v, 0.3, causal, return_lse=True)
        o_v, l_v = oracle.attention_varlen(q.reshape(B * Sq, Hq, D), k.reshape(B * Sk, Hkv, D),
                                           v.reshape(B * Sk, Hkv, D), cq, ck, 0.3, causal,
                                           return_lse=True)
        np.testing.assert_array_equal(o_v, o_d.reshape(B * Sq, Hq, D))
        np.testing.assert_array_equal(l_v, l_d.transpose(1, 0, 2).reshape(Hq, B * Sq))


def test_varlen_sequences_are_independent_and_empty_ones_write_nothing():
    """Changing one sequence's keys leaves the other sequences' rows unchanged;
    a sequence without keys gives O = 0 and lse = -inf; one without queries
    owns no rows."""
    lens_q, lens_k = [5, 0, 7, 3], [6, 4, 0, 9]
    cq = np.concatenate([[0], np.cumsum(lens_q)])
    ck = np.concatenate([[0], np.cumsum(lens_k)])
    g = torch.Generator().manual_seed(22)
    q = torch.randn(int(cq[-1]), 4, 8, generator=g).to(torch.bfloat16)
    k = torch.randn(int(ck[-1]), 2, 8, generator=g).to(torch.bfloat16)
    v = torch.randn(int(ck[-1]), 2, 8, generator=g).to(torch.bfloat16)
    o, l = oracle.attention_varlen(q, k, v, cq, ck, 0.4, True, return_lse=True)
    assert np.array_equal(o[5:12], np.zeros((7, 4, 8)))       # sequence 2 has no keys
    assert np.all(np.isneginf(l[:, 5:12]))
    k2 = k.clone()
    k2[10:19] += 1.0                                          # sequence 3's keys only
    o2 = oracle.attention_varlen(q, k2, v, cq, ck, 0.4, True)
    assert np.array_equal(o2[:12], o[:12])
    assert np.max(np.abs(o2[12:] - o[12:])) > 1e-6


def test_paged_decode_identity_pages_equal_contiguous_decode():
    """Pages laid out in order (page_table[b] = b*P .. b*P + P-1) are the
    contiguous cache: the same result, bit for bit, per sequence length."""
    B, Hq, Hkv, D, ps, P = 3, 8, 2, 16, 32, 4
    cap = ps * P
    q, kc, vc, _ = fa_inputs.decode_inputs(B, Hq, Hkv, cap, D, seed=23, L=cap)
    kp = kc.reshape(B * P, ps, Hkv, D)
    vp = vc.reshape(B * P, ps, Hkv, D)
    table = [[b * P + p for p in range(P)] for b in range(B)]
    lens = [1, 77, cap]
    o, l = oracle.decode_paged(q, kp, vp, table, lens, 0.3, return_lse=True)
    for b in range(B):
        ob, lb = oracle.decode(q[b:b + 1], kc[b:b + 1], vc[b:b + 1], lens[b], 0.3,
                               return_lse=True)
        np.testing.assert_array_equal(o[b, 0], ob[0])
        np.testing.assert_array_equal(l[b, 0], lb[0])


def test_paged_decode_follows_the_page_table():
    """Scattering the same pages to other physical slots, with the table
    updated to match, leaves the result unchanged; pointing the table at a
    different page changes it."""
    B, Hq, Hkv, D, ps, P = 2, 4, 1, 8, 32, 3
    q, kc, vc, _ = fa_inputs.decode_inputs(B, Hq, Hkv, ps * P, D, seed=24, L=ps * P)
    kp = kc.reshape(B * P, ps, Hkv, D)
    vp = vc.reshape(B * P, ps, Hkv, D)
    table = [[b * P + p for p in range(P)] for b in range(B)]
    lens = [80, 96]
    base = oracle.decode_paged(q, kp, vp, table, lens, 0.5)
    perm = torch.randperm(B * P, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(B * P)
    kp2, vp2 = kp[perm], vp[perm]                    # physical slot i holds old page perm[i]
    table2 = [[int(inv[x]) for x in row] for row in table]
    np.testing.assert_array_equal(oracle.decode_paged(q, kp2, vp2, table2, lens, 0.5), base)
    table3 = [row[:] for row in table]
    table3[1][0] = table[0][0]                        # sequence 1 reads sequence 0's first page
    changed = oracle.decode_paged(q, kp, vp, table3, lens, 0.5)
    np.testing.assert_array_equal(changed[0], base[0])
    assert np.max(np.abs(changed[1] - base[1])) > 1e-6


def test_paged_decode_several_new_tokens_is_causal_within_them():
    """Sq new tokens: token s equals a single-token decode over the first
    L - Sq + s + 1 tokens (it sees itself and the tokens before it)."""
    B, Sq, Hq, Hkv, D, ps, P = 2, 3, 4, 2, 8, 32, 3
    g = torch.Generator().manual_seed(25)
    kp = torch.randn(B * P, ps, Hkv, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(B * P, ps, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(B, Sq, Hq, D, generator=g).to(torch.bfloat16)
    table = [[b * P + p for p in range(P)] for b in range(B)]
    lens = [70, 2]                      # sequence 1: token 0 of 3 sees no key
    o, l = oracle.decode_paged(q, kp, vp, table, lens, 0.4, return_lse=True)
    for b in range(B):
        kc = kp[b * P:(b + 1) * P].reshape(1, P * ps, Hkv, D)
        vc = vp[b * P:(b + 1) * P].reshape(1, P * ps, Hkv, D)
        for s_ in range(Sq):
            vis = lens[b] - Sq + s_ + 1
            ob, lb = oracle.decode(q[b:b + 1, s_], kc, vc, max(vis, 0), 0.4, return_lse=True)
            np.testing.assert_array_equal(o[b, s_], ob[0])
            np.testing.assert_array_equal(l[b, s_], lb[0])


# ---------------------------------------------------------------------------
# 12. Backward pass: gradients of sum(O * dO).
# ---------------------------------------------------------------------------
def test_bwd_matches_central_differences_of_the_forward():
    """Each gradient entry against (f(x + h) - f(x - h)) / 2h of the forward
    oracle's loss sum(O * dO), in fp64: independent of the backward code."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 5, 7, 4
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.float64, seed=30)
    dout = torch.randn(B, Sq, Hq, D, generator=torch.Generator().manual_seed(31),
                       dtype=torch.float64)
    for causal in (True, False):
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, 0.7, causal)
        loss = lambda q_, k_, v_: float((oracle.attention(q_, k_, v_, 0.7, causal)  # noqa: E731
                                         * dout.numpy()).sum())
        h = 1e-5
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            flat = x.reshape(-1)
            num = np.zeros(flat.numel())
            for n in range(flat.numel()):
                xp, xm = flat.clone(), flat.clone()
                xp[n] += h
                xm[n] -= h
                args = [q, k, v]
                idx = "qkv".index(name)
                args[idx] = xp.reshape(x.shape)
                fp = loss(*args)
                args[idx] = xm.reshape(x.shape)
                num[n] = (fp - loss(*args)) / (2 * h)
            np.testing.assert_allclose(g.reshape(-1), num, rtol=0, atol=1e-7, err_msg=name)


def test_bwd_matches_torch_autograd_fp64():
    """torch CPU fp64 scaled_dot_product_attention + autograd, GQA via
    repeat_interleave (whose gradient sums a group's heads), bottom-right
    causal via an explicit mask."""
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 9, 13, 8
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=32)
    dout = torch.randn(B, Sq, Hq, D, generator=torch.Generator().manual_seed(33))
    for causal in (True, False):
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, 0.3, causal)
        qt, kt, vt = (x.to(torch.float64).requires_grad_() for x in (q, k, v))
        G = Hq // Hkv
        mask = None
        if causal:
            mask = torch.arange(Sk)[None, :] <= torch.arange(Sq)[:, None] + (Sk - Sq)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt.permute(0, 2, 1, 3), kt.repeat_interleave(G, 2).permute(0, 2, 1, 3),
            vt.repeat_interleave(G, 2).permute(0, 2, 1, 3), attn_mask=mask, scale=0.3)
        (o.permute(0, 2, 1, 3) * dout.to(torch.float64)).sum().backward()
        np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=0, atol=1e-11)


def test_bwd_key_gradients_sum_to_zero_and_uniform_value_gradients():
    """Softmax rows are shift invariant, so sum_j dS_ij = 0 and (non-causal)
    sum_j dK_j = 0; with Q = 0 every row weights its keys equally, so
    dV_j = sum_i dO_i / Sk."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 6, 10, 8
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, torch.bfloat16, seed=34)
    dout = torch.randn(B, Sq, Hq, D, generator=torch.Generator().manual_seed(35))
    _, dk, _ = oracle.attention_bwd(q, k, v, dout, 0.5, False)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    q0 = torch.zeros_like(q)
    _, _, dv = oracle.attention_bwd(q0, k, v, dout, 0.5, False)
    want = dout.to(torch.float64).numpy().sum(axis=1) / Sk          # [B, Hq, D], Hq == Hkv
    for j in range(Sk):
        np.testing.assert_allclose(dv[:, j], want, atol=1e-12)


# ---------------------------------------------------------------------------
# 13. Stored oracle values (tests/golden/oracle_tiny.txt, written by
#     tests/golden/make_golden.py from the oracle alone): drift guard.
# ---------------------------------------------------------------------------
def test_golden_oracle_values_unchanged():
    with open(os.path.join(GOLDEN, "oracle_tiny.txt")) as f:
        lines = [ln for ln in f.read().splitlines() if ln and not ln.startswith("#")]
    assert len(lines) % 2 == 0 and lines
    for hdr, vals in zip(lines[0::2], lines[1::2]):
        _, name, B, Hq, Hkv, Sq, Sk, D, causal, dts, scale, seed = hdr.split()
        dt = torch.bfloat16 if dts == "bf16" else torch.float16
        q, k, v = fa_inputs.prefill_inputs(int(B), int(Hq), int(Hkv), int(Sq), int(Sk),
                                           int(D), dt, int(seed))
        o = oracle.attention(q, k, v, float(scale), bool(int(causal)))
        ref = np.array([float(x) for x in vals.split()])
        np.testing.assert_allclose(o.ravel(), ref, rtol=0, atol=1e-15)
