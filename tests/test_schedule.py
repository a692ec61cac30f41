"""Host copy of the persistent prefill scheduler's work-item decode: every
(b, query head, 256-row query block) appears exactly once; items of one K/V
head are contiguous (kv-head-major, for L2 reuse of K/V -- the "hkv-major"
decode of the gfx950 README's persistent mode); within a K/V head and batch
entry the query blocks run longest-first."""
import pytest

from tests.test_abi import lib  # noqa: F401  (fixture)


@pytest.mark.parametrize("B,Hq,Hkv,Sq", [(1, 128, 8, 8192), (4, 16, 16, 4096), (2, 8, 8, 1000),
                                         (1, 2, 1, 128), (3, 6, 3, 300)])
def test_items_are_a_bijection_in_kv_head_major_order(lib, B, Hq, Hkv, Sq):  # noqa: F811
    import attention_fa_fwd_04_gb300 as fa
    n_qb = (Sq + 255) // 256
    n, *_ = fa.fa_prefill_work_item(0, B, Hq, Hkv, Sq)
    assert n == B * Hq * n_qb
    G = Hq // Hkv
    seen = set()
    prev = None
    for w in range(n):
        _, b, hq, qb = fa.fa_prefill_work_item(w, B, Hq, Hkv, Sq)
        assert 0 <= b < B and 0 <= hq < Hq and 0 <= qb < n_qb
        seen.add((b, hq, qb))
        key = (hq // G, b)
        if prev is not None:
            assert key >= prev[0]                      # kv-head-major, then batch
            if key == prev[0]:
                assert qb <= prev[1]                   # longest query blocks first
        prev = (key, qb)
    assert len(seen) == n


def test_work_item_rejects_bad_shapes(lib):  # noqa: F811
    import attention_fa_fwd_04_gb300 as fa
    assert fa.fa_prefill_work_item(0, 1, 6, 4, 128)[0] == -1
    assert fa.fa_prefill_work_item(0, 1, 4, 0, 128)[0] == -1
