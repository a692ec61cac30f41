"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects invalid arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from attention_fa_fwd_04_gb300 import build
    build.build()
    import attention_fa_fwd_04_gb300 as fa
    return fa.load()


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_abi():
    syms = declared_symbols()
    for s in ("fa_prefill_fwd", "fa_decode_fwd", "fa_status_string"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    import attention_fa_fwd_04_gb300 as fa
    syms = declared_symbols()
    assert set(fa.EXPORTS) == set(syms), (fa.EXPORTS, syms)
    for s in syms:
        assert hasattr(lib, s), f"{s} missing from libfa_gb300.so"


def test_status_strings(lib):
    import attention_fa_fwd_04_gb300 as fa
    for st in range(7):
        assert fa.fa_status_string(st).startswith("FA_")
    assert fa.fa_status_string(99) == "unknown status"


FAKE = 0x10000  # a 16-byte-aligned non-null address: never dereferenced on these paths


@pytest.mark.parametrize("kw", [
    dict(D=96), dict(D=0), dict(Hq=6, Hkv=4), dict(Hkv=0), dict(B=-1), dict(Sq=-3),
    dict(Sk=-1), dict(dtype=7), dict(scale=float("inf")), dict(scale=float("nan")),
    dict(q=0), dict(o=0), dict(k=0), dict(v=0), dict(q=FAKE + 8), dict(o=FAKE + 2),
])
def test_prefill_rejects_invalid_arguments(lib, kw):
    import attention_fa_fwd_04_gb300 as fa
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, Hq=4, Hkv=2, Sq=16, Sk=16, D=64,
             scale=0.125, causal=1, dtype=fa.FA_BF16, stream=0)
    a.update(kw)
    st = fa.fa_prefill_fwd(a["q"], a["k"], a["v"], a["o"], a["B"], a["Hq"], a["Hkv"], a["Sq"],
                           a["Sk"], a["D"], a["scale"], a["causal"], a["dtype"], a["stream"])
    assert st == fa.FA_ERR_INVALID_ARG


def test_prefill_empty_problems_are_noops(lib):
    import attention_fa_fwd_04_gb300 as fa
    for B, Hq, Sq in ((0, 4, 16), (1, 0, 16), (1, 4, 0)):
        assert fa.fa_prefill_fwd(0, 0, 0, 0, B, Hq, 2, Sq, 16, 64, 0.1, 1, fa.FA_BF16, 0) == fa.FA_OK


@pytest.mark.parametrize("kw", [
    dict(D=80), dict(Hq=3, Hkv=2), dict(Hkv=0), dict(cap=-1), dict(B=-2),
    dict(scale=float("-inf")), dict(q=0), dict(o=0), dict(kc=0), dict(vc=0), dict(vl=0),
    dict(vl=FAKE + 2), dict(kc=FAKE + 4), dict(B=70000),
])
def test_decode_rejects_invalid_arguments(lib, kw):
    import attention_fa_fwd_04_gb300 as fa
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, vl=FAKE, o=FAKE, B=1, Hq=8, Hkv=2, cap=128, D=128,
             scale=0.088, stream=0)
    a.update(kw)
    st = fa.fa_decode_fwd(a["q"], a["kc"], a["vc"], a["vl"], a["o"], a["B"], a["Hq"], a["Hkv"],
                          a["cap"], a["D"], a["scale"], a["stream"])
    assert st == fa.FA_ERR_INVALID_ARG


def test_decode_empty_problems_are_noops(lib):
    import attention_fa_fwd_04_gb300 as fa
    assert fa.fa_decode_fwd(0, 0, 0, 0, 0, 0, 8, 2, 128, 128, 0.1, 0) == fa.FA_OK
    assert fa.fa_decode_fwd(0, 0, 0, 0, 0, 1, 0, 2, 128, 128, 0.1, 0) == fa.FA_OK


def test_lse_variants_reject_missing_or_misaligned_lse(lib):
    import attention_fa_fwd_04_gb300 as fa
    for lse in (0, FAKE + 2):
        assert fa.fa_prefill_fwd_lse(FAKE, FAKE, FAKE, FAKE, lse, 1, 4, 2, 16, 16, 64, 0.125, 1,
                                     fa.FA_BF16, 0) == fa.FA_ERR_INVALID_ARG
        assert fa.fa_decode_fwd_lse(FAKE, FAKE, FAKE, FAKE, FAKE, lse, 1, 8, 2, 128, 128, 0.088,
                                    0) == fa.FA_ERR_INVALID_ARG
    # the remaining argument rules are the plain entry points'
    assert fa.fa_prefill_fwd_lse(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 16, 16, 96, 0.125, 1,
                                 fa.FA_BF16, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_decode_fwd_lse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 3, 2, 128, 128, 0.088,
                                0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_prefill_fwd_lse(0, 0, 0, 0, 0, 0, 4, 2, 16, 16, 64, 0.1, 1, fa.FA_BF16,
                                 0) == fa.FA_OK


def test_rescale_count_rejects_a_null_output(lib):
    import attention_fa_fwd_04_gb300 as fa
    assert lib.fa_prefill_rescale_count(0, None) == fa.FA_ERR_INVALID_ARG
