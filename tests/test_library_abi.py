"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/dsa_indexer.h declares, and rejects bad arguments on the host before
any device work (no compute calls here)."""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_paged_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa_indexer.h")


@pytest.fixture(scope="module")
def lib():
    dsa.build()
    return dsa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_calls():
    names = declared_functions()
    for must in ("dsa_paged_mqa_logits_metadata", "dsa_fp8_fp4_paged_mqa_logits",
                 "dsa_top_k_per_row"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(dsa.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name
    assert set(declared_functions()) == set(dsa.EXPORTED)


def test_constants_match_header():
    src = open(HEADER).read()
    for macro, val in (("DSA_FP8_PAGE_BYTES", dsa.FP8_PAGE_BYTES),
                       ("DSA_FP4_PAGE_BYTES", dsa.FP4_PAGE_BYTES),
                       ("DSA_MXFP4_PAGE_BYTES", dsa.MXFP4_PAGE_BYTES),
                       ("DSA_MAX_TOPK", dsa.MAX_TOPK), ("DSA_BLOCK_KV", dsa.BLOCK_KV)):
        assert re.search(rf"#define {macro} {val}\b", src), macro


def test_status_strings(lib):
    for code in range(8):
        assert dsa.status_string(code)
    assert dsa.status_string(99) == "unknown status"


def test_schedule_words(lib):
    assert lib.dsa_schedule_words(148, 134) == 8 + 2 * 149 + 5 * 135
    assert lib.dsa_schedule_words(0, 5) == -1


P = ctypes.c_void_p


def _logits_call(lib, **kw):
    a = dict(q=P(16), kv=P(16), pstride=8448, npages=4, fmt=0, w=P(16), ctx=P(16), bt=P(16),
             btst=4, ind=None, sched=P(16), nsms=1, out=P(16), odt=0, ost=64, T=1, H=64, D=128,
             bkv=64, status=None, stream=None)
    a.update(kw)
    return lib.dsa_fp8_fp4_paged_mqa_logits(a["q"], a["kv"], a["pstride"], a["npages"], a["fmt"],
                                            a["w"], a["ctx"], a["bt"], a["btst"], a["ind"],
                                            a["sched"], a["nsms"], a["out"], a["odt"], a["ost"],
                                            a["T"], a["H"], a["D"], a["bkv"], a["status"],
                                            a["stream"])


def test_host_checks_logits(lib):
    assert _logits_call(lib, H=32) == dsa.DSA_ERR_UNSUPPORTED
    assert _logits_call(lib, D=64) == dsa.DSA_ERR_UNSUPPORTED
    assert _logits_call(lib, bkv=32) == dsa.DSA_ERR_UNSUPPORTED
    assert _logits_call(lib, fmt=7) == dsa.DSA_ERR_UNSUPPORTED
    assert _logits_call(lib, odt=5) == dsa.DSA_ERR_UNSUPPORTED
    assert _logits_call(lib, T=0) == dsa.DSA_OK            # nothing to do, no device touched
    assert _logits_call(lib, q=None) == dsa.DSA_ERR_INVALID_ARG
    assert _logits_call(lib, pstride=8440) == dsa.DSA_ERR_INVALID_ARG
    assert _logits_call(lib, pstride=8456) == dsa.DSA_ERR_INVALID_ARG   # not a multiple of 16
    assert _logits_call(lib, fmt=1, pstride=4800) == dsa.DSA_ERR_INVALID_ARG
    assert _logits_call(lib, npages=0) == dsa.DSA_ERR_INVALID_ARG
    assert _logits_call(lib, ost=60) == dsa.DSA_ERR_INVALID_ARG
    assert _logits_call(lib, q=P(17)) == dsa.DSA_ERR_INVALID_ARG       # misaligned
    assert _logits_call(lib, nsms=0) == dsa.DSA_ERR_INVALID_ARG


def test_host_checks_metadata_and_topk(lib):
    assert lib.dsa_paged_mqa_logits_metadata(P(16), None, 4, 32, 8, P(16), None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_paged_mqa_logits_metadata(P(16), None, -1, 64, 8, P(16), None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_paged_mqa_logits_metadata(P(16), None, 4, 64, 8, None, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_paged_mqa_logits_metadata_for_keys(P(16), None, 4, 64, 8, 3, P(16), None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_paged_mqa_logits_metadata_for_keys(P(16), None, 4, 32, 8, dsa.KV_FP4, P(16), None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_top_k_per_row(P(16), 0, 64, None, P(16), 2, 0, P(16), 8, None, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_top_k_per_row(P(16), 0, 64, None, P(16), 2, 4096, P(16), 4096, None, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_top_k_per_row(P(16), 0, 64, None, P(16), 2, 16, P(16), 8, None, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_top_k_per_row(P(16), 0, 62, None, P(16), 2, 16, P(16), 16, None, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_top_k_per_row(P(16), 0, 64, None, P(16), 0, 16, P(16), 16, None, None) == \
        dsa.DSA_OK


def test_host_checks_selftest(lib):
    st = P(256)
    assert lib.dsa_selftest_wait_timeout(999, st, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_selftest_wait_timeout(2_000_000_000, st, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_selftest_wait_timeout(1_000_000, None, None) == dsa.DSA_ERR_INVALID_ARG


def test_host_checks_dcp(lib):
    E, U, OK = dsa.DSA_ERR_INVALID_ARG, dsa.DSA_ERR_UNSUPPORTED, dsa.DSA_OK
    pack = lib.dsa_dcp_pack_topk
    # logits, dtype, stride, idx, idx_stride, rows, k, rank, world, interleave, packed, stream
    assert pack(P(16), 7, 64, P(16), 16, 2, 16, 0, 2, 1, P(16), None) == U           # logits dtype
    assert pack(P(16), 0, 64, P(16), 16, 2, 0, 0, 2, 1, P(16), None) == U            # k < 1
    assert pack(P(16), 0, 64, P(16), 16, 2, 4096, 0, 2, 1, P(16), None) == U         # k > max
    assert pack(P(16), 0, 64, P(16), 16, 2, 16, 0, 9, 1, P(16), None) == U           # world > max
    assert pack(P(16), 0, 64, P(16), 16, 2, 16, 2, 2, 1, P(16), None) == E           # rank >= world
    assert pack(P(16), 0, 64, P(16), 16, 2, 16, 0, 2, 0, P(16), None) == E           # interleave < 1
    assert pack(P(16), 0, 64, P(16), 8, 2, 16, 0, 2, 1, P(16), None) == E            # idx_stride < k
    assert pack(P(16), 0, 1 << 22, P(16), 16, 2, 16, 0, 4, 1, P(16), None) == E      # ids past 2^24
    assert pack(P(16), 0, 64, P(16), 16, 2, 16, 0, 2, 1, P(20), None) == E       # packed alignment
    assert pack(P(16), 0, 64, None, 16, 2, 16, 0, 2, 1, P(16), None) == E            # null
    assert pack(None, 0, 64, None, 16, 0, 16, 0, 2, 1, None, None) == OK             # no rows
    merge = lib.dsa_dcp_merge_topk
    # gathered, world, rows, k, out, out_stride, stream
    assert merge(P(16), 0, 2, 16, P(16), 16, None) == U
    assert merge(P(16), 9, 2, 16, P(16), 16, None) == U
    assert merge(P(16), 2, 2, 4096, P(16), 4096, None) == U
    assert merge(P(16), 2, 2, 16, P(16), 15, None) == E
    assert merge(P(20), 2, 2, 16, P(16), 16, None) == E
    assert merge(P(16), 2, 2, 16, None, 16, None) == E
    assert merge(None, 2, 0, 16, None, 16, None) == OK


def test_product_path_has_no_fallback():
    """The package imports nothing from the oracle and has no CPU compute path."""
    pkg = os.path.dirname(dsa.__file__)
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "oracle" not in src, fn
            assert "numpy" not in src, fn
