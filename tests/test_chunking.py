"""Row chunking of the decode step under a logits budget: the native slice
planner against the oracle's rule (CPU), and on the GPU the chunked step
(one native call, a schedule per slice, one reused logits scratch) against
the unchunked step, bit for bit."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W


@pytest.fixture(scope="module")
def lib():
    dsa.build()
    return dsa.lib()


# ---------------------------------------------------------------------------
# CPU
# ---------------------------------------------------------------------------

def test_slice_planner_equals_the_oracle(lib):
    rng = np.random.default_rng(11)
    cases = [(134, 120064, 16 << 20), (1000, 4096, 819200), (40, 64, 5120), (0, 64, 100),
             (17, 64, 0), (33, 64, 2048), (2**20, 1024, 64 << 20)]
    for _ in range(300):
        rows = int(rng.integers(1, 5000))
        width = int(rng.integers(1, 300)) * 64
        budget = int(rng.integers(16, 6000)) * width * 2 + int(rng.integers(0, 2 * width))
        cases.append((rows, width, budget))
    for rows, width, budget in cases:
        assert dsa.decode_chunk_ranges(rows, width, budget) == oracle.decode_chunk_ranges(rows, width, budget), \
            (rows, width, budget)


def test_slice_planner_errors(lib):
    n = ctypes.c_int32(0)
    buf = (ctypes.c_int32 * 8)()
    E = dsa.DSA_ERR_INVALID_ARG
    f = lib.dsa_decode_chunk_ranges
    assert f(10, 64, -1, ctypes.cast(buf, ctypes.c_void_p), 4, ctypes.byref(n)) == E
    assert f(100, 64, 15 * 64 * 2, ctypes.cast(buf, ctypes.c_void_p), 4, ctypes.byref(n)) == E
    assert f(100, 0, 10**6, ctypes.cast(buf, ctypes.c_void_p), 4, ctypes.byref(n)) == E
    assert f(100, 64, 16 * 128, ctypes.cast(buf, ctypes.c_void_p), 4, ctypes.byref(n)) == E  # 7 slices > 4
    assert f(100, 64, 16 * 128, None, 0, None) == E
    assert f(100, 64, 16 * 128, ctypes.cast(buf, ctypes.c_void_p), 4, None) == E
    assert f(100, 64, 10**9, None, 0, ctypes.byref(n)) == dsa.DSA_OK and n.value == 0


def test_scratch_sizes(lib):
    # fp32 logits count 4 bytes a column: the budget holds half as many rows
    sb, sw = dsa.indexer_decode_scratch(134, dsa.LOGITS_F32, 120064, 32 << 20, 152)
    r = oracle.decode_chunk_ranges(134, 2 * 120064, 32 << 20)
    assert sb == (r[0][1] - r[0][0]) * 120064 * 4 and sw == dsa.schedule_words(152, r[0][1] - r[0][0])
    sb, sw = dsa.indexer_decode_scratch(134, dsa.LOGITS_BF16, 120064, 0, 152)
    assert sb == 134 * 120064 * 2 and sw == dsa.schedule_words(152, 134)


def test_decode_step_host_checks(lib):
    P = ctypes.c_void_p

    def call(**kw):
        a = dict(q=P(16), qs=None, kv=P(16), pst=8448, npages=4, fmt=0, w=P(16), ctx=P(16), bt=P(16), bts=4,
                 ind=None, T=64, H=64, D=128, bkv=64, nsms=8, odt=1, ost=256, budget=16 * 256 * 2,
                 scr=P(16), scrb=16 * 256 * 2, sched=P(16), schw=10**6, k=16, out=P(16), outs=16,
                 status=None, stream=None)
        a.update(kw)
        return lib.dsa_indexer_decode_topk(*a.values())

    assert call(H=32) == dsa.DSA_ERR_UNSUPPORTED
    assert call(k=4096) == dsa.DSA_ERR_UNSUPPORTED
    assert call(odt=7) == dsa.DSA_ERR_UNSUPPORTED
    assert call(scrb=16 * 256 * 2 - 1) == dsa.DSA_ERR_INVALID_ARG       # scratch below one slice
    assert call(schw=dsa.schedule_words(8, 16) - 1) == dsa.DSA_ERR_INVALID_ARG
    assert call(budget=15 * 256 * 2) == dsa.DSA_ERR_INVALID_ARG         # not even 16 rows
    assert call(outs=8) == dsa.DSA_ERR_INVALID_ARG
    assert call(q=None) == dsa.DSA_ERR_INVALID_ARG
    assert call(T=0) == dsa.DSA_OK


# ---------------------------------------------------------------------------
# GPU
# ---------------------------------------------------------------------------

MANY_ROWS = dict(request_lens=[300, 517, 70, 1000, 129, 2100, 64, 700, 1500, 65],
                 rows_per_request=[5, 7, 3, 9, 6, 4, 8, 1, 11, 2])   # 56 rows, slices cut requests


@pytest.mark.gpu
@pytest.mark.parametrize("kv_format,ldt", [(W.KV_FP8, W.LOGITS_F32), (W.KV_FP8, W.LOGITS_BF16),
                                           (W.KV_FP4, W.LOGITS_BF16), (W.KV_MXFP4, W.LOGITS_BF16)])
@pytest.mark.parametrize("slice_rows", [16, 32, 48, 0])
def test_chunked_step_equals_one_pass(kv_format, ldt, slice_rows):
    from gpu_helpers import run_path
    wl = W.build("chunk", **MANY_ROWS, kv_format=kv_format, logits_dtype=ldt, topk=128, seed=21)
    ref = run_path(wl)
    assert int(ref["status"].item()) == 0
    g = ref["dev_wl"]
    eb = 4 if ldt == W.LOGITS_F32 else 2
    budget = slice_rows * g.logits_stride * eb + (eb if slice_rows else 0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dsa.indexer_decode_topk(g.q, g.kv_cache, g.weights, g.context_lens, g.block_table, g.topk,
                                  indices=g.indices, kv_format=kv_format, logits_dtype=ldt,
                                  logits_stride=g.logits_stride, logits_budget=budget, status=status,
                                  q_scale=g.q_scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, ref["idx"])
    if slice_rows:
        ranges = dsa.decode_chunk_ranges(g.num_rows, g.logits_stride * eb // 2, budget)
        assert len(ranges) == -(-g.num_rows // slice_rows)


@pytest.mark.gpu
def test_chunked_step_plain_decode_rows():
    from gpu_helpers import run_path
    wl = W.build("chunk_plain", [int(x) for x in np.linspace(64, 3000, 40)], [1] * 40, topk=256,
                 plain_indices=True, seed=22)
    ref = run_path(wl, use_indices=False)
    g = ref["dev_wl"]
    out = dsa.indexer_decode_topk(g.q, g.kv_cache, g.weights, g.context_lens, g.block_table, g.topk,
                                  indices=None, logits_stride=g.logits_stride,
                                  logits_budget=16 * g.logits_stride * 4)   # fp32: 16-row slices
    torch.cuda.synchronize()
    assert torch.equal(out, ref["idx"])
