"""Prefill over the paged cache: token rows tagged (cu_seqlen_ks, cu_seqlen_ke)
against the oracle, and against the decode path on the same rows."""
import ctypes
import types

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W

P = ctypes.c_void_p
# last n_r tokens of each request as rows; a length-0 request with one row
MIX = dict(request_lens=[300, 517, 0, 70, 1000], rows_per_request=[100, 517, 1, 3, 250])


@pytest.fixture(scope="module")
def lib():
    dsa.build()
    return dsa.lib()


def test_host_checks_prefill(lib):
    E, OK = dsa.DSA_ERR_INVALID_ARG, dsa.DSA_OK
    f = lib.dsa_prefill_rows
    assert f(P(16), P(16), -1, P(16), 2, P(16), P(16), None, None) == E
    assert f(P(16), P(16), 4, P(16), 0, P(16), P(16), None, None) == E
    assert f(P(16), None, 4, P(16), 2, P(16), P(16), None, None) == E
    assert f(None, None, 0, None, 2, None, None, None, None) == OK
    g = lib.dsa_prefill_mqa_logits
    a = [P(16), None, P(16), 8448, 4, 0, P(16), P(16), P(16), P(16), 4, 2, P(16), 8, P(16), 0, 64, 4, 64, 128,
         64, None, None]
    bad = list(a)
    bad[8] = None                                   # request ids
    assert g(*bad) == E
    bad = list(a)
    bad[11] = 0                                     # no requests
    assert g(*bad) == E
    bad = list(a)
    bad[18] = 32                                    # heads
    assert g(*bad) == dsa.DSA_ERR_UNSUPPORTED
    bad = list(a)
    bad[1] = P(16)                                  # q scales with FP8 keys
    assert g(*bad) == E


def _view(pf, ctx):
    return types.SimpleNamespace(num_rows=pf.num_rows, context_lens=torch.as_tensor(ctx))


def _run(pf, status):
    g = pf.to("cuda")
    idx, logits = dsa.prefill_topk(g.q, g.kv_cache, g.weights, g.cu_seqlen_ks, g.cu_seqlen_ke,
                                   g.local_cu_seq_lens, g.block_table, g.topk, kv_format=g.kv_format,
                                   logits_dtype=g.logits_dtype, logits_stride=g.logits_stride, status=status,
                                   q_scale=g.q_scale)
    torch.cuda.synchronize()
    return idx, logits


@pytest.mark.gpu
def test_prefill_rows_kernel_equals_oracle():
    rng = np.random.default_rng(5)
    starts = np.array([0, 5, 5, 9, 200, 200, 1000], dtype=np.int32)
    ks, ke = [0, 0, 5, 5, 9, 1000], [3, 5, 6, 9, 9, 1000]
    for _ in range(300):
        r = int(rng.integers(0, 6))
        ks.append(int(starts[r]))
        ke.append(int(starts[r] + rng.integers(0, starts[r + 1] - starts[r] + 1)))
    ks, ke = np.array(ks, np.int32), np.array(ke, np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx, req = dsa.prefill_rows(torch.from_numpy(ks).cuda(), torch.from_numpy(ke).cuda(),
                                torch.from_numpy(starts).cuda(), status=st)
    torch.cuda.synchronize()
    want_ctx, want_req = oracle.prefill_rows(ks, ke, starts)
    assert int(st.item()) == 0
    assert np.array_equal(ctx.cpu().numpy(), want_ctx) and np.array_equal(req.cpu().numpy(), want_req)


@pytest.mark.gpu
@pytest.mark.parametrize("kv_format,ldt", [(W.KV_FP8, W.LOGITS_F32), (W.KV_FP8, W.LOGITS_BF16),
                                           (W.KV_FP4, W.LOGITS_BF16), (W.KV_MXFP4, W.LOGITS_BF16)])
def test_prefill_logits_and_topk_vs_oracle(kv_format, ldt):
    from gpu_helpers import check_logits, check_topk_exact, check_topk_tie_band
    wl = W.build("pf", **MIX, kv_format=kv_format, logits_dtype=ldt, topk=64, seed=31)
    pf = W.prefill_view(wl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, logits = _run(pf, st)
    assert int(st.item()) == 0
    ref, bound = oracle.prefill_logits(pf)
    ctx, _ = oracle.prefill_rows(pf.cu_seqlen_ks, pf.cu_seqlen_ke, pf.local_cu_seq_lens)
    check_logits(_view(pf, ctx), logits, ref=ref, bound=bound)
    check_topk_exact(logits, idx, torch.from_numpy(ctx), pf.topk)
    check_topk_tie_band(idx, ref, bound, torch.from_numpy(ctx), pf.topk, range(pf.num_rows))


@pytest.mark.gpu
@pytest.mark.parametrize("kv_format", [W.KV_FP8, W.KV_FP4])
def test_prefill_equals_decode_path_on_the_same_rows(kv_format):
    from gpu_helpers import run_path
    wl = W.build("pf", **MIX, kv_format=kv_format, topk=128, seed=32)
    dec = run_path(wl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, logits = _run(W.prefill_view(wl), st)
    assert int(st.item()) == 0
    ctx = wl.context_lens.numpy()
    for t in range(wl.num_rows):
        n = (int(ctx[t]) + 63) // 64 * 64
        assert torch.equal(logits[t, :n], dec["logits"][t, :n]), t
    assert torch.equal(idx, dec["idx"])


@pytest.mark.gpu
def test_prefill_full_size_sampled_rows():
    from gpu_helpers import check_logits, check_topk_exact
    wl = W.config("prefill")
    pf = W.prefill_view(wl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, logits = _run(pf, st)
    assert int(st.item()) == 0
    rows = [0, 1, 63, 64, 2047, 4095, 4096, 4097, 6000, 8190, 8191]
    ref, bound = oracle.prefill_logits(pf, rows=np.array(rows, np.int32))
    ctx, _ = oracle.prefill_rows(pf.cu_seqlen_ks, pf.cu_seqlen_ke, pf.local_cu_seq_lens)
    check_logits(_view(pf, ctx), logits, rows=rows, ref=ref, bound=bound)
    check_topk_exact(logits, idx, torch.from_numpy(ctx), pf.topk, rows=rows)


@pytest.mark.gpu
def test_prefill_request_id_outside_the_table_is_reported():
    wl = W.build("pf", [300, 200], [4, 4], topk=16, seed=33)
    g = W.prefill_view(wl).to("cuda")
    ctx, req = dsa.prefill_rows(g.cu_seqlen_ks, g.cu_seqlen_ke, g.local_cu_seq_lens)
    req[5:] = 2                                     # only requests 0 and 1 have a table row
    sched = dsa.paged_mqa_logits_metadata(ctx, req)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.prefill_mqa_logits(g.q, g.kv_cache, g.weights, ctx, req, g.block_table, sched,
                           logits_stride=g.logits_stride, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == dsa.DSA_ERR_BAD_BLOCK
