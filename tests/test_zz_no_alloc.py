"""The allocation-free decode step (dsa_indexer_decode_topk_static).

Some callers cannot call cudaMalloc: code running inside an allocator's own
callbacks, a plugin whose host framework owns every device allocation and
passes only the op's tensors, a serving loop whose memory is fixed after
start-up.  For them the library keeps the step's scratch (the logits of a row
slice and its schedule) in a fixed device array of its own.  These tests call
that entry point through the C ABI and check that its top-k equals the
caller-scratch entry point's (dsa_indexer_decode_topk) bit for bit, on two
calls in a row: the array keeps the first call's contents, which the second
must not depend on.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W


def _static_call(g, k, logits_dtype, logits_stride, out, status):
    lib = dsa.lib()
    qq = g.q.view(torch.uint8) if g.q.dtype != torch.uint8 else g.q
    return lib.dsa_indexer_decode_topk_static(
        ctypes.c_void_p(qq.data_ptr()),
        None if g.q_scale is None else ctypes.c_void_p(g.q_scale.data_ptr()),
        ctypes.c_void_p(g.kv_cache.data_ptr()), int(g.kv_cache.stride(0)), int(g.kv_cache.shape[0]),
        int(g.kv_format), ctypes.c_void_p(g.weights.data_ptr()), ctypes.c_void_p(g.context_lens.data_ptr()),
        ctypes.c_void_p(g.block_table.data_ptr()), int(g.block_table.stride(0)),
        None if g.indices is None else ctypes.c_void_p(g.indices.data_ptr()), g.num_rows,
        dsa.NUM_HEADS, dsa.HEAD_DIM, dsa.BLOCK_KV, dsa.device_num_sms(), int(logits_dtype), int(logits_stride),
        int(k), ctypes.c_void_p(out.data_ptr()), int(out.stride(0)), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _reference(g, logits_dtype):
    # the caller-scratch entry point, all rows in one pass
    return dsa.indexer_decode_topk(g.q, g.kv_cache, g.weights, g.context_lens, g.block_table, g.topk,
                                   indices=g.indices, kv_format=g.kv_format, logits_dtype=logits_dtype,
                                   logits_stride=g.logits_stride, logits_budget=0, q_scale=g.q_scale)


@pytest.mark.gpu
def test_static_scratch_step_equals_caller_scratch_step():
    dsa.build()
    dev = torch.device("cuda")
    # 64 rows of ~40K columns: 10 MB of fp32 logits, so the fixed 8 MiB array
    # runs them in two slices
    lens = [36000 + 131 * r for r in range(32)]
    big = W.build("static_a", lens, [2] * 32, topk=2048, seed=31, device=dev)
    # the second call: another workload (FP4 keys, bf16 logits, ragged groups)
    # into the same array, which still holds the first call's logits
    small = W.build("static_b", [300, 517, 70, 1000, 129, 2100, 64, 700],
                    [5, 7, 3, 9, 6, 4, 8, 1], kv_format=W.KV_FP4, logits_dtype=W.LOGITS_BF16,
                    topk=128, seed=32, device=dev)
    cases = [(big, W.LOGITS_F32), (small, W.LOGITS_BF16)]
    refs = [_reference(g, ldt) for g, ldt in cases]
    torch.cuda.synchronize()
    for (g, ldt), ref in zip(cases, refs):
        out = torch.full((g.num_rows, g.topk), -7, dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        rc = _static_call(g, g.topk, ldt, g.logits_stride, out, status)
        torch.cuda.synchronize()
        assert rc == dsa.DSA_OK, dsa.status_string(rc)
        assert int(status.item()) == 0, dsa.status_string(int(status.item()))
        assert torch.equal(out, ref)
    # rows too wide for the array: 16 fp32 rows of 140000 columns exceed
    # 8 MiB; the call is refused before any launch and leaves `out` untouched
    out = torch.full((small.num_rows, small.topk), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = _static_call(small, small.topk, W.LOGITS_F32, 140032, out, status)
    torch.cuda.synchronize()
    assert rc == dsa.DSA_ERR_SCRATCH_TOO_SMALL
    assert int(status.item()) == 0 and bool((out == -7).all())
