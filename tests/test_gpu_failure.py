"""Failure detection on the GPU without a fault: a bounded pipeline wait that
nothing satisfies gives up after its time limit, the host reads
DSA_ERR_TIMEOUT from the status word, and the context keeps working."""
import time

import pytest
import torch

import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W
from gpu_helpers import run_path, check_logits, check_topk_exact

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dsa.selftest_wait_timeout(20_000_000, st)   # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == dsa.DSA_ERR_TIMEOUT
    assert elapsed >= 0.015, elapsed            # it did wait, then gave up
    assert elapsed < 2.0, elapsed
    # the context is intact: a normal step runs and matches the oracle
    wl = W.config("tiny")
    out = run_path(wl)
    assert int(out["status"].item()) == dsa.DSA_OK
    check_logits(wl, out["logits"])
    check_topk_exact(out["logits"], out["idx"], wl.context_lens, wl.topk)


def test_first_error_wins():
    st = torch.full((1,), dsa.DSA_ERR_BAD_BLOCK, dtype=torch.int32, device="cuda")
    dsa.selftest_wait_timeout(1_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == dsa.DSA_ERR_BAD_BLOCK
