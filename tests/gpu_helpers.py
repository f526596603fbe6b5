"""Shared helpers of the GPU parity tests: run the path through the binding,
and compare its results with the CPU oracle.

Accuracy bar (stated with the indexer's decode path):
  logits    |gpu - oracle| <= 1e-3 * A + 1e-6 for every s < L_t, where
            A = kscale * sum_h sum_d |w q k| (oracle's bound); BF16 logits
            add the half-ulp of their rounding, 2^-9 * (|oracle| + tol);
            columns L_t <= s < round_up(L_t, 64) are -inf.
  top-k     bit-exact against the oracle's top-k of the GPU's own logits;
            against the oracle's top-k of the oracle's logits, a column may
            differ only when its oracle score is within tolerance of the
            k-th score.
"""
import numpy as np
import torch

import oracle
import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W

REL_TOL = 1e-3
ABS_TOL = 1e-6


def run_path(wl, num_sms=None, use_indices=True, logits_out=None, groups_for_keys=True):
    """metadata -> logits -> top-k on cuda:0; returns a dict of device tensors.

    groups_for_keys: the schedule's groups sized for the workload's key
    format (else the 8-row groups of the plain metadata call)."""
    dev = torch.device("cuda")
    g = wl if wl.q.is_cuda else wl.to(dev)
    ind = g.indices if use_indices else None
    if num_sms is None:
        num_sms = dsa.device_num_sms()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sched = dsa.paged_mqa_logits_metadata(g.context_lens, ind, num_sms,
                                          kv_format=g.kv_format if groups_for_keys else None)
    logits = dsa.fp8_fp4_paged_mqa_logits(
        g.q, g.kv_cache, g.weights, g.context_lens, g.block_table, sched, indices=ind,
        kv_format=g.kv_format, logits_dtype=g.logits_dtype, logits_stride=g.logits_stride,
        num_sms=num_sms, status=status, out=logits_out, q_scale=g.q_scale)
    idx = dsa.top_k_per_row(logits, None, g.context_lens, g.topk, status=status)
    torch.cuda.synchronize()
    return dict(sched=sched, logits=logits, idx=idx, status=status, num_sms=num_sms, dev_wl=g)


def logits_tolerance(bound, ref, bf16):
    tol = REL_TOL * bound + ABS_TOL
    if bf16:
        tol = tol + 2.0 ** -9 * (np.abs(ref) + tol)
    return tol


def check_logits(wl, gpu_logits, rows=None, ref=None, bound=None):
    """Element-wise comparison of GPU logits with the oracle on the given rows."""
    T = wl.num_rows
    rows = list(range(T)) if rows is None else list(rows)
    if ref is None:
        ref, bound = oracle.workload_logits(wl, rows=np.array(rows, dtype=np.int32))
    g = gpu_logits[rows].float().cpu().double().numpy()
    ctx = wl.context_lens.cpu().numpy()
    bf16 = gpu_logits.dtype == torch.bfloat16
    worst = 0.0
    for i, t in enumerate(rows):
        L = int(ctx[t])
        if L > 0:
            tol = logits_tolerance(bound[i, :L], ref[i, :L], bf16)
            err = np.abs(g[i, :L] - ref[i, :L])
            bad = np.nonzero(~(err <= tol))[0]
            assert bad.size == 0, (
                f"row {t}: {bad.size} columns off, first {bad[:5]} gpu={g[i, bad[:5]]} "
                f"ref={ref[i, bad[:5]]} tol={tol[bad[:5]]}")
            worst = max(worst, float(np.max(err / tol)))
        pad_end = (L + 63) // 64 * 64
        assert np.all(np.isneginf(g[i, L:pad_end])), f"row {t}: columns past L_t not -inf"
    return ref, bound, worst


def check_topk_exact(gpu_logits, gpu_idx, ctx, k, rows=None):
    """GPU top-k equals the oracle top-k of the same GPU logits, bit for bit."""
    rows = list(range(gpu_logits.shape[0])) if rows is None else list(rows)
    sc = gpu_logits[rows].float().cpu().double().numpy()
    ends = ctx.cpu().numpy()[rows]
    cpu = oracle.top_k_per_row(sc, ends, k)
    got = gpu_idx[rows].cpu().numpy()
    mism = np.nonzero(np.any(cpu != got, axis=1))[0]
    assert mism.size == 0, f"rows {np.array(rows)[mism[:5]]} differ from the oracle top-k"


def check_topk_tie_band(gpu_idx, ref, bound, ctx, k, rows):
    """GPU top-k against the oracle's top-k of the oracle logits, up to the tie band."""
    ends = ctx.cpu().numpy()[list(rows)]
    ref_idx = oracle.top_k_per_row(ref, ends, k)
    got = gpu_idx[list(rows)].cpu().numpy()
    for i in range(len(rows)):
        a = set(ref_idx[i][ref_idx[i] >= 0].tolist())
        b = set(got[i][got[i] >= 0].tolist())
        assert len(a) == len(b)
        diff = a ^ b
        if not diff:
            continue
        L = int(ends[i])
        vals = ref[i, :L]
        kth_col = sorted(a, key=lambda s: (-vals[s], s))[-1]
        kth = vals[kth_col]
        tol_k = REL_TOL * bound[i, kth_col] + ABS_TOL
        for s in diff:
            tol_s = REL_TOL * bound[i, s] + ABS_TOL
            assert abs(vals[s] - kth) <= tol_s + tol_k, (rows[i], s, vals[s], kth)


def sample_rows(T, n, seed=0):
    rng = np.random.default_rng(seed)
    if T <= n:
        return list(range(T))
    pick = set(rng.choice(T, size=n - 2, replace=False).tolist()) | {0, T - 1}
    return sorted(pick)
