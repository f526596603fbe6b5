"""GPU parity of the indexer decode path against the CPU oracle, through the
C ABI (binding -> libdsa_indexer.so), on seeded synthetic inputs.

Small cases run the oracle on every row (several tiles, ragged tails, groups
longer than 8 rows, empty rows); the full-size decode workloads compare every
row's logits element by element with the oracle, every row's top-k bit for
bit with the oracle's top-k of the GPU logits, and every row's top-k with the
oracle's top-k of the oracle logits up to the tie band."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_paged_gb300 as dsa
import workloads as W
from gpu_helpers import check_logits, check_topk_exact, check_topk_tie_band, logits_tolerance, run_path
from schedule_check import check_schedule

pytestmark = pytest.mark.gpu

MIXED = dict(request_lens=[1, 63, 64, 65, 127, 128, 129, 300, 1000, 2500],
             rows_per_request=[1, 2, 1, 3, 1, 6, 8, 2, 4, 11])


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    dsa.build()
    dsa.lib()


def _full_check(wl, num_sms=None, use_indices=True, groups_for_keys=True):
    out = run_path(wl, num_sms=num_sms, use_indices=use_indices, groups_for_keys=groups_for_keys)
    assert int(out["status"].item()) == 0, dsa.status_string(int(out["status"].item()))
    ref, bound, worst = check_logits(wl, out["logits"])
    check_topk_exact(out["logits"], out["idx"], wl.context_lens, wl.topk)
    check_topk_tie_band(out["idx"], ref, bound, wl.context_lens, wl.topk, list(range(wl.num_rows)))
    return out, worst


# ---------------------------------------------------------------- metadata
# The pages fix the metadata call's inputs and purpose, not its split rule, so
# its words are checked for validity and balance (schedule_check), and the
# logits below are compared with the oracle at several SM counts.

@pytest.mark.parametrize("name", ["tiny", "plain", "mtp", "varlen"])
def test_metadata_valid(name):
    ctx, ind = W.config_rows(name)
    for S in (1, 7, 148, dsa.device_num_sms(), 1023):
        for use_ind in (True, False):
            ids = ind if use_ind else None
            got = dsa.paged_mqa_logits_metadata(ctx.cuda(), None if ids is None else ids.cuda(), S)
            check_schedule(got.cpu().numpy(), ctx.numpy(), None if ids is None else ids.numpy(), S)


def test_metadata_ragged_groups():
    wl = W.build("mixed", **MIXED, topk=64)
    for S in (1, 3, 5, 64, 152):
        got = dsa.paged_mqa_logits_metadata(wl.context_lens.cuda(), wl.indices.cuda(), S)
        check_schedule(got.cpu().numpy(), wl.context_lens.numpy(), wl.indices.numpy(), S)


@pytest.mark.parametrize("kv_format,cap", [(W.KV_FP8, 8), (W.KV_FP4, 4), (W.KV_MXFP4, 6)])
def test_metadata_groups_for_keys(kv_format, cap):
    """Groups sized for the key format's row pass: the header records the
    size, and every group is at most that size and cut only where full."""
    wl = W.build("mixed", **MIXED, topk=64)
    ctx, ids = wl.context_lens.numpy(), wl.indices.numpy()
    for S in (1, 5, 152):
        got = dsa.paged_mqa_logits_metadata(wl.context_lens.cuda(), wl.indices.cuda(), S,
                                            kv_format=kv_format).cpu().numpy()
        assert got[7] == cap
        check_schedule(got, ctx, ids, S)


@pytest.mark.parametrize("requests", [450, 900])
def test_metadata_long_batch(requests):
    """More rows than one CTA pass (chunked scans), random run lengths and zero-length rows."""
    rng = np.random.default_rng(5)
    ctx, ids = [], []
    for r in range(requests):
        n = int(rng.integers(1, 14))
        L = int(rng.integers(0, 3000))
        for j in range(n):
            ctx.append(max(0, L - n + 1 + j))
            ids.append(r)
    ctx = np.array(ctx, dtype=np.int32)
    ids = np.array(ids, dtype=np.int32)
    for S in (1, 148, 1023):
        got = dsa.paged_mqa_logits_metadata(torch.from_numpy(ctx).cuda(), torch.from_numpy(ids).cuda(), S)
        check_schedule(got.cpu().numpy(), ctx, ids, S)


@pytest.mark.parametrize("T", [1023, 1024, 1025, 4097])
def test_metadata_chunk_boundaries(T):
    rng = np.random.default_rng(T)
    ctx = rng.integers(0, 5000, T).astype(np.int32)
    for ids in (None, (np.arange(T) // 3).astype(np.int32)):
        for S in (7, 152):
            got = dsa.paged_mqa_logits_metadata(torch.from_numpy(ctx).cuda(),
                                                None if ids is None else torch.from_numpy(ids).cuda(), S)
            check_schedule(got.cpu().numpy(), ctx, ids, S)


def test_metadata_skewed_group_sizes():
    """Many full 8-row groups and a few 1-row groups, and the reverse: the
    balance holds when one end of the row-count order dominates."""
    rng = np.random.default_rng(9)
    for heavy in (True, False):
        ctx, ids = [], []
        for r in range(60):
            n = 8 if (r % 10 != 0) == heavy else 1
            L = int(rng.integers(2000, 40000))
            for j in range(n):
                ctx.append(L - n + 1 + j)
                ids.append(r)
        ctx = np.array(ctx, dtype=np.int32)
        ids = np.array(ids, dtype=np.int32)
        for S in (13, 152):
            got = dsa.paged_mqa_logits_metadata(torch.from_numpy(ctx).cuda(), torch.from_numpy(ids).cuda(), S)
            check_schedule(got.cpu().numpy(), ctx, ids, S)


# ---------------------------------------------------------------- logits + top-k, small

def test_tiny_config():
    _full_check(W.config("tiny"))


def test_mixed_ragged():
    _full_check(W.build("mixed", **MIXED, topk=64, seed=1))


@pytest.mark.parametrize("S", [1, 5, 37])
def test_mixed_any_sm_split(S):
    _full_check(W.build("mixed", **MIXED, topk=256, seed=2), num_sms=S)


def test_plain_decode_equals_arange():
    kw = dict(request_lens=[700, 1, 130, 4097, 64], rows_per_request=[1] * 5, topk=128, seed=3)
    a = run_path(W.build("arange", **kw))
    b = run_path(W.build("plain", plain_indices=True, **kw), use_indices=False)
    for t, L in enumerate(kw["request_lens"]):      # the specified span of each row
        end = (L + 63) // 64 * 64
        assert torch.equal(a["logits"][t, :end], b["logits"][t, :end]), t
    assert torch.equal(a["idx"], b["idx"])
    check_logits(W.build("plain", plain_indices=True, **kw), b["logits"])


def test_varlen_equals_padded():
    """Varlen rows give the logits of a (B, max_n) padded batch on its valid rows."""
    wl = W.build("v", request_lens=[900, 333, 1500], rows_per_request=[3, 1, 5], topk=64, seed=4)
    slot_row, max_n = W.padded_rows(wl)
    src = []
    t = 0
    for n in wl.rows_per_request:
        for j in range(max_n):
            src.append(t + min(j, n - 1))
        t += n
    src = torch.tensor(src)
    pad = W.Workload(**{**wl.__dict__})
    pad.q, pad.weights = wl.q[src], wl.weights[src]
    pad.context_lens, pad.block_table = wl.context_lens[src], wl.block_table[src]
    pad.indices = None
    a = run_path(wl)
    b = run_path(pad, use_indices=False)
    valid = (slot_row >= 0).nonzero().flatten()
    la = a["logits"][slot_row[valid]]
    lb = b["logits"][valid]
    check_logits(wl, a["logits"])
    check_logits(pad, b["logits"])
    ctx = wl.context_lens[slot_row[valid]]
    for i in range(la.shape[0]):                    # the specified span of each row
        end = (int(ctx[i]) + 63) // 64 * 64
        fin = torch.isfinite(la[i, :end])
        assert torch.equal(fin, torch.isfinite(lb[i, :end]))
        assert torch.allclose(la[i, :end][fin], lb[i, :end][fin], rtol=1e-5, atol=1e-5)


def test_padded_page_stride():
    _full_check(W.build("stride", request_lens=[777, 2048], rows_per_request=[2, 3], topk=100,
                        page_stride=8704, seed=5))


def test_bf16_logits_fp8_keys():
    _full_check(W.build("bf16", **MIXED, topk=64, logits_dtype=W.LOGITS_BF16, seed=6))


def test_zero_length_and_short_rows():
    wl = W.build("short", request_lens=[0, 5, 64, 0], rows_per_request=[1, 1, 1, 1], topk=16,
                 seed=7)
    out = run_path(wl)
    assert int(out["status"].item()) == 0
    check_logits(wl, out["logits"])
    idx = out["idx"].cpu()
    assert torch.equal(idx[0], torch.full((16,), -1, dtype=torch.int32))
    assert idx[1, :5].tolist() == [0, 1, 2, 3, 4] and torch.all(idx[1, 5:] == -1)
    check_topk_exact(out["logits"], out["idx"], wl.context_lens, 16)


def test_empty_batch():
    dev = torch.device("cuda")
    ctx = torch.zeros(0, dtype=torch.int32, device=dev)
    sched = dsa.paged_mqa_logits_metadata(ctx, None, 8)
    assert sched.cpu()[:8].tolist() == [0x44534132, 0, 0, 8, 0, 0, 128, 8]
    check_schedule(sched.cpu().numpy(), np.zeros(0, np.int32), None, 8)
    lg = torch.empty((0, 64), device=dev)
    out = dsa.top_k_per_row(lg, None, ctx, 8)
    assert out.shape == (0, 8)


# ---------------------------------------------------------------- device faults (reported, never hang)

def test_bad_block_id_reported():
    wl = W.build("bad", request_lens=[300], rows_per_request=[1], topk=8, seed=8)
    wl.block_table[0, 2] = wl.num_pages + 5
    out = run_path(wl)
    assert int(out["status"].item()) == dsa.DSA_ERR_BAD_BLOCK


def test_schedule_mode_mismatch_reported():
    """A varlen schedule used by a plain call: the kpool fault class, caught."""
    wl = W.build("mm", request_lens=[300, 200], rows_per_request=[2, 1], topk=8, seed=9).to("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    S = dsa.device_num_sms()
    sched = dsa.paged_mqa_logits_metadata(wl.context_lens, wl.indices, S)
    dsa.fp8_fp4_paged_mqa_logits(wl.q, wl.kv_cache, wl.weights, wl.context_lens, wl.block_table,
                                 sched, indices=None, logits_stride=wl.logits_stride, num_sms=S,
                                 status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == dsa.DSA_ERR_SCHEDULE_MISMATCH
    st.zero_()
    dsa.fp8_fp4_paged_mqa_logits(wl.q, wl.kv_cache, wl.weights, wl.context_lens, wl.block_table,
                                 sched, indices=wl.indices, logits_stride=wl.logits_stride,
                                 num_sms=S - 1, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == dsa.DSA_ERR_SCHEDULE_MISMATCH


# ---------------------------------------------------------------- top-k on its own

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_topk_standalone(dtype):
    g = torch.Generator().manual_seed(11)
    R, C = 12, 40000
    x = torch.randn((R, C), generator=g)
    x[1] = torch.round(x[1] * 2)           # heavy ties
    x[2, 5000:] = float("-inf")
    x[3, ::9] = float("nan")
    x[4] = 0.0
    x[4, ::2] = -0.0
    x[5, :] = torch.arange(C, dtype=torch.float32)   # strictly increasing
    x = x.to(dtype).cuda()
    ends = torch.tensor([C, C, C, C, C, C, 1, 0, 2047, 2049, 30001, 17], dtype=torch.int32)
    starts = torch.tensor([0, 3, 0, 7, 0, 1000, 0, 0, 0, 0, 5, 0], dtype=torch.int32)
    for k in (1, 7, 256, 2048):
        got = dsa.top_k_per_row(x, starts.cuda(), ends.cuda(), k).cpu().numpy()
        ref = oracle.top_k_per_row(x.float().cpu().double().numpy(), ends, k, row_starts=starts)
        assert np.array_equal(got, ref), k


@pytest.mark.parametrize("C", [5000, 8192, 16384])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_topk_short_rows(C, dtype):
    """Row strides of at most 16384 columns take the short-row kernel."""
    g = torch.Generator().manual_seed(C)
    R = 14
    x = torch.randn((R, C), generator=g) * 3
    x[1] = torch.round(x[1] * 2)           # heavy ties
    x[2, C // 3:] = float("-inf")
    x[3, ::9] = float("nan")
    x[4] = 0.0
    x[4, ::2] = -0.0
    x[5, :] = torch.arange(C, dtype=torch.float32)
    x[12] = 1.5                            # every key equal
    x[13, :] = torch.randn(C, generator=g) * 1e-30  # tiny magnitudes, both signs
    x = x.to(dtype).cuda()
    ends = torch.tensor([C, C, C, C, C, C, 1, 0, 2047, 2049, C - 3, 17, C, C], dtype=torch.int32)
    starts = torch.tensor([0, 3, 0, 7, 0, 1000, 0, 0, 0, 0, 5, 0, 2, 0], dtype=torch.int32)
    for k in (1, 7, 256, 2048):
        got = dsa.top_k_per_row(x, starts.cuda(), ends.cuda(), k).cpu().numpy()
        ref = oracle.top_k_per_row(x.float().cpu().double().numpy(), ends, k, row_starts=starts)
        assert np.array_equal(got, ref), k
        got = dsa.top_k_per_row(x, None, ends.cuda(), k).cpu().numpy()
        assert np.array_equal(got, oracle.top_k_per_row(x.float().cpu().double().numpy(), ends, k)), k


# ---------------------------------------------------------------- full-size workloads, every row

def _full_size_every_row(name):
    """The configuration's whole step in the launch configuration bench.py
    times (every SM, the schedule from the metadata call): all rows, all
    columns of the logits against the oracle, then both top-k checks."""
    wl = W.config(name, device="cuda")
    out = run_path(wl)
    assert int(out["status"].item()) == 0, dsa.status_string(int(out["status"].item()))
    host = wl.to("cpu")
    ref, bound, _ = check_logits(host, out["logits"])
    check_topk_exact(out["logits"], out["idx"], host.context_lens, wl.topk)
    check_topk_tie_band(out["idx"], ref, bound, host.context_lens, wl.topk, list(range(wl.num_rows)))


@pytest.mark.parametrize("name", ["plain", "mtp", "varlen"])
def test_full_size_every_row(name):
    _full_size_every_row(name)


def test_topk_long_row_general_path():
    """A row longer than the shared-memory bitmaps takes the general path."""
    g = torch.Generator().manual_seed(12)
    x = torch.randn((2, 300032), generator=g)
    x[1, 100000:] = torch.round(x[1, 100000:])
    x = x.cuda()
    ends = torch.tensor([300032, 290001], dtype=torch.int32)
    starts = torch.tensor([0, 17], dtype=torch.int32)
    for k in (5, 2048):
        got = dsa.top_k_per_row(x, starts.cuda(), ends.cuda(), k).cpu().numpy()
        ref = oracle.top_k_per_row(x.cpu().double().numpy(), ends, k, row_starts=starts)
        assert np.array_equal(got, ref), k


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_topk_sampled_path_boundary(dtype):
    """Rows of 2^18 - 1, 2^18 and 2^18 + 1 columns: the last one no longer fits
    the sampled path's bitmaps and takes the exact passes; the stride 16384 + 8
    also sits just above the short-row kernel's largest stride."""
    g = torch.Generator().manual_seed(13)
    C = (1 << 18) + 8
    x = torch.randn((4, C), generator=g)
    x[3] = torch.round(x[3] * 4)                # heavy ties across the whole row
    x = x.to(dtype).cuda()
    ends = torch.tensor([(1 << 18) - 1, 1 << 18, (1 << 18) + 1, C], dtype=torch.int32)
    for k in (1, 2048):
        got = dsa.top_k_per_row(x, None, ends.cuda(), k).cpu().numpy()
        ref = oracle.top_k_per_row(x.float().cpu().double().numpy(), ends, k)
        assert np.array_equal(got, ref), k
    x2 = x[:, :16392].contiguous()              # stride 16392: the long-row kernel on short rows
    ends2 = torch.tensor([16392, 9000, 2049, 1], dtype=torch.int32)
    got = dsa.top_k_per_row(x2, None, ends2.cuda(), 2048).cpu().numpy()
    assert np.array_equal(got, oracle.top_k_per_row(x2.float().cpu().double().numpy(), ends2, 2048))


@pytest.mark.parametrize("C", [40000, 131072, 131080])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_topk_more_rows_than_sms(C, dtype):
    """More rows than SMs with strides up to 2^17 take the two-rows-per-SM
    geometry (2^17 + 8 keeps the one-row geometry): special rows as in the
    short-row test, plus rows of random lengths up to the stride."""
    S = dsa.device_num_sms()
    R = S + 48
    g = torch.Generator().manual_seed(C + R)
    x = torch.randn((R, C), generator=g)
    x[1] = torch.round(x[1] * 2)           # heavy ties: the sample's candidates overflow
    x[2, C // 3:] = float("-inf")
    x[3, ::9] = float("nan")
    x[4] = 0.0
    x[4, ::2] = -0.0
    x[5, :] = torch.arange(C, dtype=torch.float32)
    x[12] = 1.5                            # every key equal
    x[13, :] = torch.randn(C, generator=g) * 1e-30
    x[14, ::37] = float("inf")             # +inf among finite scores
    x[15, :] = torch.randn(C, generator=g) * 1e-39   # subnormal fp32 magnitudes
    x[16, :] = float("nan")                # NaN-dominated: the sample threshold falls to NaN
    x[16, ::13] = torch.randn(C // 13 + 1, generator=g)[: x[16, ::13].numel()]
    x[17, :] = float("-inf")               # -inf everywhere but a few columns
    x[17, ::501] = torch.randn(x[17, ::501].numel(), generator=g)
    x = x.to(dtype).cuda()
    ends = torch.randint(0, C + 1, (R,), generator=g, dtype=torch.int32)
    ends[:18] = torch.tensor([C, C, C, C, C, C, 1, 0, 2047, 2049, C - 3, 17, C, C, C, C, C, C],
                             dtype=torch.int32)
    starts = torch.randint(0, 4000, (R,), generator=g, dtype=torch.int32)
    starts[:18] = torch.tensor([0, 3, 0, 7, 0, 1000, 0, 0, 0, 0, 5, 0, 2, 0, 0, 9, 0, 1], dtype=torch.int32)
    host = x.float().cpu().double().numpy()
    for k in (7, 2048):
        got = dsa.top_k_per_row(x, starts.cuda(), ends.cuda(), k).cpu().numpy()
        assert np.array_equal(got, oracle.top_k_per_row(host, ends, k, row_starts=starts)), k


# ---------------------------------------------------------------- FP4 keys (e2m1 + e4m3/16 + fp32/token)

@pytest.mark.parametrize("logits_dtype", [W.LOGITS_F32, W.LOGITS_BF16])
def test_fp4_mixed_ragged(logits_dtype):
    _full_check(W.build("fp4", **MIXED, topk=64, kv_format=W.KV_FP4, logits_dtype=logits_dtype,
                        seed=13))


def test_fp4_with_8_row_groups():
    """The FP4 call on a schedule built for 8-row groups (several row passes
    a group) gives the oracle's logits too."""
    _full_check(W.build("fp4", **MIXED, topk=64, kv_format=W.KV_FP4, seed=13), groups_for_keys=False)


@pytest.mark.parametrize("S", [1, 7])
def test_fp4_any_sm_split(S):
    _full_check(W.build("fp4s", request_lens=[700, 129, 1500], rows_per_request=[3, 8, 5], topk=128,
                        kv_format=W.KV_FP4, seed=14), num_sms=S)


def test_fp4_padded_page_stride():
    _full_check(W.build("fp4p", request_lens=[333, 1024], rows_per_request=[2, 4], topk=100,
                        kv_format=W.KV_FP4, page_stride=4864 + 16 * 9, seed=15))


def test_fp4_full_size_every_row():
    _full_size_every_row("fp4_varlen")


# ---------------------------------------------------------------- MXFP4 keys and q

@pytest.mark.parametrize("logits_dtype", [W.LOGITS_F32, W.LOGITS_BF16])
def test_mxfp4_mixed_ragged(logits_dtype):
    _full_check(W.build("mxfp4", **MIXED, topk=64, kv_format=W.KV_MXFP4, logits_dtype=logits_dtype,
                        seed=41))


def test_mxfp4_with_8_row_groups():
    """The MXFP4 call on a schedule built for 8-row groups gives the oracle's logits too."""
    _full_check(W.build("mxfp4", **MIXED, topk=64, kv_format=W.KV_MXFP4, seed=41), groups_for_keys=False)


@pytest.mark.parametrize("S", [1, 7])
def test_mxfp4_any_sm_split(S):
    _full_check(W.build("mxfp4", [700, 1300], [3, 5], topk=128, kv_format=W.KV_MXFP4, seed=42), num_sms=S)


def test_mxfp4_padded_page_stride():
    _full_check(W.build("mxfp4", [500, 90], [2, 1], topk=32, kv_format=W.KV_MXFP4,
                        page_stride=4352 + 16 * 5, seed=43))


def test_mxfp4_block_scales_far_below_the_largest():
    """Blocks 2^12 and 2^20 below their token's or row's largest scale: the
    block-scaled MMA applies each block's powers of two exactly."""
    wl = W.build("mxfp4", [300, 517], [2, 3], topk=64, kv_format=W.KV_MXFP4, seed=44)
    es = W._page_views(wl.kv_cache, W.KV_MXFP4)["bscale"]          # [pages, 64, 4] ue8m0
    ok = es != W.UE8M0_NAN
    es[..., 1] = torch.where(ok[..., 1], (es[..., 1].int() - 12).clamp(min=0).to(torch.uint8), es[..., 1])
    es[::2, :, 3] = torch.where(ok[::2, :, 3], (es[::2, :, 3].int() - 20).clamp(min=0).to(torch.uint8),
                                es[::2, :, 3])
    wl.q_scale[:, ::3, 2] = (wl.q_scale[:, ::3, 2].int() - 12).clamp(min=0).to(torch.uint8)
    wl.q_scale[:, 1::5, 0] = (wl.q_scale[:, 1::5, 0].int() - 20).clamp(min=0).to(torch.uint8)
    _full_check(wl)


def test_mxfp4_nan_scale_gives_non_finite_logit():
    """A NaN block scale (ue8m0 code 255, OCP MX) on a live key block or on one
    head's q block makes exactly the logits whose dot product it enters
    non-finite, as in the oracle (whose ReLU keeps the NaN); every other logit
    matches the oracle."""
    wl = W.build("mxfp4", [300, 517], [2, 3], topk=64, kv_format=W.KV_MXFP4, seed=45)
    es = W._page_views(wl.kv_cache, W.KV_MXFP4)["bscale"]   # [pages, 64, 4] ue8m0
    # key token 70 of row 0's table (its second page, slot 6), block 2
    es[int(wl.block_table[0, 1]), 6, 2] = W.UE8M0_NAN
    # q of row 3 (the second request), head 5, block 0
    wl.q_scale[3, 5, 0] = W.UE8M0_NAN
    out = run_path(wl)
    assert int(out["status"].item()) == 0, dsa.status_string(int(out["status"].item()))
    ref, bound = oracle.workload_logits(wl)
    g = out["logits"].float().cpu().double().numpy()
    ctx = wl.context_lens.cpu().numpy()
    planted = 0
    for t in range(wl.num_rows):
        L = int(ctx[t])
        bad_ref = ~np.isfinite(ref[t, :L])
        assert np.array_equal(~np.isfinite(g[t, :L]), bad_ref), f"row {t}: non-finite columns differ"
        planted += int(bad_ref.sum())
        ok = np.nonzero(~bad_ref)[0]
        tol = logits_tolerance(bound[t, ok], ref[t, ok], out["logits"].dtype == torch.bfloat16)
        assert np.all(np.abs(g[t, ok] - ref[t, ok]) <= tol), f"row {t}: finite logits off"
    # row 3's every column, and column 70 of the two rows of request 0
    assert planted >= int(ctx[3]) + 2, planted


def test_mxfp4_full_size_every_row():
    _full_size_every_row("mxfp4_varlen")


# ---------------------------------------------------------------- CUDA graphs

def test_step_replays_from_a_cuda_graph():
    """The three calls allocate, free and synchronise nothing, so a decode
    step captures into a CUDA graph; replaying it after the inputs change in
    place gives the direct run's results for the new inputs."""
    wl = W.build("graph", **MIXED, topk=64, seed=51).to("cuda")
    S = dsa.device_num_sms()
    sched = torch.empty(dsa.schedule_words(S, wl.num_rows), dtype=torch.int32, device="cuda")
    logits = torch.empty((wl.num_rows, wl.logits_stride), dtype=torch.float32, device="cuda")
    idx = torch.empty((wl.num_rows, wl.topk), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, w = wl.q.clone(), wl.weights.clone()

    def step():
        dsa.paged_mqa_logits_metadata(wl.context_lens, wl.indices, S, out=sched)
        dsa.fp8_fp4_paged_mqa_logits(q, wl.kv_cache, w, wl.context_lens, wl.block_table, sched,
                                     indices=wl.indices, logits_stride=wl.logits_stride, num_sms=S,
                                     out=logits, status=st)
        dsa.top_k_per_row(logits, None, wl.context_lens, wl.topk, out=idx, status=st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    first = idx.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="relaxed"):
        step()
    q.copy_(torch.roll(wl.q, 1, dims=0))         # new inputs, same buffers
    w.copy_(wl.weights * 2.0 - 0.1)
    idx.zero_()
    graph.replay()
    torch.cuda.synchronize()
    replayed = idx.clone()
    step()                                        # the same step launched directly
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(replayed, idx)
    assert not torch.equal(replayed, first)
