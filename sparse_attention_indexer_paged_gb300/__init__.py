"""Python binding of libdsa_indexer (the GB300 DSA indexer decode path).

Thin ctypes layer over the C ABI of ``include/dsa_indexer.h``: it only turns
torch tensors into pointers, sizes and the current CUDA stream, and allocates
outputs the caller did not pass (torch is used for device memory and streams
only).  Every step of the path runs in the library's kernels; there is no
fallback.  If the library has not been built, every call raises.

Decode step (the three calls of the C ABI):

    sched  = paged_mqa_logits_metadata(context_lens, indices, num_sms)
    logits = fp8_fp4_paged_mqa_logits(q, kv_cache, weights, context_lens,
                                      block_table, sched, indices=indices)
    idx    = top_k_per_row(logits, None, context_lens, k)

The same step as one native call, optionally in row slices whose logits fit a
byte budget:

    idx = indexer_decode_topk(q, kv_cache, weights, context_lens, block_table,
                              k, indices=indices, logits_budget=16 << 20)

MXFP4 keys and q (kv_format=KV_MXFP4; q packed e2m1 with ue8m0 q_scale):

    logits = fp8_fp4_paged_mqa_logits(..., kv_format=KV_MXFP4, q_scale=q_scale)

Prefill rows tagged (cu_seqlen_ks, cu_seqlen_ke), straight from the paged
cache with a block table per request:

    idx, logits = prefill_topk(q, kv_cache, weights, cu_seqlen_ks, cu_seqlen_ke,
                               local_cu_seq_lens, block_table, k)

Decode context parallelism (this rank's shard of every request's keys; the
gather goes through torch.distributed):

    idx = dcp_topk(logits, local_idx, k, rank, world, interleave)

Every call is stream-ordered on the current CUDA stream and allocates,
frees and synchronises nothing inside the library, so a step can be
captured into a CUDA graph.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB_PATH, build  # noqa: F401

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_SCHEDULE_MISMATCH = 3
DSA_ERR_CUDA = 4
DSA_ERR_BAD_BLOCK = 5
DSA_ERR_TIMEOUT = 6
DSA_ERR_NO_DEVICE = 7
DSA_ERR_SCRATCH_TOO_SMALL = 8

KV_FP8 = 0
KV_FP4 = 1
KV_MXFP4 = 2
LOGITS_F32 = 0
LOGITS_BF16 = 1

BLOCK_KV = 64
NUM_HEADS = 64
HEAD_DIM = 128
FP8_PAGE_BYTES = 8448
FP4_PAGE_BYTES = 4864
MXFP4_PAGE_BYTES = 4352
MAX_TOPK = 2048
# fixed device scratch of indexer_decode_topk_static
STATIC_SCHEDULE_WORDS = 16384
STATIC_LOGITS_BYTES = 8 << 20

# C entry points and their argument types
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_SIGS = {
    "dsa_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "dsa_version": ([], ctypes.c_int),
    "dsa_schedule_words": ([_I32, _I32], _I64),
    "dsa_device_num_sms": ([], _I32),
    "dsa_paged_mqa_logits_metadata": ([_P, _P, _I32, _I32, _I32, _P, _P], ctypes.c_int),
    "dsa_paged_mqa_logits_metadata_for_keys": ([_P, _P, _I32, _I32, _I32, _I32, _P, _P], ctypes.c_int),
    "dsa_fp8_fp4_paged_mqa_logits": ([_P, _P, _I64, _I64, _I32, _P, _P, _P, _I64, _P, _P, _I32,
                                      _P, _I32, _I64, _I32, _I32, _I32, _I32, _P, _P],
                                     ctypes.c_int),
    "dsa_top_k_per_row": ([_P, _I32, _I64, _P, _P, _I32, _I32, _P, _I64, _P, _P], ctypes.c_int),
    "dsa_selftest_wait_timeout": ([_I64, _P, _P], ctypes.c_int),
    "dsa_dcp_pack_topk": ([_P, _I32, _I64, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P], ctypes.c_int),
    "dsa_dcp_merge_topk": ([_P, _I32, _I32, _I32, _P, _I64, _P], ctypes.c_int),
    "dsa_prefill_rows": ([_P, _P, _I32, _P, _I32, _P, _P, _P, _P], ctypes.c_int),
    "dsa_mxfp4_paged_mqa_logits": ([_P, _P, _P, _I64, _I64, _P, _P, _P, _I64, _P, _P, _I32, _P, _I32, _I64,
                                    _I32, _I32, _I32, _I32, _P, _P], ctypes.c_int),
    "dsa_prefill_mqa_logits": ([_P, _P, _P, _I64, _I64, _I32, _P, _P, _P, _P, _I64, _I32, _P, _I32, _P,
                                _I32, _I64, _I32, _I32, _I32, _I32, _P, _P], ctypes.c_int),
    "dsa_decode_chunk_ranges": ([_I64, _I64, _I64, _P, _I32, _P], ctypes.c_int),
    "dsa_indexer_decode_scratch": ([_I32, _I32, _I64, _I64, _I32, _P, _P], ctypes.c_int),
    "dsa_indexer_decode_topk": ([_P, _P, _P, _I64, _I64, _I32, _P, _P, _P, _I64, _P, _I32, _I32, _I32,
                                 _I32, _I32, _I32, _I64, _I64, _P, _I64, _P, _I64, _I32, _P, _I64,
                                 _P, _P], ctypes.c_int),
    "dsa_indexer_decode_topk_static": ([_P, _P, _P, _I64, _I64, _I32, _P, _P, _P, _I64, _P, _I32, _I32, _I32,
                                        _I32, _I32, _I32, _I64, _I32, _P, _I64, _P, _P], ctypes.c_int),
}
EXPORTED = tuple(_SIGS)

_lib = None


class DsaError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib().dsa_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{what}: {msg} (status {code})")
        self.code = code


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdsa_indexer is not built ({LIB_PATH}); "
                               "run __graft_entry__.build() or "
                               "sparse_attention_indexer_paged_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(code: int, what: str):
    if code != DSA_OK:
        raise DsaError(code, what)


def _dev_i32(x, device):
    if x is None:
        return None
    if not torch.is_tensor(x):
        x = torch.as_tensor(x)
    return x.to(device=device, dtype=torch.int32).contiguous()


def status_string(code: int) -> str:
    return lib().dsa_status_string(int(code)).decode()


def device_num_sms() -> int:
    n = lib().dsa_device_num_sms()
    if n < 0:
        raise DsaError(-n, "dsa_device_num_sms")
    return int(n)


def schedule_words(num_sms: int, num_rows: int) -> int:
    return int(lib().dsa_schedule_words(int(num_sms), int(num_rows)))


def paged_mqa_logits_metadata(context_lens, indices=None, num_sms=None, block_kv=BLOCK_KV,
                              out=None, kv_format=None):
    """Per-SM work schedule (int32 device tensor) for the logits call.

    kv_format None: groups of up to 8 rows (dsa_paged_mqa_logits_metadata);
    KV_FP8 / KV_FP4 / KV_MXFP4: groups sized for that key format's logits
    call (dsa_paged_mqa_logits_metadata_for_keys)."""
    ctx = context_lens
    device = ctx.device
    T = int(ctx.shape[0])
    if num_sms is None:
        num_sms = device_num_sms()
    words = schedule_words(num_sms, T)
    if out is None:
        out = torch.empty(words, dtype=torch.int32, device=device)
    assert out.dtype == torch.int32 and out.is_contiguous() and out.numel() >= words
    ctx = _dev_i32(ctx, device)
    ind = _dev_i32(indices, device)
    if kv_format is None:
        _check(lib().dsa_paged_mqa_logits_metadata(_ptr(ctx), _ptr(ind), T, int(block_kv),
                                                   int(num_sms), _ptr(out), _stream(device)),
               "paged_mqa_logits_metadata")
    else:
        _check(lib().dsa_paged_mqa_logits_metadata_for_keys(_ptr(ctx), _ptr(ind), T, int(block_kv),
                                                            int(num_sms), int(kv_format), _ptr(out),
                                                            _stream(device)),
               "paged_mqa_logits_metadata_for_keys")
    return out


def fp8_fp4_paged_mqa_logits(q, kv_cache, weights, context_lens, block_table, schedule,
                             indices=None, kv_format=KV_FP8, logits_dtype=LOGITS_F32,
                             logits_stride=None, num_sms=None, out=None, status=None,
                             page_stride=None, q_scale=None):
    """Varlen paged MQA logits [num_rows, logits_stride] (fp32 or bf16).

    q [T, 64, 128] e4m3 codes (uint8 or float8_e4m3fn); kv_cache [num_pages,
    page_stride] uint8 pages; weights [T, 64] fp32; context_lens [T];
    block_table [T, max_pages] int32; schedule from paged_mqa_logits_metadata.
    Columns >= round_up(L_t, 64) of a row are not specified.  MXFP4 keys
    (kv_format=KV_MXFP4) take MXFP4 q: packed e2m1 [T, 64, 64] and q_scale
    ue8m0 [T, 64, 4].
    """
    device = q.device
    T = int(q.shape[0])
    if num_sms is None:
        num_sms = device_num_sms()
    ctx = _dev_i32(context_lens, device)
    bt = _dev_i32(block_table, device)
    if bt.dim() == 1:
        bt = bt.view(max(T, 1), -1)
    ind = _dev_i32(indices, device)
    if logits_stride is None:
        mx = int(ctx.max().item()) if T else 0
        logits_stride = max(BLOCK_KV, (mx + BLOCK_KV - 1) // BLOCK_KV * BLOCK_KV)
    dt = torch.float32 if logits_dtype == LOGITS_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((T, logits_stride), dtype=dt, device=device)
    assert out.dtype == dt and out.stride(-1) == 1 and out.stride(0) == logits_stride
    qq = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    assert qq.is_contiguous() and weights.is_contiguous() and weights.dtype == torch.float32
    assert kv_cache.dim() == 2 and kv_cache.stride(1) == 1
    pstride = kv_cache.stride(0) if page_stride is None else int(page_stride)
    if kv_format == KV_MXFP4:
        assert q_scale is not None and q_scale.is_contiguous()
        _check(lib().dsa_mxfp4_paged_mqa_logits(
            _ptr(qq), _ptr(q_scale), _ptr(kv_cache), pstride, int(kv_cache.shape[0]), _ptr(weights),
            _ptr(ctx), _ptr(bt), int(bt.stride(0)), _ptr(ind), _ptr(schedule), int(num_sms),
            _ptr(out), int(logits_dtype), int(logits_stride), T, NUM_HEADS, HEAD_DIM, BLOCK_KV,
            _ptr(status), _stream(device)), "mxfp4_paged_mqa_logits")
        return out
    _check(lib().dsa_fp8_fp4_paged_mqa_logits(
        _ptr(qq), _ptr(kv_cache), pstride, int(kv_cache.shape[0]), int(kv_format), _ptr(weights),
        _ptr(ctx), _ptr(bt), int(bt.stride(0)), _ptr(ind), _ptr(schedule), int(num_sms),
        _ptr(out), int(logits_dtype), int(logits_stride), T, NUM_HEADS, HEAD_DIM, BLOCK_KV,
        _ptr(status), _stream(device)), "fp8_fp4_paged_mqa_logits")
    return out


def top_k_per_row(logits, row_starts, row_ends, k, out=None, status=None):
    """Top-k columns of each row in [row_start, row_end): int32 [rows, k], ascending, -1 padded."""
    device = logits.device
    R = int(logits.shape[0])
    if logits.dtype == torch.float32:
        dt = LOGITS_F32
    elif logits.dtype == torch.bfloat16:
        dt = LOGITS_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    assert logits.stride(-1) == 1
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=device)
    assert out.dtype == torch.int32 and out.stride(-1) == 1
    starts = _dev_i32(row_starts, device)
    ends = _dev_i32(row_ends, device)
    _check(lib().dsa_top_k_per_row(_ptr(logits), dt, int(logits.stride(0)), _ptr(starts),
                                   _ptr(ends), R, int(k), _ptr(out), int(out.stride(0)),
                                   _ptr(status), _stream(device)), "top_k_per_row")
    return out


def selftest_wait_timeout(timeout_ns, status):
    """Launch the bounded-wait self-test: a wait nothing satisfies runs out
    after timeout_ns and records DSA_ERR_TIMEOUT in `status` (device int32)."""
    _check(lib().dsa_selftest_wait_timeout(int(timeout_ns), _ptr(status), _stream(status.device)),
           "selftest_wait_timeout")


# ---------------------------------------------------------------------------
# decode context parallelism: per-rank top-k -> (score, global id) packs ->
# rank-major all-gather -> exact merge into the global top-k
# ---------------------------------------------------------------------------

def dcp_pack_topk(logits, local_idx, k, rank, world, interleave, out=None):
    """This rank's local top-k columns as fp32 (score, global id) pairs [rows, k, 2]."""
    if logits.dtype == torch.float32:
        dt = LOGITS_F32
    elif logits.dtype == torch.bfloat16:
        dt = LOGITS_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    assert logits.stride(-1) == 1 and local_idx.dtype == torch.int32 and local_idx.stride(-1) == 1
    R = int(logits.shape[0])
    if out is None:
        out = torch.empty((R, int(k), 2), dtype=torch.float32, device=logits.device)
    assert out.is_contiguous() and out.shape == (R, int(k), 2)
    _check(lib().dsa_dcp_pack_topk(_ptr(logits), dt, int(logits.stride(0)), _ptr(local_idx),
                                   int(local_idx.stride(0)), R, int(k), int(rank), int(world),
                                   int(interleave), _ptr(out), _stream(logits.device)), "dcp_pack_topk")
    return out


def dcp_merge_topk(gathered, k, out=None):
    """gathered fp32 [world, rows, k, 2] (rank-major) -> int32 [rows, k] global top-k ids."""
    assert gathered.dtype == torch.float32 and gathered.is_contiguous() and gathered.dim() == 4
    world, R = int(gathered.shape[0]), int(gathered.shape[1])
    if out is None:
        out = torch.empty((R, int(k)), dtype=torch.int32, device=gathered.device)
    _check(lib().dsa_dcp_merge_topk(_ptr(gathered), world, R, int(k), _ptr(out), int(out.stride(0)),
                                    _stream(gathered.device)), "dcp_merge_topk")
    return out


def dcp_gather_candidates(packed, world, group=None):
    """All-gather every rank's packs along a new leading dim: [world, rows, k, 2],
    rank r's pack at index r (torch.distributed; NCCL on GPUs)."""
    packed = packed.contiguous()
    flat = torch.empty((int(world) * packed.shape[0],) + tuple(packed.shape[1:]), dtype=packed.dtype,
                       device=packed.device)
    torch.distributed.all_gather_into_tensor(flat, packed, group=group)
    return flat.view((int(world),) + tuple(packed.shape))


def dcp_topk(logits, local_idx, k, rank, world, interleave, group=None, out=None):
    """The global top-k of a decode-context-parallel step on this rank: pack the
    local top-k, all-gather over `group`, merge (every rank gets the result)."""
    packed = dcp_pack_topk(logits, local_idx, k, rank, world, interleave)
    gathered = dcp_gather_candidates(packed, world, group) if world > 1 else packed.unsqueeze(0)
    return dcp_merge_topk(gathered, k, out=out)


def decode_chunk_ranges(rows, width, budget):
    """[(start, end), ...] row slices whose BF16 logits (2 * width bytes a row)
    fit `budget` bytes; [] means one pass over all rows."""
    cap = max(1, (int(rows) + 15) // 16)
    buf = (ctypes.c_int32 * (2 * cap))()
    n = ctypes.c_int32(0)
    _check(lib().dsa_decode_chunk_ranges(int(rows), int(width), int(budget), ctypes.cast(buf, _P), cap,
                                         ctypes.byref(n)), "decode_chunk_ranges")
    return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n.value)]


def indexer_decode_scratch(num_rows, logits_dtype, logits_stride, logits_budget, num_sms):
    """(logits scratch bytes, schedule words) that indexer_decode_topk needs."""
    sb, sw = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().dsa_indexer_decode_scratch(int(num_rows), int(logits_dtype), int(logits_stride),
                                            int(logits_budget), int(num_sms), ctypes.byref(sb),
                                            ctypes.byref(sw)), "indexer_decode_scratch")
    return int(sb.value), int(sw.value)


def indexer_decode_topk(q, kv_cache, weights, context_lens, block_table, k, indices=None,
                        kv_format=KV_FP8, logits_dtype=LOGITS_F32, logits_stride=None,
                        logits_budget=0, num_sms=None, out=None, status=None, scratch=None,
                        schedule=None, page_stride=None, q_scale=None):
    """The whole decode step (schedule, logits, top-k) in one native call; with
    a logits budget (bytes) the rows run in slices whose logits fit it.
    Returns int32 [T, k] top-k columns, ascending, -1 padded."""
    device = q.device
    T = int(q.shape[0])
    if num_sms is None:
        num_sms = device_num_sms()
    ctx = _dev_i32(context_lens, device)
    bt = _dev_i32(block_table, device)
    ind = _dev_i32(indices, device)
    if logits_stride is None:
        mx = int(ctx.max().item()) if T else 0
        logits_stride = max(BLOCK_KV, (mx + BLOCK_KV - 1) // BLOCK_KV * BLOCK_KV)
    sb, sw = indexer_decode_scratch(T, logits_dtype, logits_stride, logits_budget, num_sms)
    if scratch is None:
        scratch = torch.empty(max(sb, 16), dtype=torch.uint8, device=device)
    if schedule is None:
        schedule = torch.empty(max(sw, 1), dtype=torch.int32, device=device)
    if out is None:
        out = torch.empty((T, int(k)), dtype=torch.int32, device=device)
    assert out.dtype == torch.int32 and out.stride(-1) == 1
    qq = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    assert qq.is_contiguous() and weights.is_contiguous() and weights.dtype == torch.float32
    assert kv_cache.dim() == 2 and kv_cache.stride(1) == 1
    pstride = kv_cache.stride(0) if page_stride is None else int(page_stride)
    _check(lib().dsa_indexer_decode_topk(
        _ptr(qq), _ptr(q_scale), _ptr(kv_cache), pstride, int(kv_cache.shape[0]), int(kv_format), _ptr(weights),
        _ptr(ctx), _ptr(bt), int(bt.stride(0)), _ptr(ind), T, NUM_HEADS, HEAD_DIM, BLOCK_KV,
        int(num_sms), int(logits_dtype), int(logits_stride), int(logits_budget), _ptr(scratch),
        int(scratch.numel() * scratch.element_size()), _ptr(schedule), int(schedule.numel()), int(k),
        _ptr(out), int(out.stride(0)), _ptr(status), _stream(device)), "indexer_decode_topk")
    return out


def indexer_decode_topk_static(q, kv_cache, weights, context_lens, block_table, k, indices=None,
                               kv_format=KV_FP8, logits_dtype=LOGITS_F32, logits_stride=None, num_sms=None,
                               out=None, status=None, page_stride=None, q_scale=None):
    """indexer_decode_topk without any device allocation inside the library:
    the step's logits and schedule live in the library's fixed device array
    (STATIC_LOGITS_BYTES of logits), and the rows run in slices that fit it.
    For callers that cannot allocate device memory; calls that overlap on the
    GPU share that array and must be ordered by the caller.  Returns int32
    [T, k] top-k columns (allocated here only when `out` is None)."""
    device = q.device
    T = int(q.shape[0])
    if num_sms is None:
        num_sms = device_num_sms()
    ctx = _dev_i32(context_lens, device)
    bt = _dev_i32(block_table, device)
    ind = _dev_i32(indices, device)
    if logits_stride is None:
        mx = int(ctx.max().item()) if T else 0
        logits_stride = max(BLOCK_KV, (mx + BLOCK_KV - 1) // BLOCK_KV * BLOCK_KV)
    if out is None:
        out = torch.empty((T, int(k)), dtype=torch.int32, device=device)
    assert out.dtype == torch.int32 and out.stride(-1) == 1
    qq = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    assert qq.is_contiguous() and weights.is_contiguous() and weights.dtype == torch.float32
    assert kv_cache.dim() == 2 and kv_cache.stride(1) == 1
    pstride = kv_cache.stride(0) if page_stride is None else int(page_stride)
    _check(lib().dsa_indexer_decode_topk_static(
        _ptr(qq), _ptr(q_scale), _ptr(kv_cache), pstride, int(kv_cache.shape[0]), int(kv_format), _ptr(weights),
        _ptr(ctx), _ptr(bt), int(bt.stride(0)), _ptr(ind), T, NUM_HEADS, HEAD_DIM, BLOCK_KV,
        int(num_sms), int(logits_dtype), int(logits_stride), int(k), _ptr(out), int(out.stride(0)),
        _ptr(status), _stream(device)), "indexer_decode_topk_static")
    return out


def prefill_rows(cu_seqlen_ks, cu_seqlen_ke, local_cu_seq_lens, status=None):
    """(context_lens, request_ids) int32 [T] of prefill rows tagged (ks, ke)."""
    device = cu_seqlen_ks.device
    T = int(cu_seqlen_ks.shape[0])
    ks = _dev_i32(cu_seqlen_ks, device)
    ke = _dev_i32(cu_seqlen_ke, device)
    cu = _dev_i32(local_cu_seq_lens, device)
    ctx = torch.empty(T, dtype=torch.int32, device=device)
    req = torch.empty(T, dtype=torch.int32, device=device)
    _check(lib().dsa_prefill_rows(_ptr(ks), _ptr(ke), T, _ptr(cu), int(cu.shape[0]) - 1, _ptr(ctx), _ptr(req),
                                  _ptr(status), _stream(device)), "prefill_rows")
    return ctx, req


def prefill_mqa_logits(q, kv_cache, weights, context_lens, request_ids, block_table, schedule,
                       kv_format=KV_FP8, logits_dtype=LOGITS_F32, logits_stride=None, num_sms=None,
                       out=None, status=None, page_stride=None, q_scale=None):
    """Logits [T, logits_stride] of prefill rows over the paged cache; block_table
    is per request ([B, max_pages]) and row t reads row request_ids[t]."""
    device = q.device
    T = int(q.shape[0])
    if num_sms is None:
        num_sms = device_num_sms()
    ctx = _dev_i32(context_lens, device)
    req = _dev_i32(request_ids, device)
    bt = _dev_i32(block_table, device)
    if logits_stride is None:
        mx = int(ctx.max().item()) if T else 0
        logits_stride = max(BLOCK_KV, (mx + BLOCK_KV - 1) // BLOCK_KV * BLOCK_KV)
    dt = torch.float32 if logits_dtype == LOGITS_F32 else torch.bfloat16
    if out is None:
        out = torch.empty((T, logits_stride), dtype=dt, device=device)
    assert out.dtype == dt and out.stride(-1) == 1 and out.stride(0) == logits_stride
    qq = q.view(torch.uint8) if q.dtype != torch.uint8 else q
    assert qq.is_contiguous() and weights.is_contiguous() and weights.dtype == torch.float32
    pstride = kv_cache.stride(0) if page_stride is None else int(page_stride)
    _check(lib().dsa_prefill_mqa_logits(
        _ptr(qq), _ptr(q_scale), _ptr(kv_cache), pstride, int(kv_cache.shape[0]), int(kv_format), _ptr(weights), _ptr(ctx),
        _ptr(req), _ptr(bt), int(bt.stride(0)), int(bt.shape[0]), _ptr(schedule), int(num_sms), _ptr(out),
        int(logits_dtype), int(logits_stride), T, NUM_HEADS, HEAD_DIM, BLOCK_KV, _ptr(status),
        _stream(device)), "prefill_mqa_logits")
    return out


def prefill_topk(q, kv_cache, weights, cu_seqlen_ks, cu_seqlen_ke, local_cu_seq_lens, block_table, k,
                 kv_format=KV_FP8, logits_dtype=LOGITS_F32, logits_stride=None, num_sms=None,
                 status=None, logits_out=None, q_scale=None):
    """The prefill step over the paged cache: row tags -> (length, request),
    schedule, logits, top-k.  Returns (top-k [T, k] int32 request-local token
    positions, ascending, -1 padded; logits)."""
    if num_sms is None:
        num_sms = device_num_sms()
    ctx, req = prefill_rows(cu_seqlen_ks, cu_seqlen_ke, local_cu_seq_lens, status=status)
    sched = paged_mqa_logits_metadata(ctx, req, num_sms)
    logits = prefill_mqa_logits(q, kv_cache, weights, ctx, req, block_table, sched, kv_format=kv_format,
                                logits_dtype=logits_dtype, logits_stride=logits_stride, num_sms=num_sms,
                                out=logits_out, status=status, q_scale=q_scale)
    idx = top_k_per_row(logits, None, ctx, k, status=status)
    return idx, logits
