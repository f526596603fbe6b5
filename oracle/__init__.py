"""ctypes front end of the CPU oracle (oracle/dsa_oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__ (build, and one
check in smoke) and bench.py's cpu_baseline / reference leg.  The product
package never imports it.

Every array crosses as numpy; tensors are converted on the host.  fp64 out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_dsa.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK = 0
ORACLE_ERR_ARG = 1
ORACLE_ERR_GROUPING = 2
ORACLE_ERR_CONTEXT = 3
ORACLE_ERR_BLOCK_TABLE = 4
ORACLE_ERR_BLOCK_ID = 5
ORACLE_ERR_STRIDE = 6

def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain -O2, IEEE arithmetic)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i32, i64, dbl, u8 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_uint8
            L.oracle_version.restype = ctypes.c_int
            L.oracle_set_plant.argtypes = [ctypes.c_int]
            L.oracle_e4m3_value.argtypes = [u8]
            L.oracle_e4m3_value.restype = dbl
            L.oracle_e2m1_value.argtypes = [u8]
            L.oracle_e2m1_value.restype = dbl
            L.oracle_ue8m0_value.argtypes = [u8]
            L.oracle_ue8m0_value.restype = dbl
            L.oracle_validate.argtypes = [P, P, P, i64, i32, i64, i32, i64]
            L.oracle_validate.restype = ctypes.c_int
            L.oracle_paged_mqa_logits.argtypes = [P, P, P, i64, i64, i32, P, P, P, i64, i32, i32,
                                                  i32, i32, P, i32, P, P, i64, i32]
            L.oracle_paged_mqa_logits.restype = ctypes.c_int
            L.oracle_top_k_per_row.argtypes = [P, i64, P, P, i32, i32, P, i64, i32]
            L.oracle_top_k_per_row.restype = ctypes.c_int
            L.oracle_dcp_global_id.argtypes = [i64, i32, i32, i32]
            L.oracle_dcp_global_id.restype = i64
            L.oracle_dcp_local_len.argtypes = [i64, i32, i32, i32]
            L.oracle_dcp_local_len.restype = i64
            L.oracle_dcp_pack.argtypes = [P, i64, P, i64, i32, i32, i32, i32, i32, P]
            L.oracle_dcp_pack.restype = ctypes.c_int
            L.oracle_dcp_merge.argtypes = [P, i32, i32, i32, P, i64]
            L.oracle_dcp_merge.restype = ctypes.c_int
            L.oracle_decode_chunk_ranges.argtypes = [i64, i64, i64, P, i64]
            L.oracle_prefill_rows.argtypes = [P, P, i32, P, i32, P, P]
            L.oracle_prefill_rows.restype = ctypes.c_int
            L.oracle_decode_chunk_ranges.restype = i64
            _lib = L
    return _lib


def _np(x, dtype):
    """numpy copy/view of a torch tensor or array-like, C-contiguous, given dtype."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"oracle {what} returned status {code}")
        self.code = code


def set_plant(p: int) -> None:
    lib().oracle_set_plant(int(p))


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code) & 0xFF)


def e2m1_value(nibble: int) -> float:
    return lib().oracle_e2m1_value(int(nibble) & 0xF)


def ue8m0_value(code: int) -> float:
    return lib().oracle_ue8m0_value(int(code) & 0xFF)


def validate(context_lens, indices, block_table, num_pages, logits_stride, block_kv=64) -> int:
    cl = _np(context_lens, np.int32)
    ind = _np(indices, np.int32)
    bt = _np(block_table, np.int32)
    T = cl.shape[0]
    bt2 = bt.reshape(T, -1) if T else bt.reshape(0, max(1, bt.size))
    return lib().oracle_validate(_ptr(cl), _ptr(ind), _ptr(bt2), bt2.shape[1], T,
                                 int(num_pages), int(block_kv), int(logits_stride))


def paged_mqa_logits(q, kv_cache, page_stride, kv_format, weights, context_lens, block_table,
                     out_cols, rows=None, with_bound=True, block_kv=64, nthreads=0, q_scale=None):
    """fp64 logits (and bound) of the selected rows: arrays [n_sel, out_cols].
    q is e4m3 [T, H, D]; with q_scale (MXFP4 keys), packed e2m1 [T, H, D/2]."""
    qn = _np(q, np.uint8)
    qs = _np(q_scale, np.uint8)
    kv = _np(kv_cache, np.uint8)
    w = _np(weights, np.float32)
    cl = _np(context_lens, np.int32)
    bt = _np(block_table, np.int32)
    T = cl.shape[0]
    H = w.shape[1] if w.ndim == 2 else w.size // max(T, 1)
    D = qn.size // max(T * H, 1) * (2 if qs is not None else 1)
    bt2 = bt.reshape(T, -1)
    rws = None if rows is None else _np(rows, np.int32)
    n_sel = T if rws is None else rws.shape[0]
    num_pages = kv.shape[0] if kv.ndim == 2 else kv.size // page_stride
    logits = np.empty((n_sel, out_cols), dtype=np.float64)
    bound = np.empty((n_sel, out_cols), dtype=np.float64) if with_bound else None
    st = lib().oracle_paged_mqa_logits(_ptr(qn), _ptr(qs), _ptr(kv), int(page_stride), int(num_pages),
                                       int(kv_format), _ptr(w), _ptr(cl), _ptr(bt2),
                                       bt2.shape[1], T, H, D, int(block_kv), _ptr(rws),
                                       n_sel, _ptr(logits), _ptr(bound), int(out_cols),
                                       int(nthreads))
    if st != ORACLE_OK:
        raise OracleError(st, "paged_mqa_logits")
    return logits, bound


def top_k_per_row(scores, row_ends, k, row_starts=None, nthreads=0):
    """Stable per-row top-k of an fp64 score matrix [rows, stride] -> int32 [rows, k]."""
    sc = _np(scores, np.float64)
    if sc.ndim == 1:
        sc = sc.reshape(1, -1)
    ends = _np(row_ends, np.int32)
    starts = _np(row_starts, np.int32)
    R = ends.shape[0]
    out = np.empty((R, k), dtype=np.int32)
    st = lib().oracle_top_k_per_row(_ptr(sc), sc.shape[1], _ptr(starts), _ptr(ends), R, int(k),
                                    _ptr(out), k, int(nthreads))
    if st != ORACLE_OK:
        raise OracleError(st, "top_k_per_row")
    return out


def workload_logits(wl, rows=None, with_bound=True, nthreads=0, out_cols=None):
    """Oracle logits of a workloads.Workload (host copies are made as needed)."""
    return paged_mqa_logits(wl.q, wl.kv_cache, wl.page_stride, wl.kv_format, wl.weights,
                            wl.context_lens, wl.block_table,
                            wl.logits_stride if out_cols is None else out_cols,
                            rows=rows, with_bound=with_bound, nthreads=nthreads,
                            q_scale=getattr(wl, "q_scale", None))


# ---------------------------------------------------------------------------
# DCP sharding and exact merge of per-rank top-k candidates
# ---------------------------------------------------------------------------

def dcp_global_id(local, rank, world, interleave):
    return int(lib().oracle_dcp_global_id(int(local), int(rank), int(world), int(interleave)))


def dcp_local_len(length, rank, world, interleave):
    return int(lib().oracle_dcp_local_len(int(length), int(rank), int(world), int(interleave)))


def dcp_pack(local_scores, local_idx, k, rank, world, interleave):
    """[rows, k, 2] float64 (score, global id) of a rank's local top-k."""
    sc = _np(local_scores, np.float64)
    if sc.ndim == 1:
        sc = sc.reshape(1, -1)
    li = _np(local_idx, np.int32)
    if li.ndim == 1:
        li = li.reshape(1, -1)
    out = np.zeros((sc.shape[0], int(k), 2), dtype=np.float64)
    st = lib().oracle_dcp_pack(_ptr(sc), sc.shape[1], _ptr(li), li.shape[1], sc.shape[0], int(k),
                               int(rank), int(world), int(interleave), _ptr(out))
    if st != ORACLE_OK:
        raise OracleError(st, "dcp_pack")
    return out


def dcp_merge(gathered, k):
    """gathered [world, rows, k, 2] (score, global id) -> int32 [rows, k] global top-k."""
    g = _np(gathered, np.float64)
    world, rows = g.shape[0], g.shape[1]
    out = np.zeros((rows, int(k)), dtype=np.int32)
    st = lib().oracle_dcp_merge(_ptr(g), world, rows, int(k), _ptr(out), int(k))
    if st != ORACLE_OK:
        raise OracleError(st, "dcp_merge")
    return out


# ---------------------------------------------------------------------------
# row chunking of the decode step under a logits budget
# ---------------------------------------------------------------------------

def decode_chunk_ranges(rows, width, budget):
    """[(start, end), ...] slices of the rows whose BF16 logits fit `budget`
    bytes; [] means one pass over all rows."""
    cap = max(1, (int(rows) + 15) // 16)
    buf = np.zeros(2 * cap, dtype=np.int32)
    n = lib().oracle_decode_chunk_ranges(int(rows), int(width), int(budget), _ptr(buf), cap)
    if n < 0:
        raise OracleError(-n, "decode_chunk_ranges")
    return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n)]


# ---------------------------------------------------------------------------
# prefill rows over the paged cache
# ---------------------------------------------------------------------------

def prefill_rows(cu_seqlen_ks, cu_seqlen_ke, local_cu_seq_lens):
    """(context_lens, request_ids) int32 [T] of prefill rows tagged (ks, ke)."""
    ks = _np(cu_seqlen_ks, np.int32)
    ke = _np(cu_seqlen_ke, np.int32)
    cu = _np(local_cu_seq_lens, np.int32)
    T, B = ks.shape[0], cu.shape[0] - 1
    ctx = np.zeros(T, dtype=np.int32)
    req = np.zeros(T, dtype=np.int32)
    st = lib().oracle_prefill_rows(_ptr(ks), _ptr(ke), T, _ptr(cu), B, _ptr(ctx), _ptr(req))
    if st != ORACLE_OK:
        raise OracleError(st, "prefill_rows")
    return ctx, req


def prefill_logits(pf, rows=None, with_bound=True, nthreads=0):
    """Oracle logits of a workloads.Prefill (selected rows, or all): each row's
    keys [0, ke - ks) of its request, read through the request's block-table row."""
    ctx, req = prefill_rows(pf.cu_seqlen_ks, pf.cu_seqlen_ke, pf.local_cu_seq_lens)
    bt = _np(pf.block_table, np.int32)[req]          # the row-indexed view of the request table
    return paged_mqa_logits(pf.q, pf.kv_cache, pf.page_stride, pf.kv_format, pf.weights, ctx, bt,
                            pf.logits_stride, rows=rows, with_bound=with_bound, nthreads=nthreads,
                            q_scale=getattr(pf, "q_scale", None))
