"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* number formats: every e4m3 code against torch's float8_e4m3fn conversion and
  the named values of the OCP FP8 spec; every e2m1 code against the OCP MX
  spec's table (tests/golden/);
* closed forms: a one-hot query reads a single decoded key value back;
  logits(q) - logits(-q) and logits(q) + logits(-q) reduce the ReLU away and
  leave a plain matrix product, checked against numpy's matmul over keys
  decoded by torch;
* brute force on tiny unpaged inputs (dense numpy evaluation over keys gathered
  and decoded independently of the oracle);
* invariants: permuting physical pages, padding the varlen batch to
  (B, max_n), and plain decode (indices = None) against indices = arange(B);
* top-k against a brute-force Python sort on random, tie-heavy, bf16-rounded,
  -inf and NaN rows;
* argument validation (grouping, causal limits, block table);
* planted mistakes: each deliberate error switched on inside the oracle makes
  at least one of the pins above fail.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            out.append((int(a, 16), float(b)))
    return out


# ---------------------------------------------------------------------------
# independent decoding of a workload (torch float8 for e4m3, golden table for e2m1)
# ---------------------------------------------------------------------------

def _e2m1_table():
    tab = np.zeros(16)
    for code, val in _read_golden("e2m1_ocp_mx.txt"):
        tab[code] = val
    return tab


def dense_keys(wl, t):
    """Keys of row t, decoded without the oracle: (values [L, D] fp64, scale [L] fp64)."""
    L = int(wl.context_lens[t])
    kv = wl.kv_cache.numpy()
    bt = wl.block_table.numpy()
    s = np.arange(L)
    page = bt[t, s // 64]
    slot = s % 64
    if wl.kv_format == W.KV_FP8:
        codes = kv[page[:, None], slot[:, None] * 128 + np.arange(128)[None, :]]
        vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
        sc = kv[page[:, None], 8192 + slot[:, None] * 4 + np.arange(4)[None, :]]
        scale = sc.copy().view(np.float32).reshape(-1).astype(np.float64)
        return vals, scale
    tab = _e2m1_table()
    packed = kv[page[:, None], slot[:, None] * 64 + np.arange(64)[None, :]]
    lo = tab[packed & 0xF]
    hi = tab[packed >> 4]
    el = np.empty((L, 128))
    el[:, 0::2] = lo
    el[:, 1::2] = hi
    if wl.kv_format == W.KV_MXFP4:
        esc = kv[page[:, None], 4096 + slot[:, None] * 4 + np.arange(4)[None, :]]
        es = torch.from_numpy(esc.copy()).view(torch.float8_e8m0fnu).double().numpy()
        return el * np.repeat(es, 32, axis=1), np.ones(L)
    bsc = kv[page[:, None], 4096 + slot[:, None] * 8 + np.arange(8)[None, :]]
    bs = torch.from_numpy(bsc.copy()).view(torch.float8_e4m3fn).double().numpy()
    vals = el * np.repeat(bs, 16, axis=1)
    sc = kv[page[:, None], 4608 + slot[:, None] * 4 + np.arange(4)[None, :]]
    scale = sc.copy().view(np.float32).reshape(-1).astype(np.float64)
    return vals, scale


def dense_q(wl, t):
    if wl.q_scale is None:
        return wl.q[t].view(torch.float8_e4m3fn).double().numpy()  # [H, D]
    tab = _e2m1_table()
    packed = wl.q[t].numpy()                                        # [H, D/2]
    el = np.empty((packed.shape[0], 2 * packed.shape[1]))
    el[:, 0::2] = tab[packed & 0xF]
    el[:, 1::2] = tab[packed >> 4]
    es = wl.q_scale[t].view(torch.float8_e8m0fnu).double().numpy()  # [H, D/32]
    return el * np.repeat(es, 32, axis=1)


def small_workload(seed=0, H=64, kv_format=W.KV_FP8, lens=(150, 77, 203), rows=(1, 3, 2)):
    return W.build("pin", list(lens), list(rows), kv_format=kv_format, heads=H, seed=seed,
                   topk=16)


# ---------------------------------------------------------------------------
# pin checks (plain functions so the planted-mistake test can run them too)
# ---------------------------------------------------------------------------

def check_e4m3_vs_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(mine[ok]))
    for code, val in _read_golden("e4m3_ocp_fp8.txt"):
        got = oracle.e4m3_value(code)
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val)


def check_ue8m0_vs_torch():
    """The OCP MX E8M0 scale against torch's float8_e8m0fnu, all 256 codes."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    mine = np.array([oracle.ue8m0_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])


def check_e2m1_vs_spec():
    for code, val in _read_golden("e2m1_ocp_mx.txt"):
        got = oracle.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def check_bruteforce(kv_format=W.KV_FP8, H=64, seed=0):
    wl = small_workload(seed=seed, H=H, kv_format=kv_format)
    lg, bd = oracle.workload_logits(wl)
    for t in range(wl.num_rows):
        L = int(wl.context_lens[t])
        K, ks = dense_keys(wl, t)
        Q = dense_q(wl, t)
        w = wl.weights[t].double().numpy()
        S = Q @ K.T                                  # [H, L]
        ref = ks * (w @ np.maximum(S, 0.0))
        mag = ks * (np.abs(w)[:, None] * (np.abs(Q) @ np.abs(K).T)).sum(axis=0)
        tol = 1e-12 * (mag + 1e-300)
        assert np.all(np.abs(lg[t, :L] - ref) <= tol), t
        assert np.allclose(bd[t, :L], mag, rtol=1e-12, atol=0)
        assert np.all(np.isneginf(lg[t, L:]))


def check_one_hot_reads_key():
    """H = 1, w = 1, q = e_d: logit[s] = kscale[s] * max(k[s, d], 0)."""
    wl = small_workload(seed=5, H=1, lens=(130,), rows=(1,))
    d = 37
    q = torch.zeros_like(wl.q)
    q[0, 0, d] = 0x38                                 # e4m3 1.0
    wl.q = q
    wl.weights = torch.ones_like(wl.weights)
    lg, _ = oracle.workload_logits(wl)
    K, ks = dense_keys(wl, 0)
    assert np.array_equal(lg[0, :130], ks * np.maximum(K[:, d], 0.0))


def _neg_q(wl):
    w2 = W.Workload(**{**wl.__dict__})
    # exact negation of every code: the e4m3 sign bit, or both e2m1 nibbles' sign bits
    w2.q = wl.q ^ (0x88 if wl.q_scale is not None else 0x80)
    return w2


def check_relu_identities(kv_format=W.KV_FP8):
    """logits(q) - logits(-q) = ks * (w^T Q) K^T and logits(q) + logits(-q) = ks * w^T |Q K^T|."""
    wl = small_workload(seed=7, kv_format=kv_format)
    lp, bp = oracle.workload_logits(wl)
    lm, _ = oracle.workload_logits(_neg_q(wl))
    for t in range(wl.num_rows):
        L = int(wl.context_lens[t])
        K, ks = dense_keys(wl, t)
        Q = dense_q(wl, t)
        w = wl.weights[t].double().numpy()
        lin = ks * ((w @ Q) @ K.T)
        absr = ks * (w @ np.abs(Q @ K.T))
        tol = 1e-12 * (bp[t, :L] + 1e-300)
        assert np.all(np.abs((lp[t, :L] - lm[t, :L]) - lin) <= 2 * tol)
        assert np.all(np.abs((lp[t, :L] + lm[t, :L]) - absr) <= 2 * tol)


def check_weight_scaling():
    wl = small_workload(seed=9)
    a, _ = oracle.workload_logits(wl)
    wl2 = W.Workload(**{**wl.__dict__})
    wl2.weights = wl.weights * 4.0                    # exact power-of-two scaling
    b, _ = oracle.workload_logits(wl2)
    fin = np.isfinite(a)
    assert np.array_equal(b[fin], 4.0 * a[fin])


def check_page_permutation():
    wl = small_workload(seed=11)
    a, _ = oracle.workload_logits(wl)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(wl.num_pages, generator=g)      # new slot of old page p = perm[p]
    kv2 = torch.empty_like(wl.kv_cache)
    kv2[perm] = wl.kv_cache
    bt2 = wl.block_table.clone()
    m = bt2 >= 0
    bt2[m] = perm[bt2[m].long()].to(torch.int32)
    wl2 = W.Workload(**{**wl.__dict__})
    wl2.kv_cache, wl2.block_table = kv2, bt2
    b, _ = oracle.workload_logits(wl2)
    assert np.array_equal(a, b)


def check_varlen_equals_padded():
    wl = small_workload(seed=13, lens=(300, 129, 64, 1), rows=(2, 5, 1, 1))
    a, _ = oracle.workload_logits(wl)
    slot_row, max_n = W.padded_rows(wl)
    # padded batch: every request gets max_n rows; padding rows repeat the
    # request's last row (its q, weights, block table and causal limit)
    src = []
    t = 0
    for n in wl.rows_per_request:
        for j in range(max_n):
            src.append(t + min(j, n - 1))
        t += n
    src = torch.tensor(src)
    wl2 = W.Workload(**{**wl.__dict__})
    wl2.q, wl2.weights = wl.q[src], wl.weights[src]
    wl2.context_lens, wl2.block_table = wl.context_lens[src], wl.block_table[src]
    wl2.indices = None
    b, _ = oracle.workload_logits(wl2)
    valid = slot_row >= 0
    assert np.array_equal(b[valid.numpy()], a[slot_row[valid].numpy()])


def check_topk_bruteforce(seed=0):
    rng = np.random.default_rng(seed)
    cases = []
    for kind in ("random", "ties", "bf16", "inf", "nan", "short", "empty", "start"):
        R, C = 5, 97
        x = rng.standard_normal((R, C))
        if kind == "ties":
            x = rng.integers(-3, 3, (R, C)).astype(np.float64)
            x[0, :] = 0.0
            x[1, ::2] = -0.0
        elif kind == "bf16":
            x = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
        elif kind == "inf":
            x[:, 50:] = -np.inf
        elif kind == "nan":
            x[:, ::7] = np.nan
        ends = rng.integers(0, C + 1, R).astype(np.int32)
        starts = np.zeros(R, np.int32)
        if kind == "short":
            ends = np.minimum(ends, 9)
        if kind == "empty":
            ends[:] = 0
        if kind == "start":
            starts = rng.integers(0, 40, R).astype(np.int32)
            ends = np.maximum(ends, starts)
        cases.append((x, starts, ends))
    for x, starts, ends in cases:
        for k in (1, 8, 16, 100):
            got = oracle.top_k_per_row(x, ends, k, row_starts=starts)
            for r in range(x.shape[0]):
                cols = range(int(starts[r]), int(ends[r]))
                key = (lambda s: (1, 0.0, s) if np.isnan(x[r, s]) else (0, -x[r, s], s))
                pick = sorted(sorted(cols, key=key)[:k])
                ref = pick + [-1] * (k - len(pick))
                assert list(got[r]) == ref, (r, k)


def check_fp4_bruteforce():
    check_bruteforce(kv_format=W.KV_FP4, seed=21)


def check_mxfp4_bruteforce():
    check_bruteforce(kv_format=W.KV_MXFP4, seed=23)
    check_relu_identities(kv_format=W.KV_MXFP4)


def check_dcp_mapping():
    """Each rank's tokens, enumerated in global order, are its local positions
    0, 1, ...; the mapping and the shard lengths must agree with that."""
    for world in (1, 2, 3, 4):
        for inter in (1, 2, 3, 5):
            L = 97
            owned = {r: [g for g in range(L) if (g // inter) % world == r] for r in range(world)}
            assert sum(len(v) for v in owned.values()) == L
            for r, gs in owned.items():
                assert oracle.dcp_local_len(L, r, world, inter) == len(gs)
                for local, g in enumerate(gs):
                    assert oracle.dcp_global_id(local, r, world, inter) == g


def _dcp_merge_of_shards(sc, ends, k, world, inter):
    """Per-rank oracle top-k over each rank's own columns, packed, gathered
    rank-major and merged."""
    rows = sc.shape[0]
    packs = []
    for r in range(world):
        cols = [g for g in range(sc.shape[1]) if (g // inter) % world == r]
        loc = sc[:, cols] if cols else np.zeros((rows, 1))
        loc_ends = np.array([sum(1 for g in cols if g < e) for e in ends], dtype=np.int32)
        lidx = oracle.top_k_per_row(loc, loc_ends, k)
        packs.append(oracle.dcp_pack(loc, lidx, k, r, world, inter))
    return oracle.dcp_merge(np.stack(packs), k)


def check_dcp_merge_is_global_topk(seed=0):
    """The merge of per-rank top-k equals the top-k of the whole row (the
    exactness argument of _merge_dcp_topk_global), ties and NaN included."""
    rng = np.random.default_rng(seed)
    rows, L = 5, 300
    sc = np.round(rng.standard_normal((rows, L)) * 3) / 2   # coarse grid: many ties
    sc[0, ::7] = np.nan
    sc[1, :50] = -np.inf
    ends = np.array([L, 260, 17, 1, 0], dtype=np.int32)
    for world, inter, k in ((1, 1, 16), (2, 1, 16), (3, 4, 37), (4, 64, 64), (2, 7, 1), (3, 1, 300)):
        got = _dcp_merge_of_shards(sc, ends, k, world, inter)
        want = oracle.top_k_per_row(sc, ends, k)
        assert np.array_equal(got, want), (world, inter, k)


def check_all_zero_keys():
    """All-zero keys (e4m3 code 0, scale 1): every logit below L_t is exactly 0,
    and the top-k is the first k positions (equal scores go to the lower
    column)."""
    wl = small_workload(seed=9)
    views = W._page_views(wl.kv_cache, wl.kv_format)
    views["values"][:] = 0
    views["scale"][:] = torch.tensor([1.0], dtype=torch.float32).view(torch.uint8)
    lg, _ = oracle.workload_logits(wl, with_bound=False)
    ctx = wl.context_lens.numpy()
    for t in range(wl.num_rows):
        L = int(ctx[t])
        assert np.all(lg[t, :L] == 0.0) and np.all(np.isneginf(lg[t, L:]))
    k = 16
    got = oracle.top_k_per_row(lg, ctx, k)
    for t in range(wl.num_rows):
        L = int(ctx[t])
        want = list(range(min(k, L))) + [-1] * (k - min(k, L))
        assert got[t].tolist() == want


def check_chunk_ranges():
    """Row chunking under a BF16 logits budget (sparse_attn_indexer docs,
    _decode_chunk_ranges).  Worked by hand from the rule's statement:
      134 rows x 120064 columns, 16 MiB: a slice may hold
        floor(16777216 / 240128) = 69 -> 64 rows = 4 units; 134 rows = 9 units
        (the last partial); ceil(9 / 4) = 3 slices of 3 units: 48, 48, 38.
      1000 rows x 4096 columns, 819200 B: 100 -> 96 rows = 6 units; 63 units;
        11 slices, 63 = 11 * 5 + 8, so eight of 6 units then three of 5:
        96 x 8, 80, 80, then the tail 1000 - 928 = 72.
      40 rows x 64 columns, 5120 B (= 40 rows exactly): fits, one pass.
    Then properties any correct reading has, on a sweep."""
    assert oracle.decode_chunk_ranges(134, 120064, 16 << 20) == [(0, 48), (48, 96), (96, 134)]
    want = [(96 * i, 96 * (i + 1)) for i in range(8)] + [(768, 848), (848, 928), (928, 1000)]
    assert oracle.decode_chunk_ranges(1000, 4096, 819200) == want
    assert oracle.decode_chunk_ranges(40, 64, 5120) == []
    assert oracle.decode_chunk_ranges(0, 64, 100) == []
    assert oracle.decode_chunk_ranges(17, 64, 0) == []
    assert oracle.decode_chunk_ranges(33, 64, 16 * 64 * 2) == [(0, 16), (16, 32), (32, 33)]
    for bad in ((10, 64, -1), (100, 64, 15 * 64 * 2), (100, 0, 1000)):
        with pytest.raises(oracle.OracleError):
            oracle.decode_chunk_ranges(*bad)
    rng = np.random.default_rng(4)
    for _ in range(400):
        rows = int(rng.integers(1, 3000))
        width = int(rng.integers(1, 200)) * 64
        per_rows = int(rng.integers(16, 4000))
        budget = per_rows * width * 2 + int(rng.integers(0, width * 2))
        r = oracle.decode_chunk_ranges(rows, width, budget)
        if rows * width * 2 <= budget:
            assert r == []
            continue
        limit = budget // (2 * width) // 16 * 16
        assert r[0][0] == 0 and r[-1][1] == rows
        sizes = [e - s for s, e in r]
        assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
        assert all(0 < n <= limit for n in sizes)                  # every slice fits the budget
        assert all(n % 16 == 0 for n in sizes[:-1])               # whole units but the tail
        units = [(n + 15) // 16 for n in sizes]
        assert (len(r) - 1) * (limit // 16) < (rows + 15) // 16   # no fewer slices would do
        assert max(units) - min(units) <= 1                       # as even as the units allow
        assert units == sorted(units, reverse=True)               # larger slices first


def check_prefill_rows():
    """Prefill row tags -> (causal length, request), worked by hand from the
    CPU indexer's prefill branch (request = sorted search of ks to the right,
    minus one; length = ke - ks).  Requests [0,5), [5,5) (empty), [5,9):
      (0, 3) -> request 0, length 3      (0, 5) -> 0, 5
      (5, 6) -> three starts <= 5, so request 2, length 1
      (5, 9) -> 2, 4                      (9, 9) -> past the last start: 2, length 0
    Then the prefill logits of a chunk equal the decode logits (pinned by
    brute force) of the same rows with the same causal limits."""
    ctx, req = oracle.prefill_rows([0, 0, 5, 5, 9], [3, 5, 6, 9, 9], [0, 5, 5, 9])
    assert ctx.tolist() == [3, 5, 1, 4, 0] and req.tolist() == [0, 0, 2, 2, 2]
    for kv_format in (W.KV_FP8, W.KV_FP4):
        wl = W.build("pf", [300, 517, 0, 70], [100, 40, 1, 3], kv_format=kv_format, topk=32, seed=7)
        pf = W.prefill_view(wl)
        got, _ = oracle.prefill_logits(pf, with_bound=False)
        want, _ = oracle.workload_logits(wl, with_bound=False)
        assert np.array_equal(got, want)


PIN_CHECKS = [
    check_e4m3_vs_torch, check_e2m1_vs_spec, check_bruteforce, check_one_hot_reads_key,
    check_relu_identities, check_weight_scaling, check_page_permutation,
    check_varlen_equals_padded, check_topk_bruteforce, check_fp4_bruteforce,
    check_ue8m0_vs_torch, check_mxfp4_bruteforce,
    check_dcp_mapping, check_dcp_merge_is_global_topk, check_chunk_ranges, check_prefill_rows,
    check_all_zero_keys,
]


# ---------------------------------------------------------------------------
# tests
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    oracle.set_plant(0)
    check()


def test_bruteforce_few_heads():
    for H in (1, 2):
        check_bruteforce(H=H, seed=H)


def test_fp4_relu_identities():
    check_relu_identities(kv_format=W.KV_FP4)


def test_fp4_unit_keys_closed_form():
    """FP4 keys all 1.0 (code 0x2, block scale 1.0, token scale 1): logit = sum_h w_h relu(sum_d q_hd)."""
    wl = small_workload(seed=3, kv_format=W.KV_FP4, lens=(70,), rows=(1,))
    kv = wl.kv_cache.clone()
    for p in wl.block_table[0, :2].tolist():
        kv[p, :4096] = 0x22
        kv[p, 4096:4608] = 0x38
        kv[p, 4608:4864] = torch.tensor([1.0] * 64, dtype=torch.float32).view(torch.uint8)
    wl.kv_cache = kv
    lg, _ = oracle.workload_logits(wl)
    Q = dense_q(wl, 0)
    w = wl.weights[0].double().numpy()
    ref = float(w @ np.maximum(Q.sum(axis=1), 0.0))
    assert np.allclose(lg[0, :70], ref, rtol=1e-13, atol=0)


def test_plain_equals_arange():
    wl = W.config("tiny")
    B = wl.num_rows
    assert oracle.validate(wl.context_lens, None, wl.block_table, wl.num_pages,
                           wl.logits_stride) == 0
    assert oracle.validate(wl.context_lens, torch.arange(B, dtype=torch.int32), wl.block_table,
                           wl.num_pages, wl.logits_stride) == 0


def test_topk_all_equal_picks_first_k():
    x = np.zeros((1, 50))
    assert list(oracle.top_k_per_row(x, [50], 10)[0]) == list(range(10))
    x = np.full((1, 50), -np.inf)
    assert list(oracle.top_k_per_row(x, [50], 3)[0]) == [0, 1, 2]


def test_topk_short_rows_pad():
    x = np.arange(10, dtype=np.float64)[None, :]
    assert list(oracle.top_k_per_row(x, [4], 6)[0]) == [0, 1, 2, 3, -1, -1]
    assert list(oracle.top_k_per_row(x, [0], 3)[0]) == [-1, -1, -1]


def test_validate_errors():
    wl = small_workload(seed=1)
    ok = dict(context_lens=wl.context_lens, indices=wl.indices, block_table=wl.block_table,
              num_pages=wl.num_pages, logits_stride=wl.logits_stride)
    assert oracle.validate(**ok) == oracle.ORACLE_OK
    bad = dict(ok, indices=torch.tensor([0, 1, 1, 1, 0, 2], dtype=torch.int32))
    assert oracle.validate(**bad) == oracle.ORACLE_ERR_GROUPING
    cl = wl.context_lens.clone()
    cl[2] = cl[1] - 1
    assert oracle.validate(**dict(ok, context_lens=cl)) == oracle.ORACLE_ERR_CONTEXT
    bt = wl.block_table.clone()
    bt[2, 0] = (bt[1, 0] + 1) % wl.num_pages
    assert oracle.validate(**dict(ok, block_table=bt)) == oracle.ORACLE_ERR_BLOCK_TABLE
    bt = wl.block_table.clone()
    bt[0, 0] = wl.num_pages
    assert oracle.validate(**dict(ok, block_table=bt)) == oracle.ORACLE_ERR_BLOCK_ID
    assert oracle.validate(**dict(ok, logits_stride=wl.logits_stride - 64)) == oracle.ORACLE_ERR_STRIDE


# plant id -> the mistake it switches on inside the oracle
PLANTS = {
    1: "query operand transposed (q[d][h] for q[h][d])",
    2: "ReLU dropped",
    3: "page index s / 128 for s / 64 (wrong block size)",
    4: "sign flipped inside the ReLU",
    5: "head weight dropped",
    6: "FP4 block scale index d / 32 for d / 16",
    7: "top-k order reversed",
    8: "DCP merge keeps the smallest scores",
    9: "DCP merge breaks score ties to the higher global id",
    10: "row chunking counts whole 16-row units only (drops the partial one)",
    11: "row chunking gives the smaller slices first",
    12: "prefill causal length taken as ke instead of ke - ks",
    13: "ue8m0 scale with bias 128 instead of 127",
}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda p: PLANTS[p])
def test_planted_mistake_is_caught(plant):
    caught = []
    oracle.set_plant(plant)
    try:
        for check in PIN_CHECKS:
            try:
                check()
            except AssertionError:
                caught.append(check.__name__)
    finally:
        oracle.set_plant(0)
    assert caught, f"no pin caught plant {plant}: {PLANTS[plant]}"
