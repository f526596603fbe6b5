"""The seeded synthetic inputs against the decode configurations they stand
for: request counts, context ranges, rows per request and their causal
limits (every named workload, without building its key pool), and the paging
and quantisation recipe on small builds (block tables, poisoned unused pages,
per-token e4m3 key scales, e4m3 queries, head weights ~ N(0, 1) / sqrt(H)),
and the FP4 and MXFP4 quantisers against the error bounds of their formats."""
import math

import pytest
import torch

import workloads as W

# name: (requests, context range, rows per request range, k, seed)
SPECS = {
    "tiny": (2, (300, 517), (1, 1), 256, 0),
    "plain": (64, (4096, 32768), (1, 1), 2048, 1),
    "mtp": (128, (8192, 65536), (2, 2), 2048, 2),
    "varlen": (40, (120000 - 2048, 120000 + 2048), (1, 6), 2048, 3),
    "fp4_varlen": (40, (120000 - 2048, 120000 + 2048), (1, 6), 2048, 4),
    "mxfp4_varlen": (40, (120000 - 2048, 120000 + 2048), (1, 6), 2048, 6),
}


@pytest.mark.parametrize("name", list(SPECS))
def test_config_shapes_and_causal_limits(name):
    B, (lo, hi), (rlo, rhi), k, seed = SPECS[name]
    kw = W.config_spec(name)
    L, n = kw["request_lens"], kw["rows_per_request"]
    assert len(L) == B == len(n) and kw["topk"] == k and kw["seed"] == seed
    assert all(lo <= x <= hi for x in L) and all(rlo <= x <= rhi for x in n)
    if name == "tiny":
        assert L == [300, 517]
    if name.endswith("varlen"):
        assert len(set(n)) >= 4                     # a real mix of row counts
    assert kw.get("kv_format", W.KV_FP8) == {"fp4_varlen": W.KV_FP4,
                                             "mxfp4_varlen": W.KV_MXFP4}.get(name, W.KV_FP8)
    ctx, ids = W.config_rows(name)
    t = 0
    for r in range(B):                              # row j of request r sees L_r - n_r + 1 + j keys
        for j in range(n[r]):
            assert int(ctx[t]) == L[r] - n[r] + 1 + j and int(ids[t]) == r
            t += 1
    assert t == ctx.numel()
    assert W.config_rows(name, plain_indices=True)[1] is None


def _used_pages(wl):
    used = set()
    for r, L in enumerate(wl.request_lens):
        t0 = sum(wl.rows_per_request[:r])
        used.update(int(p) for p in wl.block_table[t0, : math.ceil(L / W.PAGE_TOKENS)])
    return used


def test_small_fp8_build_recipe():
    wl = W.build("recipe", request_lens=[300, 517, 64, 0], rows_per_request=[1, 3, 2, 1], seed=7)
    T = sum(wl.rows_per_request)
    assert wl.q.shape == (T, W.HEADS, W.HEAD_DIM) and wl.weights.shape == (T, W.HEADS)
    # block table: a request's rows share one row of it; pages are distinct and
    # drawn from a pool at least twice the pages in use
    t = 0
    for r, n in enumerate(wl.rows_per_request):
        for j in range(1, n):
            assert torch.equal(wl.block_table[t + j], wl.block_table[t])
        t += n
    used = _used_pages(wl)
    need = sum(math.ceil(L / W.PAGE_TOKENS) for L in wl.request_lens)
    assert len(used) == need and all(0 <= p < wl.num_pages for p in used)
    assert wl.num_pages >= 2 * need
    views = W._page_views(wl.kv_cache, W.KV_FP8)
    vals = W.e4m3_decode(views["values"].contiguous())
    scale = views["scale"].contiguous().view(torch.float32).squeeze(-1)
    # every unused page and every slot past a request's length is poisoned
    for p in range(wl.num_pages):
        if p not in used:
            assert torch.isnan(scale[p]).all() and torch.isnan(vals[p]).all()
    last = int(wl.block_table[0, 300 // W.PAGE_TOKENS])
    assert torch.isnan(scale[last, 300 % W.PAGE_TOKENS:]).all()
    # each written token: positive fp32 scale = amax / 448, its largest code is +-448
    for r, L in enumerate(wl.request_lens):
        t0 = sum(wl.rows_per_request[:r])
        for s in range(L):
            p, o = int(wl.block_table[t0, s // W.PAGE_TOKENS]), s % W.PAGE_TOKENS
            assert scale[p, o] > 0
            assert float(vals[p, o].abs().max()) == 448.0
    # queries are e4m3 codes of N(0, 1) draws; weights N(0, 1) / sqrt(H)
    q = W.e4m3_decode(wl.q)
    assert torch.isfinite(q).all() and float(q.abs().max()) <= 448.0
    assert abs(float(q.std()) - 1.0) < 0.05
    assert abs(float(wl.weights.std()) * math.sqrt(W.HEADS) - 1.0) < 0.1


def test_builds_are_seeded():
    a = W.build("s", request_lens=[200, 90], rows_per_request=[2, 1], seed=11)
    b = W.build("s", request_lens=[200, 90], rows_per_request=[2, 1], seed=11)
    c = W.build("s", request_lens=[200, 90], rows_per_request=[2, 1], seed=12)
    for f in ("q", "weights", "block_table", "kv_cache"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert not torch.equal(a.kv_cache, c.kv_cache)


def _e2m1(codes):
    mag = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=torch.float32)[(codes & 7).long()]
    return torch.where((codes & 8) != 0, -mag, mag)


def _unpack(packed):
    lo, hi = packed & 0xF, packed >> 4                # element 2i is the low nibble of byte i
    return torch.stack((lo, hi), dim=-1).flatten(-2)


def test_fp4_quantiser_invariants():
    g0 = torch.Generator().manual_seed(21)
    k = torch.randn((257, W.HEAD_DIM), generator=g0) * torch.rand((257, 1), generator=g0) * 5
    k[3] = 0.0                                        # an all-zero token
    k[4, :16] = 0.0                                   # an all-zero block
    packed, bs, g = W.quantize_keys_fp4(k)
    assert packed.shape == (257, W.HEAD_DIM // 2) and bs.shape == (257, W.HEAD_DIM // 16)
    amax = k.abs().amax(dim=-1)
    assert float(g[3]) == 1.0
    nz = amax > 0
    assert torch.allclose(g[nz] * 448.0 * 6.0, amax[nz], rtol=1e-6)
    bsv = W.e4m3_decode(bs)                           # per-16 block scales, e4m3
    codes = _e2m1(_unpack(packed)).view(257, -1, 16)
    step = bsv * g[:, None]                           # one block's unit
    deq = codes * step[..., None]
    err = (deq - k.view(257, -1, 16)).abs()
    assert (err <= step[..., None] + 1e-30).all()     # within one unit: half the widest e2m1 gap
    bmax = k.view(257, -1, 16).abs().amax(dim=-1)
    live = bmax > 0
    assert (codes.abs().amax(dim=-1)[live] == 6.0).all()   # each block's largest element saturates the code range
    assert (codes[4, 0] == 0).all() and (codes[3] == 0).all()


def test_mxfp4_quantiser_invariants():
    g0 = torch.Generator().manual_seed(22)
    x = torch.randn((9, 5, W.HEAD_DIM), generator=g0) * 3
    x[0, 0, :32] = 0.0                                # an all-zero block
    packed, sc = W.quantize_mxfp4(x)
    assert packed.shape == (9, 5, W.HEAD_DIM // 2) and sc.shape == (9, 5, W.HEAD_DIM // 32)
    blocks = x.view(9, 5, -1, 32)
    amax = blocks.abs().amax(dim=-1)
    live = amax > 0
    want = torch.floor(torch.log2(amax[live])) - 2 + 127
    assert torch.equal(sc[live].float(), want) and int(sc[0, 0, 0]) == 127
    scale = torch.exp2(sc.float() - 127)
    codes = _e2m1(_unpack(packed)).view(9, 5, -1, 32)
    err = (codes * scale[..., None] - blocks).abs()
    assert (err <= 2 * scale[..., None]).all()        # saturation at 6 of a block max in [4, 8) units
    assert (codes[0, 0, 0] == 0).all()
