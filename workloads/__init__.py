"""Seeded synthetic inputs for the DSA indexer decode path.

This module is shared by the tests, the CPU oracle's callers and ``bench.py``.
It builds inputs only: request lengths, row flattening, paged key caches in the
two storage formats, query codes, head weights and block tables.  It holds none
of the indexer's arithmetic (no logits, no top-k, no schedule).

Storage formats (one page = ``PAGE_TOKENS`` = 64 tokens, head_dim D = 128):

* FP8 page, ``FP8_PAGE_BYTES`` = 8448 B::

      [0, 8192)     token j's 128 e4m3 codes at byte 128*j
      [8192, 8448)  token j's fp32 key scale at byte 8192 + 4*j

  The stored key is ``k[s, d] = e4m3(code) * scale[s]``.  This is the
  per-token payload the sparse_attn_indexer docs give for the FP8 K-gather
  workspace (``head_dim`` FP8 plus 4 bytes of fp32 scale,
  ``_gather_workspace_shapes``), with values and scales split inside a page.

* FP4 page, ``FP4_PAGE_BYTES`` = 4864 B::

      [0, 4096)     token j's 64 bytes of packed e2m1 at 64*j
                    (element 2i = low nibble of byte i, 2i+1 = high nibble)
      [4096, 4608)  token j's 8 e4m3 block scales at 4096 + 8*j
                    (block b covers elements 16b .. 16b+15)
      [4608, 4864)  token j's fp32 token scale at 4608 + 4*j

  The stored key is ``k[s, d] = e2m1 * e4m3(block_scale[s, d // 16]) * g[s]``.

* MXFP4 page, ``MXFP4_PAGE_BYTES`` = 4352 B (the pages' own FP4 cache:
  ``head_dim // 2`` packed bytes and ``head_dim // 32`` ue8m0 scales a token,
  ``_gather_workspace_shapes``)::

      [0, 4096)     token j's 64 bytes of packed e2m1 (as FP4)
      [4096, 4352)  token j's 4 ue8m0 block scales at 4096 + 4*j
                    (block b covers elements 32b .. 32b+31)

  The stored key is ``k[s, d] = e2m1 * 2^(block_scale[s, d // 32] - 127)``;
  q is stored the same way (packed e2m1 ``[T, H, D/2]`` and ue8m0
  ``q_scale [T, H, D/32]``).

Pages live in a pool ``kv_cache`` of shape ``[num_pages, page_stride]`` (uint8);
``page_stride`` is at least the page size and a multiple of 16.  Pages that no
request uses, and the tail of each request's last page, are poisoned (e4m3 NaN
codes and NaN scales) so that any read past a row's causal limit shows up.

Row flattening follows the varlen decode description in PR 47469 ("Route
SM100 sparse-indexer decode through varlen paged MQA logits", Purpose and
Changes): request r contributes ``n_r`` adjacent rows that share the request id
``indices[t] = r``; row j of request r sees ``L_r - n_r + 1 + j`` keys.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE_TOKENS = 64
HEADS = 64
HEAD_DIM = 128

KV_FP8 = 0
KV_FP4 = 1
KV_MXFP4 = 2

LOGITS_F32 = 0
LOGITS_BF16 = 1

FP8_VALUES_BYTES = PAGE_TOKENS * HEAD_DIM            # 8192
FP8_PAGE_BYTES = FP8_VALUES_BYTES + PAGE_TOKENS * 4  # 8448
FP4_VALUES_BYTES = PAGE_TOKENS * HEAD_DIM // 2       # 4096
FP4_BSCALE_OFFSET = FP4_VALUES_BYTES                 # 4096
FP4_BSCALE_BYTES = PAGE_TOKENS * HEAD_DIM // 16      # 512
FP4_GSCALE_OFFSET = FP4_BSCALE_OFFSET + FP4_BSCALE_BYTES  # 4608
FP4_PAGE_BYTES = FP4_GSCALE_OFFSET + PAGE_TOKENS * 4  # 4864
MX_BLOCK = 32
MXFP4_SCALE_OFFSET = FP4_VALUES_BYTES                 # 4096
MXFP4_PAGE_BYTES = MXFP4_SCALE_OFFSET + PAGE_TOKENS * HEAD_DIM // MX_BLOCK  # 4352
UE8M0_NAN = 0xFF

E4M3_NAN = 0x7F
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def page_bytes(kv_format: int) -> int:
    return {KV_FP8: FP8_PAGE_BYTES, KV_FP4: FP4_PAGE_BYTES, KV_MXFP4: MXFP4_PAGE_BYTES}[kv_format]


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclass
class Workload:
    """One batch of decode-indexer inputs (host or device tensors)."""

    name: str
    kv_format: int
    q: torch.Tensor              # uint8 [T, H, D] e4m3 codes
    weights: torch.Tensor        # float32 [T, H]
    context_lens: torch.Tensor   # int32 [T]  (causal limit L_t of each row)
    indices: torch.Tensor | None  # int32 [T] request id per row, or None (plain)
    block_table: torch.Tensor    # int32 [T, max_pages], row-indexed, -1 padded
    kv_cache: torch.Tensor       # uint8 [num_pages, page_stride]
    page_stride: int
    logits_stride: int           # >= round_up(max L_t, 64)
    topk: int
    logits_dtype: int            # LOGITS_F32 or LOGITS_BF16
    request_lens: list[int] = field(default_factory=list)
    rows_per_request: list[int] = field(default_factory=list)
    seed: int = 0
    q_scale: torch.Tensor | None = None  # uint8 [T, H, D/32] ue8m0 (MXFP4 only; q is then packed e2m1)

    @property
    def num_rows(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    def to(self, device) -> "Workload":
        def mv(x):
            return None if x is None else x.to(device)
        return Workload(self.name, self.kv_format, mv(self.q), mv(self.weights),
                        mv(self.context_lens), mv(self.indices), mv(self.block_table),
                        mv(self.kv_cache), self.page_stride, self.logits_stride,
                        self.topk, self.logits_dtype, list(self.request_lens),
                        list(self.rows_per_request), self.seed, mv(self.q_scale))


# ---------------------------------------------------------------------------
# quantisers (input encoding only)
# ---------------------------------------------------------------------------

def e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even e4m3fn codes of ``x`` (values must be within +-448)."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def e4m3_decode(codes: torch.Tensor) -> torch.Tensor:
    """Value of e4m3fn codes via torch's own float8 conversion (float32)."""
    return codes.view(torch.float8_e4m3fn).to(torch.float32)


def e2m1_codes(x: torch.Tensor) -> torch.Tensor:
    """4-bit e2m1 codes of ``x`` (round to nearest, ties to even code, clamp +-6).

    Magnitude code m in 0..7 stands for {0, .5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the
    sign.  Ties (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) go to the even code.
    """
    a = x.abs()
    m = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
         + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
         + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
         + (a > 5.0).to(torch.uint8))
    sign = ((x < 0) & (m > 0)).to(torch.uint8) << 3
    return m | sign


def quantize_keys_fp8(keys: torch.Tensor):
    """Per-token e4m3 quantisation: scale = amax / 448 (fp32), codes = e4m3(k / scale).

    An all-zero token gets scale 1 so that every key scale is positive.
    Returns (codes uint8 [N, D], scales float32 [N]).
    """
    amax = keys.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    codes = e4m3_codes(keys / scale[:, None])
    return codes, scale


def quantize_keys_fp4(keys: torch.Tensor):
    """Two-level FP4 quantisation of keys [N, D].

    g = amax / (448 * 6) per token (1 for an all-zero token); block scale
    s_b = e4m3(amax_b / (6 g)) per 16 elements; element code = e2m1(k / (s_b g)).
    A block whose scale rounds to zero stores zero codes.
    Returns (packed uint8 [N, D/2], block scale codes uint8 [N, D/16],
    token scales float32 [N]).
    """
    n, d = keys.shape
    amax = keys.abs().amax(dim=-1)
    g = torch.where(amax > 0, amax / (E4M3_MAX * E2M1_MAX), torch.ones_like(amax)).to(torch.float32)
    blocks = keys.view(n, d // 16, 16)
    bamax = blocks.abs().amax(dim=-1)
    bs_codes = e4m3_codes(bamax / (E2M1_MAX * g[:, None]))
    bs_val = e4m3_decode(bs_codes)
    denom = bs_val * g[:, None]
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    x = blocks / safe[..., None]
    codes = e2m1_codes(x)
    codes = torch.where((denom > 0)[..., None], codes, torch.zeros_like(codes)).view(n, d)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed, bs_codes, g


def quantize_mxfp4(x: torch.Tensor):
    """OCP MX FP4 quantisation of x [..., D] in blocks of 32 along the last dim.

    Shared scale 2^(floor(log2(amax_b)) - 2) (2 = the largest e2m1 exponent),
    stored as the ue8m0 code floor(log2(amax_b)) - 2 + 127 (127, scale 1, for an
    all-zero block); element code = e2m1(x / scale), saturating at +-6.
    Returns (packed uint8 [..., D/2], scale codes uint8 [..., D/32]).
    """
    shp = x.shape
    d = shp[-1]
    blocks = x.reshape(-1, d // MX_BLOCK, MX_BLOCK).to(torch.float32)
    amax = blocks.abs().amax(dim=-1)
    expo = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 2,
                       torch.zeros_like(amax))
    expo = expo.clamp(-127, 127)
    codes_s = (expo + 127).to(torch.uint8)
    scale = torch.exp2(expo)
    codes = e2m1_codes(blocks / scale[..., None]).view(-1, d)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.view(*shp[:-1], d // 2), codes_s.view(*shp[:-1], d // MX_BLOCK)


# ---------------------------------------------------------------------------
# workload builder
# ---------------------------------------------------------------------------

def build(name: str, request_lens, rows_per_request, *, kv_format=KV_FP8, topk=2048,
          logits_dtype=LOGITS_F32, seed=0, plain_indices=False, pool_factor=2.0,
          page_stride=None, device="cpu", heads=HEADS, head_dim=HEAD_DIM,
          logits_stride=None, key_std=1.0) -> Workload:
    """Build a seeded workload.

    request_lens[r]      L_r, keys cached for request r (the last row's causal limit)
    rows_per_request[r]  n_r, query rows of request r (1 for plain decode)
    plain_indices        pass ``indices=None`` (each row its own request)
    pool_factor          physical pool size / pages used (pages are shuffled)
    """
    assert len(request_lens) == len(rows_per_request)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B = len(request_lens)
    n_r = [int(x) for x in rows_per_request]
    L_r = [int(x) for x in request_lens]
    for L, n in zip(L_r, n_r):
        assert n >= 1 and L >= n - 1, "each row needs a non-negative causal limit"
    T = sum(n_r)
    pbytes = page_bytes(kv_format)
    stride = pbytes if page_stride is None else int(page_stride)
    assert stride >= pbytes and stride % 16 == 0

    # rows
    ctx = []
    req_of_row = []
    for r in range(B):
        for j in range(n_r[r]):
            ctx.append(L_r[r] - n_r[r] + 1 + j)
            req_of_row.append(r)
    context_lens = torch.tensor(ctx, dtype=torch.int32)
    indices = None if plain_indices else torch.tensor(req_of_row, dtype=torch.int32)
    if plain_indices:
        assert all(n == 1 for n in n_r)

    # pages
    pages_r = [math.ceil(L / PAGE_TOKENS) for L in L_r]
    used = sum(pages_r)
    num_pages = max(1, int(math.ceil(used * pool_factor)))
    perm = torch.randperm(num_pages, generator=gen, device=device).to("cpu")
    max_pages = max(1, max(pages_r) if pages_r else 1)
    bt_req = torch.full((B, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for r in range(B):
        if pages_r[r]:
            bt_req[r, : pages_r[r]] = perm[cursor: cursor + pages_r[r]].to(torch.int32)
        cursor += pages_r[r]
    block_table = bt_req[torch.tensor(req_of_row, dtype=torch.long)] if T else bt_req[:0]

    # key pool, poisoned; keys are drawn request by request to bound memory
    kv = torch.empty((num_pages, stride), dtype=torch.uint8, device=device)
    _poison(kv, kv_format)
    views = _page_views(kv, kv_format)
    for r in range(B):
        L = L_r[r]
        if L == 0:
            continue
        keys = torch.randn((L, head_dim), generator=gen, device=device,
                           dtype=torch.float32) * key_std
        pos = torch.arange(L, device=device)
        page = bt_req[r].to(device=device, dtype=torch.long)[pos // PAGE_TOKENS]
        slot = pos % PAGE_TOKENS
        if kv_format == KV_FP8:
            codes, scale = quantize_keys_fp8(keys)
            views["values"][page, slot] = codes
            views["scale"][page, slot] = scale.contiguous().view(torch.uint8).view(-1, 4)
        elif kv_format == KV_FP4:
            packed, bs, g = quantize_keys_fp4(keys)
            views["values"][page, slot] = packed
            views["bscale"][page, slot] = bs
            views["scale"][page, slot] = g.contiguous().view(torch.uint8).view(-1, 4)
        else:
            packed, es = quantize_mxfp4(keys)
            views["values"][page, slot] = packed
            views["bscale"][page, slot] = es
        del keys

    qf = torch.randn((T, heads, head_dim), generator=gen, device=device, dtype=torch.float32)
    q_scale = None
    if kv_format == KV_MXFP4:
        q, q_scale = quantize_mxfp4(qf)
    else:
        q = e4m3_codes(qf)
    weights = (torch.randn((T, heads), generator=gen, device=device, dtype=torch.float32)
               / math.sqrt(heads))
    max_ctx = max(ctx) if ctx else 0
    lstride = round_up(max(max_ctx, 1), PAGE_TOKENS) if logits_stride is None else int(logits_stride)
    return Workload(name, kv_format, q, weights, context_lens.to(device),
                    None if indices is None else indices.to(device),
                    block_table.to(device), kv, stride, lstride, int(topk), int(logits_dtype),
                    L_r, n_r, seed, q_scale)


def _poison(kv: torch.Tensor, kv_format: int) -> None:
    nan4 = torch.tensor([float("nan")], dtype=torch.float32).view(torch.uint8)
    if kv_format == KV_FP8:
        kv[:, :FP8_VALUES_BYTES] = E4M3_NAN
        kv[:, FP8_VALUES_BYTES:FP8_PAGE_BYTES] = nan4.repeat(PAGE_TOKENS).to(kv.device)
        kv[:, FP8_PAGE_BYTES:] = 0xA5
    elif kv_format == KV_MXFP4:
        kv[:, :FP4_VALUES_BYTES] = 0x77          # e2m1 +6 in both nibbles
        kv[:, MXFP4_SCALE_OFFSET:MXFP4_PAGE_BYTES] = UE8M0_NAN
        kv[:, MXFP4_PAGE_BYTES:] = 0xA5
    else:
        kv[:, :FP4_VALUES_BYTES] = 0x77          # e2m1 +6 in both nibbles
        kv[:, FP4_BSCALE_OFFSET:FP4_GSCALE_OFFSET] = E4M3_NAN
        kv[:, FP4_GSCALE_OFFSET:FP4_PAGE_BYTES] = nan4.repeat(PAGE_TOKENS).to(kv.device)
        kv[:, FP4_PAGE_BYTES:] = 0xA5


def _page_views(kv: torch.Tensor, kv_format: int) -> dict:
    """Strided [num_pages, 64, bytes] views of the regions inside every page."""
    n, stride = kv.shape
    if kv_format == KV_FP8:
        return {
            "values": kv.as_strided((n, PAGE_TOKENS, HEAD_DIM), (stride, HEAD_DIM, 1), 0),
            "scale": kv.as_strided((n, PAGE_TOKENS, 4), (stride, 4, 1), FP8_VALUES_BYTES),
        }
    if kv_format == KV_MXFP4:
        return {
            "values": kv.as_strided((n, PAGE_TOKENS, HEAD_DIM // 2), (stride, HEAD_DIM // 2, 1), 0),
            "bscale": kv.as_strided((n, PAGE_TOKENS, HEAD_DIM // MX_BLOCK), (stride, HEAD_DIM // MX_BLOCK, 1),
                                    MXFP4_SCALE_OFFSET),
        }
    return {
        "values": kv.as_strided((n, PAGE_TOKENS, HEAD_DIM // 2), (stride, HEAD_DIM // 2, 1), 0),
        "bscale": kv.as_strided((n, PAGE_TOKENS, HEAD_DIM // 16), (stride, HEAD_DIM // 16, 1),
                                FP4_BSCALE_OFFSET),
        "scale": kv.as_strided((n, PAGE_TOKENS, 4), (stride, 4, 1), FP4_GSCALE_OFFSET),
    }


# ---------------------------------------------------------------------------
# the five decode configurations and small variants
# ---------------------------------------------------------------------------

def _uniform_ints(gen, lo, hi, n):
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=gen)]


def config_spec(name: str) -> dict:
    """Keyword arguments of build() for a named decode workload.

    tiny        B=2, L=[300, 517], one row each, k=256, seed 0
    plain       B=64, L ~ U{4096..32768}, one row each (indices=arange), k=2048, seed 1
    mtp         B=128, two rows each (indices=i//2), L ~ U{8192..65536}, k=2048, seed 2
    varlen      B=40, L = 120000 + U{-2048..2048}, rows ~ U{1..6}, k=2048, seed 3
    fp4_varlen  as varlen with FP4 keys and BF16 logits, seed 4
    mxfp4_varlen  as varlen with MXFP4 keys and q and BF16 logits, seed 6
    prefill     B=2, L=8192, the last 4096 tokens of each prompt as rows (T=8192),
                k=2048, seed 5 (use prefill_view for the prefill-tagged form)
    """
    g = torch.Generator()
    if name == "tiny":
        return dict(request_lens=[300, 517], rows_per_request=[1, 1], topk=256, seed=0)
    if name == "plain":
        g.manual_seed(1)
        return dict(request_lens=_uniform_ints(g, 4096, 32768, 64), rows_per_request=[1] * 64,
                    topk=2048, seed=1)
    if name == "mtp":
        g.manual_seed(2)
        return dict(request_lens=_uniform_ints(g, 8192, 65536, 128),
                    rows_per_request=[2] * 128, topk=2048, seed=2)
    if name in ("varlen", "fp4_varlen", "mxfp4_varlen"):
        seed = {"varlen": 3, "fp4_varlen": 4, "mxfp4_varlen": 6}[name]
        g.manual_seed(seed)
        lens = [120000 + d for d in _uniform_ints(g, -2048, 2048, 40)]
        rows = _uniform_ints(g, 1, 6, 40)
        kw = dict(request_lens=lens, rows_per_request=rows, topk=2048, seed=seed)
        if name == "fp4_varlen":
            kw.update(kv_format=KV_FP4, logits_dtype=LOGITS_BF16)
        if name == "mxfp4_varlen":
            kw.update(kv_format=KV_MXFP4, logits_dtype=LOGITS_BF16)
        return kw
    if name == "prefill":
        # a prefill chunk: the second halves of two 8192-token prompts
        return dict(request_lens=[8192, 8192], rows_per_request=[4096, 4096], topk=2048, seed=5)
    raise ValueError(f"unknown workload {name!r}")


def config(name: str, device="cpu", **overrides) -> Workload:
    """Build a named decode workload (see config_spec)."""
    kw = config_spec(name)
    kw.update(overrides)
    return build(name, device=device, **kw)


def config_rows(name: str, plain_indices: bool = False):
    """(context_lens, indices) of a named workload, without building its key pool."""
    kw = config_spec(name)
    ctx, ids = [], []
    for r, (L, n) in enumerate(zip(kw["request_lens"], kw["rows_per_request"])):
        for j in range(n):
            ctx.append(L - n + 1 + j)
            ids.append(r)
    ctx = torch.tensor(ctx, dtype=torch.int32)
    return ctx, (None if plain_indices else torch.tensor(ids, dtype=torch.int32))


CONFIG_NAMES = ("tiny", "plain", "mtp", "varlen", "fp4_varlen")


def padded_rows(wl: Workload):
    """The (B, max_n) padded layout of a varlen workload.

    Returns (row_of_slot [B*max_n] with -1 for padding slots, max_n).  Padding
    slots repeat the request's last row's causal limit, as a non-varlen decode
    batch padded to (B, max_decode_len) would.
    """
    n_r = wl.rows_per_request
    max_n = max(n_r) if n_r else 0
    out = []
    t = 0
    for n in n_r:
        for j in range(max_n):
            out.append(t + j if j < n else -1)
        t += n
    return torch.tensor(out, dtype=torch.long), max_n


# ---------------------------------------------------------------------------
# decode context parallelism: one rank's shard of a workload
# ---------------------------------------------------------------------------

def dcp_owner(g, world: int, interleave: int):
    """Rank holding global token g: blocks of `interleave` tokens, round robin."""
    return (g // interleave) % world


def dcp_shard(wl: Workload, rank: int, world: int, interleave: int) -> Workload:
    """Rank `rank`'s shard of `wl`: each request's tokens owned by the rank, in
    global order, repacked into fresh pages of the same format (local position
    l = the l-th owned token), a local block table and local causal limits
    (owned tokens below each row's limit).  q, weights and request ids are
    unchanged."""
    fmt = wl.kv_format
    kv = wl.kv_cache.cpu()
    bt = wl.block_table.cpu()
    ctx = wl.context_lens.cpu().to(torch.int64)
    ind = None if wl.indices is None else wl.indices.cpu()
    T = int(ctx.shape[0])
    src = _page_views(kv, fmt)
    # requests: runs of equal ids (every row alone without ids)
    runs = []
    t = 0
    while t < T:
        u = t + 1
        while ind is not None and u < T and int(ind[u]) == int(ind[t]):
            u += 1
        runs.append((t, u))
        t = u
    pages, row_pages, ctx_loc = [], [None] * T, torch.zeros(T, dtype=torch.int32)
    n_pages = 0
    for t0, t1 in runs:
        lens = ctx[t0:t1].clamp(min=0)
        t_big = t0 + int(torch.argmax(lens))
        lmax = int(lens.max())
        g = torch.arange(lmax, dtype=torch.int64)
        own = g[dcp_owner(g, world, interleave) == rank]
        n_loc = int(own.shape[0])
        np_loc = (n_loc + PAGE_TOKENS - 1) // PAGE_TOKENS
        new = torch.zeros((np_loc, kv.shape[1]), dtype=torch.uint8)
        dst = _page_views(new, fmt)
        if n_loc:
            pg = bt[t_big, own // PAGE_TOKENS].to(torch.int64)
            sl = own % PAGE_TOKENS
            loc = torch.arange(n_loc, dtype=torch.int64)
            for key in src:
                dst[key][loc // PAGE_TOKENS, loc % PAGE_TOKENS] = src[key][pg, sl]
        pages.append(new)
        ids = torch.arange(n_pages, n_pages + np_loc, dtype=torch.int32)
        n_pages += np_loc
        for tt in range(t0, t1):
            row_pages[tt] = ids
            gg = torch.arange(int(lens[tt - t0]), dtype=torch.int64)
            ctx_loc[tt] = int((dcp_owner(gg, world, interleave) == rank).sum())
    width = max(1, max(int(r.shape[0]) for r in row_pages))
    bt_loc = torch.full((T, width), -1, dtype=torch.int32)
    for tt in range(T):
        bt_loc[tt, : row_pages[tt].shape[0]] = row_pages[tt]
    pool = torch.cat(pages) if n_pages else torch.zeros((1, kv.shape[1]), dtype=torch.uint8)
    stride = round_up(max(1, int(ctx_loc.max()) if T else 1), 64)
    return Workload(f"{wl.name}-dcp{rank}of{world}i{interleave}", fmt, wl.q.cpu(), wl.weights.cpu(),
                    ctx_loc, ind, bt_loc, pool.contiguous(), int(kv.shape[1]), stride, wl.topk,
                    wl.logits_dtype, list(wl.request_lens), list(wl.rows_per_request), wl.seed,
                    None if wl.q_scale is None else wl.q_scale.cpu())


# ---------------------------------------------------------------------------
# prefill chunks in the prefill-tagged form
# ---------------------------------------------------------------------------

@dataclass
class Prefill:
    """A prefill chunk over the paged cache, tagged as the indexer's prefill
    path tags it: the requests' keys laid end to end (local_cu_seq_lens,
    [B + 1]), each token row t tagged with its request's start ks and the end
    ke of the keys it sees; block_table is per request."""

    q: torch.Tensor                  # uint8 [T, H, D]
    weights: torch.Tensor            # float32 [T, H]
    cu_seqlen_ks: torch.Tensor       # int32 [T]
    cu_seqlen_ke: torch.Tensor       # int32 [T]
    local_cu_seq_lens: torch.Tensor  # int32 [B + 1]
    block_table: torch.Tensor        # int32 [B, max_pages]
    kv_cache: torch.Tensor
    kv_format: int
    page_stride: int
    logits_stride: int
    topk: int
    logits_dtype: int
    q_scale: torch.Tensor | None = None  # MXFP4 q scales

    @property
    def num_rows(self) -> int:
        return int(self.cu_seqlen_ks.shape[0])

    @property
    def num_requests(self) -> int:
        return int(self.local_cu_seq_lens.shape[0]) - 1

    def to(self, device) -> "Prefill":
        return Prefill(*(x.to(device) if isinstance(x, torch.Tensor) else x
                         for x in (self.q, self.weights, self.cu_seqlen_ks, self.cu_seqlen_ke,
                                   self.local_cu_seq_lens, self.block_table, self.kv_cache)),
                       self.kv_format, self.page_stride, self.logits_stride, self.topk,
                       self.logits_dtype, None if self.q_scale is None else self.q_scale.to(device))


def prefill_view(wl: Workload) -> Prefill:
    """The prefill-tagged form of a workload whose rows are the last n_r
    tokens of each request (row j of request r at causal limit
    L_r - n_r + 1 + j): ks = the request's start in the concatenated keys,
    ke = ks + L_t, and one block-table row per request."""
    lens = [int(x) for x in wl.request_lens]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    ks, last = [], []
    t = 0
    for r, n in enumerate(wl.rows_per_request):
        ks += [cu[r]] * int(n)
        t += int(n)
        last.append(t - 1)
    ks = torch.tensor(ks, dtype=torch.int32)
    ctx = wl.context_lens.cpu()
    bt = wl.block_table.cpu()[torch.tensor(last, dtype=torch.int64)].contiguous()
    return Prefill(wl.q.cpu(), wl.weights.cpu(), ks, ks + ctx, torch.tensor(cu, dtype=torch.int32), bt,
                   wl.kv_cache.cpu(), wl.kv_format, wl.page_stride, wl.logits_stride, wl.topk,
                   wl.logits_dtype, None if wl.q_scale is None else wl.q_scale.cpu())
