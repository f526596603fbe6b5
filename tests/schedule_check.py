"""Validity checker for the schedule words of dsa_paged_mqa_logits_metadata.

The pages fix the metadata call's inputs and purpose (PR 47469 "Route SM100
sparse-indexer decode through varlen paged MQA logits", Purpose and Changes:
balance the requests' K-block work over the SMs, rows with equal adjacent
request ids forming one request), not a split rule.  So no oracle says which
SM gets which unit.  This checker reads no weight or tuning constant of the
library: it checks that the words are a valid work assignment for the given
rows, in the layout include/dsa_indexer.h states, and that the work is
balanced in the two quantities the logits kernel pays for:

* header fields: magic, rows, varlen flag, SM count, group and unit counts;
* groups: the maximal runs of equal request ids, cut into consecutive pieces
  of at most the header's group size, the cut only where a piece is full;
* sorted positions: a permutation of the groups, in non-decreasing row count
  (equal counts in row order), each with its own row count;
* unit starts: each group holds ceil(max causal limit / tile) units, laid end
  to end in position order;
* weights: the prefix words after the unit starts carry the weight before
  each position; every unit of a group of n rows weighs the same w(n) >= 1,
  one value per row count, not decreasing with n (w(n) = n counts (tile,
  row) pairs; the schedule may weigh rows more than linearly, and this
  checker reads the weights from the words, not from the library);
* ownership: the SMs' left ranges tile [0, m) and their right ranges tile
  [m, U), so every unit belongs to exactly one SM;
* balance: every SM owns floor or ceil of U / S units, and its weight lies
  within twice the largest unit weight of the total over S.

The real proof that any such schedule gives the right logits is the logits
parity against the oracle at several SM counts.
"""
import numpy as np

MAGIC = 0x44534132
POS_SHIFT = 24


def layout(S, T):
    left = 8
    right = left + S + 1
    grs = right + S + 1
    pos = grs + T + 1
    sus = pos + T + 1
    spp_lo = sus + T + 1
    spp_hi = spp_lo + T + 1
    return dict(left=left, right=right, grs=grs, pos=pos, sus=sus, spp_lo=spp_lo, spp_hi=spp_hi,
                words=spp_hi + T + 1)


def check_schedule(words, context_lens, indices, S, balance=True):
    """Assert that `words` is a valid, balanced schedule; return per-SM (units, weight)."""
    w = np.asarray(words).astype(np.int64)
    ctx = np.asarray(context_lens).astype(np.int64)
    ids = None if indices is None else np.asarray(indices).astype(np.int64)
    T = int(ctx.shape[0])
    L = layout(S, T)
    assert w.shape[0] >= L["words"], "schedule shorter than its layout"
    hdr = w[:8]
    assert hdr[0] == MAGIC and hdr[1] == T and hdr[2] == (0 if ids is None else 1) and hdr[3] == S, hdr
    G, U, tile, cap = int(hdr[4]), int(hdr[5]), int(hdr[6]), int(hdr[7])
    assert 0 <= G <= T and tile > 0 and cap >= 1
    sec = {k: w[L[k]: L[k] + (S + 1 if k in ("left", "right") else T + 1)] for k in
           ("left", "right", "grs", "pos", "sus", "spp_lo", "spp_hi")}

    # groups in row order
    grs = sec["grs"]
    if T == 0:
        assert G == 0
    else:
        assert grs[0] == 0 and grs[G] == T and np.all(np.diff(grs[: G + 1]) > 0)
    assert np.all(grs[G:] == T)
    starts = set(int(x) for x in grs[:G])
    for g in range(G):
        a, b = int(grs[g]), int(grs[g + 1])
        assert b - a <= cap, f"group {g} has {b - a} rows"
        if ids is None:
            assert b - a == 1
        else:
            assert np.all(ids[a:b] == ids[a]), f"group {g} mixes requests"
            if b < T and ids[b] == ids[b - 1]:
                assert b - a == cap, f"group {g} cut before it is full"
    for t in range(1, T):
        if ids is None or ids[t] != ids[t - 1]:
            assert t in starts, f"row {t} starts a request but no group"

    # sorted positions
    pos = sec["pos"]
    r0 = pos[:G] & ((1 << POS_SHIFT) - 1)
    nr = pos[:G] >> POS_SHIFT
    assert sorted(int(x) for x in r0) == sorted(starts)
    size = {int(grs[g]): int(grs[g + 1] - grs[g]) for g in range(G)}
    assert all(int(n) == size[int(a)] for a, n in zip(r0, nr)), "a position carries the wrong row count"
    for k in range(G - 1):
        assert (nr[k], r0[k]) < (nr[k + 1], r0[k + 1]), f"positions {k}, {k + 1} out of order"
    assert np.all(pos[G:] == T)

    # units and pairs along the sorted order
    tiles = np.array([(max(0, int(ctx[a: a + n].max())) + tile - 1) // tile if n else 0
                      for a, n in zip(r0, nr)], dtype=np.int64)
    sus = sec["sus"]
    assert sus[0] == 0 and np.array_equal(np.diff(sus[: G + 1]), tiles) and sus[G] == U
    assert np.all(sus[G:] == U)
    spp = (sec["spp_lo"] & 0xFFFFFFFF) | (sec["spp_hi"] << 32)
    assert spp[0] == 0 and np.all(np.diff(spp[: G + 1]) >= 0)
    wt = {}  # unit weight of each row count, read from the words
    for k in range(G):
        dw = int(spp[k + 1] - spp[k])
        if tiles[k] == 0:
            assert dw == 0, f"position {k}: weight without units"
            continue
        assert dw % int(tiles[k]) == 0, f"position {k}: weight not a whole number per unit"
        w = dw // int(tiles[k])
        assert w >= 1 and wt.setdefault(int(nr[k]), w) == w, f"position {k}: {w} per unit for {nr[k]} rows"
    ws = [wt[n] for n in sorted(wt)]
    assert all(a <= b for a, b in zip(ws, ws[1:])), f"unit weight decreases with rows: {wt}"
    P = int(spp[G])
    assert np.all(spp[G:] == P)

    # ownership
    left, right = sec["left"], sec["right"]
    assert left[0] == 0 and right[0] == U
    assert np.all(np.diff(left) >= 0) and np.all(np.diff(right) <= 0)
    assert left[S] == right[S] and 0 <= left[S] <= U

    dens = np.repeat([wt.get(int(n), 0) for n in nr], tiles)

    def pairs(a, b):
        return int(dens[a:b].sum())

    units = np.array([(left[i + 1] - left[i]) + (right[i] - right[i + 1]) for i in range(S)])
    prs = np.array([pairs(left[i], left[i + 1]) + pairs(right[i + 1], right[i]) for i in range(S)])
    assert units.sum() == U and prs.sum() == P
    if balance and U:
        assert np.all(units >= U // S) and np.all(units <= -(-U // S)), (units.min(), units.max(), U / S)
        band = 2 * max(ws)
        assert np.all(np.abs(prs - P / S) <= band), (prs.min(), prs.max(), P / S)
    return units, prs
