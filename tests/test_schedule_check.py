"""The schedule validity checker (tests/schedule_check.py) on schedules worked
out by hand: it accepts a valid one and rejects each kind of broken one.  (The
GPU tests apply it to the metadata call's output.)"""
import numpy as np
import pytest

from schedule_check import MAGIC, check_schedule


def _words(hdr, left, right, grs, pos, sus, spp):
    spp = np.asarray(spp, dtype=np.int64)
    return np.array(list(hdr) + list(left) + list(right) + list(grs) + list(pos) + list(sus) +
                    list(spp & 0xFFFFFFFF) + list(spp >> 32), dtype=np.int64)


def _two_requests():
    # rows: request 0 (L = 300, 3 tiles), request 1 (L = 517, 5 tiles); 2 SMs.
    # SM 0 takes units [0, 2) and [6, 8), SM 1 takes [2, 4) and [4, 6).
    ctx, ids, S = [300, 517], [0, 1], 2
    kw = dict(hdr=[MAGIC, 2, 1, 2, 2, 8, 128, 8], left=[0, 2, 4], right=[8, 6, 4], grs=[0, 1, 2],
              pos=[0 | 1 << 24, 1 | 1 << 24, 2], sus=[0, 3, 8], spp=[0, 3, 8])
    return ctx, ids, S, kw


def test_accepts_a_valid_schedule():
    ctx, ids, S, kw = _two_requests()
    units, pairs = check_schedule(_words(**kw), ctx, ids, S)
    assert list(units) == [4, 4] and list(pairs) == [4, 4]


def test_accepts_rows_sorted_by_group_size():
    # request 0: 3 rows (L = 130..132 -> 2 tiles), request 1: 1 row (L = 256 -> 2 tiles);
    # sorted order puts the 1-row group first; one SM owns everything
    ctx, ids, S = [130, 131, 132, 256], [0, 0, 0, 1], 1
    words = _words(hdr=[MAGIC, 4, 1, 1, 2, 4, 128, 8], left=[0, 1], right=[4, 1], grs=[0, 3, 4, 4, 4],
                   pos=[3 | 1 << 24, 0 | 3 << 24, 4, 4, 4], sus=[0, 2, 4, 4, 4], spp=[0, 2, 8, 8, 8])
    units, pairs = check_schedule(words, ctx, ids, S)
    assert list(units) == [4] and list(pairs) == [8]


@pytest.mark.parametrize("field,value", [
    ("hdr", [MAGIC + 1, 2, 1, 2, 2, 8, 128, 8]),          # wrong magic
    ("hdr", [MAGIC, 2, 0, 2, 2, 8, 128, 8]),              # plain flag on a varlen schedule
    ("left", [0, 3, 4]),                                  # SM 0 five units, SM 1 three
    ("right", [8, 6, 5]),                                 # left and right ends do not meet
    ("left", [0, 2, 5]),                                  # a unit owned twice
    ("pos", [1 | 1 << 24, 0 | 1 << 24, 2]),               # equal row counts out of row order
    ("pos", [0 | 2 << 24, 1 | 1 << 24, 2]),               # wrong row count
    ("sus", [0, 4, 8]),                                   # wrong tile count
    ("spp", [0, 3, 9]),                                   # wrong pair prefix
    ("grs", [0, 2, 2]),                                   # one group spans two requests
])
def test_rejects_a_broken_schedule(field, value):
    ctx, ids, S, kw = _two_requests()
    kw[field] = value
    with pytest.raises(AssertionError):
        check_schedule(_words(**kw), ctx, ids, S)


def test_rejects_a_group_cut_before_it_is_full():
    # one request of 9 rows must be cut 8 + 1; a 4 + 5 cut is rejected
    ctx, ids, S = [100 + i for i in range(9)], [0] * 9, 1
    ok = _words(hdr=[MAGIC, 9, 1, 1, 2, 2, 128, 8], left=[0, 1], right=[2, 1],
                grs=[0, 8] + [9] * 8, pos=[8 | 1 << 24, 0 | 8 << 24] + [9] * 8,
                sus=[0, 1] + [2] * 8, spp=[0, 1] + [9] * 8)
    check_schedule(ok, ctx, ids, S)
    bad = _words(hdr=[MAGIC, 9, 1, 1, 2, 2, 128, 8], left=[0, 1], right=[2, 1],
                 grs=[0, 4] + [9] * 8, pos=[0 | 4 << 24, 4 | 5 << 24] + [9] * 8,
                 sus=[0, 1] + [2] * 8, spp=[0, 4] + [9] * 8)
    with pytest.raises(AssertionError):
        check_schedule(bad, ctx, ids, S)


def _rows_sorted(spp):
    ctx, ids, S = [130, 131, 132, 256], [0, 0, 0, 1], 1
    words = _words(hdr=[MAGIC, 4, 1, 1, 2, 4, 128, 8], left=[0, 1], right=[4, 1], grs=[0, 3, 4, 4, 4],
                   pos=[3 | 1 << 24, 0 | 3 << 24, 4, 4, 4], sus=[0, 2, 4, 4, 4], spp=spp)
    return words, ctx, ids, S


def test_accepts_weights_growing_faster_than_rows():
    # the same two groups with a unit of n rows weighing 4n + n^2 (5 and 21)
    words, ctx, ids, S = _rows_sorted([0, 10, 52, 52, 52])
    units, weight = check_schedule(words, ctx, ids, S)
    assert list(units) == [4] and list(weight) == [52]


@pytest.mark.parametrize("spp", [
    [0, 10, 18, 18, 18],   # a 3-row unit weighs less (4) than a 1-row unit (5)
    [0, 10, 51, 51, 51],   # 41 over 2 units: not a whole weight per unit
])
def test_rejects_bad_unit_weights(spp):
    words, ctx, ids, S = _rows_sorted(spp)
    with pytest.raises(AssertionError):
        check_schedule(words, ctx, ids, S)


def test_rejects_two_weights_for_one_row_count():
    # both groups have 1 row; the prefix weighs the first one's units 1 and the second's 2
    ctx, ids, S, kw = _two_requests()
    kw["spp"] = [0, 3, 13]
    with pytest.raises(AssertionError):
        check_schedule(_words(**kw), ctx, ids, S)
