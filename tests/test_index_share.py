"""IndexShare layer schedule and the cross-layer top-k overlap metric: oracle pins and
the host side of the C ABI (no GPU needed)."""
import itertools
import random

import numpy as np
import pytest

import oracle
import top_selection_indexer_gb300 as tsi


def _kinds(anchors):
    return "".join("F" if a == layer else "S" for layer, a in enumerate(anchors))


# ------------------------------------------------------------------ schedule: oracle pins

def test_schedule_config_of_the_pages():
    # "GLM 5.2: Built for Long Horizon Tasks" §5.2: index_topk_freq = 4,
    # index_skip_topk_offset = 3, and after the offset the types run full, shared, shared,
    # shared.  The layers before the offset keep their own indexer (reading).
    anchors = oracle.index_share_layers(16, freq=4, skip_offset=3)
    assert _kinds(anchors)[3:] == "FSSS" * 3 + "F"
    assert _kinds(anchors)[:3] == "FFF"
    assert anchors[4:7] == [3, 3, 3] and anchors[8:11] == [7, 7, 7]


def test_schedule_one_full_three_shared_groups():
    # "GLM-5.2 技术报告速览" §IndexShare: groups of four layers, 1 Full + 3 Shared, each
    # Shared layer inheriting the nearest Full layer's index set.
    anchors = oracle.index_share_layers(12, freq=4, skip_offset=0)
    assert anchors == [0, 0, 0, 0, 4, 4, 4, 4, 8, 8, 8, 8]


def test_schedule_freq_one_is_plain_dsa():
    assert oracle.index_share_layers(7, freq=1, skip_offset=0) == list(range(7))


def test_schedule_explicit_pattern_overrides():
    assert oracle.index_share_layers(6, freq=4, skip_offset=3, pattern="FSFFSS") == [0, 0, 2, 3, 3, 3]
    with pytest.raises(ValueError):
        oracle.index_share_layers(3, pattern="SFF")
    with pytest.raises(ValueError):
        oracle.index_share_layers(3, pattern="FF")


# ------------------------------------------------------------- schedule: native vs oracle

def test_schedule_native_matches_oracle():
    rng = random.Random(7)
    for n, freq, off in itertools.product(range(0, 20), range(1, 6), range(0, 6)):
        assert tsi.index_share_layers(n, freq, off) == oracle.index_share_layers(n, freq, off)
    for _ in range(200):
        n = rng.randint(1, 40)
        pat = "F" + "".join(rng.choice("FS") for _ in range(n - 1))
        assert tsi.index_share_layers(n, pattern=pat) == oracle.index_share_layers(n, pattern=pat)


@pytest.mark.parametrize("args", [(4, 0, 0, "SFFF"), (4, 4, 0, "FFF"), (4, 4, 0, "FFFFF"),
                                  (4, 4, 0, "FSXS"), (4, 0, 0, None), (4, 4, -1, None),
                                  (-1, 4, 0, None)])
def test_schedule_native_rejects_bad_arguments(args):
    n, freq, off, pat = args
    with pytest.raises(tsi.TSIError) as e:
        tsi.index_share_layers(n, freq, off, pat)
    assert e.value.status == tsi.ERR_INVALID_ARG


# ------------------------------------------------------------------- overlap: oracle pins

def _brute_overlap(a, b):
    # counting formulation, independent of set arithmetic: pairs of equal non-padding
    # entries (positions are distinct within a row)
    inter = sum(1 for x in a for y in b if x >= 0 and x == y)
    return inter, sum(1 for x in a if x >= 0)


def test_overlap_matches_pair_counting():
    rng = np.random.default_rng(3)
    for _ in range(50):
        k = int(rng.integers(1, 40))
        rows = []
        for _ in range(2):
            n = int(rng.integers(0, k + 1))
            r = rng.choice(60, size=n, replace=False)
            rows.append(np.concatenate([r, -np.ones(k - n, dtype=np.int64)]))
        inter, card = oracle.topk_overlap(rows[0][None], rows[1][None])
        assert (int(inter[0]), int(card[0])) == _brute_overlap(rows[0], rows[1])


def test_overlap_special_cases():
    a = np.array([[4, 9, 1, -1], [0, 1, 2, 3], [-1, -1, -1, -1]])
    same, card = oracle.topk_overlap(a, a)
    assert same.tolist() == [3, 4, 0] and card.tolist() == [3, 4, 0]
    # order inside a row does not matter; disjoint rows share nothing
    b = np.array([[1, 4, 9, -1], [7, 6, 5, 4], [0, 1, 2, 3]])
    inter, _ = oracle.topk_overlap(a, b)
    assert inter.tolist() == [3, 0, 0]


# --------------------------------------------------------------- overlap: host-side ABI

@pytest.fixture(scope="module")
def lib():
    from top_selection_indexer_gb300 import _build

    _build.build()
    return tsi.load()


FAKE = 0x10000


def test_overlap_rejects_bad_arguments(lib):
    assert lib.tsi_topk_overlap(FAKE, FAKE, 0, 16, FAKE, FAKE, None) == tsi.OK  # no rows
    assert lib.tsi_topk_overlap(FAKE, FAKE, 4, 0, FAKE, FAKE, None) == tsi.ERR_UNSUPPORTED
    assert lib.tsi_topk_overlap(FAKE, FAKE, 4, tsi.MAX_TOPK + 1, FAKE, FAKE, None) == \
        tsi.ERR_UNSUPPORTED
    assert lib.tsi_topk_overlap(FAKE, None, 4, 16, FAKE, FAKE, None) == tsi.ERR_INVALID_ARG
    assert lib.tsi_topk_overlap(FAKE + 4, FAKE, 4, 16, FAKE, FAKE, None) == tsi.ERR_INVALID_ARG
    assert lib.tsi_topk_overlap(FAKE, FAKE, -1, 16, FAKE, FAKE, None) == tsi.ERR_INVALID_ARG
