"""GPU parity of tsi_topk_overlap (cross-layer top-k overlap) against the CPU oracle:
random index rows with padding, the index rows of two indexers, and sampled rows of a
full-size L=131072 pair (through the C ABI).  Counts are integers: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from workloads import get_config, make_indexer_inputs

pytestmark = pytest.mark.gpu


def _random_pair(rows, topk, universe, seed):
    """Two [rows, topk] index buffers: distinct positions per row, a shared part of random
    size between them, -1 padding at the tail of some rows."""
    rng = np.random.default_rng(seed)
    a = -np.ones((rows, topk), dtype=np.int32)
    b = -np.ones((rows, topk), dtype=np.int32)
    for r in range(rows):
        n = topk if rng.random() < 0.7 else int(rng.integers(0, topk + 1))
        m = min(n, universe // 2)
        pool = rng.choice(universe, size=min(universe, 2 * m), replace=False)
        common = int(rng.integers(0, m + 1))
        ra = pool[:m]
        rb = np.concatenate([ra[:common], pool[m:m + (m - common)]])
        a[r, :m] = rng.permutation(ra)
        b[r, :len(rb)] = rng.permutation(rb)
    return a, b


@pytest.mark.parametrize("rows,topk,universe", [(1, 1, 4), (37, 7, 50), (500, 64, 1000),
                                                 (300, 2048, 131072), (64, 2048, 4096)])
def test_overlap_random_rows_exact(cuda_lib, rows, topk, universe):
    a, b = _random_pair(rows, topk, universe, seed=rows * 7 + topk)
    inter, card = cuda_lib.topk_overlap(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    cuda_lib.device_status()
    ref_i, ref_c = oracle.topk_overlap(a, b)
    assert np.array_equal(inter.cpu().numpy(), ref_i)
    assert np.array_equal(card.cpu().numpy(), ref_c)


def test_overlap_all_padding_and_identical_rows(cuda_lib):
    a = -np.ones((5, 16), dtype=np.int32)
    a[1] = np.arange(16)
    a[2, :3] = [9, 2, 5]
    inter, card = cuda_lib.topk_overlap(torch.from_numpy(a).cuda(), torch.from_numpy(a).cuda())
    cuda_lib.device_status()
    assert inter.cpu().tolist() == [0, 16, 3, 0, 0]
    assert card.cpu().tolist() == [0, 16, 3, 0, 0]


def test_overlap_of_two_indexers(cuda_lib):
    # two layers' indexers over the same sequence: the Full layers of two IndexShare groups
    cfg = get_config(4).with_(T=3000, S=3000)
    idx = []
    for group in (0, 1):
        qI, kI, w = make_indexer_inputs(cfg, group, "cuda")
        idx.append(cuda_lib.indexer_topk(qI, kI, w, cfg.topk))
    inter, card = cuda_lib.topk_overlap(idx[0], idx[1])
    cuda_lib.device_status()
    ref_i, ref_c = oracle.topk_overlap(idx[0].cpu().numpy(), idx[1].cpu().numpy())
    assert np.array_equal(inter.cpu().numpy(), ref_i)
    assert np.array_equal(card.cpu().numpy(), ref_c)
    # rows with at most k causal keys select all of them in both layers
    short = np.arange(cfg.topk)
    assert np.array_equal(ref_i[short], short + 1)


def test_overlap_full_size_sampled(cuda_lib):
    cfg = get_config(4)
    idx = []
    for group in (0, 1):
        qI, kI, w = make_indexer_inputs(cfg, group, "cuda")
        # [B, T, k] -> [rows, k]: the sampled row numbers index this view
        idx.append(cuda_lib.indexer_topk(qI, kI, w, cfg.topk).view(-1, cfg.topk))
        del qI, kI, w
    n_rows = idx[0].shape[0]
    assert n_rows == cfg.B * cfg.T
    inter, card = cuda_lib.topk_overlap(idx[0], idx[1])
    cuda_lib.device_status()
    rows = np.random.default_rng(11).choice(n_rows, size=256, replace=False)
    rows[:4] = [0, cfg.topk - 1, cfg.topk, n_rows - 1]
    assert rows.min() >= 0 and rows.max() < n_rows
    sel = torch.from_numpy(rows).cuda()
    ref_i, ref_c = oracle.topk_overlap(idx[0][sel].cpu().numpy(), idx[1][sel].cpu().numpy())
    assert np.array_equal(inter[sel].cpu().numpy(), ref_i)
    assert np.array_equal(card[sel].cpu().numpy(), ref_c)
