"""Context-parallel indexer (key shards + exchange + merge): oracle pins, the host side of
the C ABI, and the exchange over a world-size-2 gloo group on CPU (no GPU needed)."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import top_selection_indexer_gb300 as tsi


def _int_inputs(L, H_I, d_I, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randint(-4, 5, (L, H_I, d_I), generator=g).float()
    k = torch.randint(-4, 5, (L, d_I), generator=g).float()
    w = torch.randint(0, 4, (L, H_I), generator=g).float()
    return q, k, w


def _split(L, cuts):
    edges = [0] + list(cuts) + [L]
    return [(edges[i], edges[i + 1]) for i in range(len(edges) - 1)]


# ------------------------------------------------------------------------- oracle pins

def test_one_shard_is_the_indexer_topk():
    L, k = 90, 16
    q, kk, w = _int_inputs(L, 3, 8, 1)
    ref_idx, ref_sc = oracle.indexer_topk(q[None], kk[None], w[None], k)
    for t in range(L):
        sc, pos = oracle.shard_topk(q[t], kk, w[t], t, 0, k)
        n = len(pos)
        assert np.array_equal(pos, ref_idx[t, :n]) and (ref_idx[t, n:] == -1).all()
        assert np.array_equal(sc, ref_sc[t, :n])


@pytest.mark.parametrize("cuts", [(40,), (1, 2), (33, 34, 80), (7, 64, 65, 89)])
def test_merge_of_shards_is_the_whole_cache(cuts):
    # integer inputs with many ties: the lower position must win across shard borders too
    L, k = 90, 16
    q, kk, w = _int_inputs(L, 2, 4, 2)
    ref_idx, _ = oracle.indexer_topk(q[None], kk[None], w[None], k)
    for t in range(0, L, 3):
        lists = [oracle.shard_topk(q[t], kk[lo:hi], w[t], t, lo, k) for lo, hi in _split(L, cuts)]
        _, pos = oracle.merge_topk(lists, k)
        n = len(pos)
        assert np.array_equal(pos, ref_idx[t, :n]) and (ref_idx[t, n:] == -1).all()


# ------------------------------------------------------------------ host-side ABI checks

FAKE = 0x10000


@pytest.fixture(scope="module")
def lib():
    from top_selection_indexer_gb300 import _build

    _build.build()
    return tsi.load()


def _shard(lib, **kw):
    a = dict(q=FAKE, k=FAKE, w=FAKE, qk=tsi.E4M3, wd=tsi.BF16, B=1, T=4, S_total=100,
             off=0, S_shard=50, H=64, d=128, topk=8, kv=None, cand=FAKE, cnt=FAKE, ws=None,
             wsb=0, stream=None)
    a.update(kw)
    return lib.tsi_indexer_topk_shard(a["q"], a["k"], a["w"], a["qk"], a["wd"], a["B"], a["T"],
                                      a["S_total"], a["off"], a["S_shard"], a["H"], a["d"],
                                      a["topk"], a["kv"], a["cand"], a["cnt"], a["ws"], a["wsb"],
                                      a["stream"])


def test_shard_rejects_bad_arguments(lib):
    assert _shard(lib, off=60) == tsi.ERR_INVALID_ARG  # shard past the end of the cache
    assert _shard(lib, off=-1) == tsi.ERR_INVALID_ARG
    assert _shard(lib, topk=0) == tsi.ERR_UNSUPPORTED
    assert _shard(lib, cand=None) == tsi.ERR_INVALID_ARG
    assert _shard(lib, cnt=FAKE + 4) == tsi.ERR_INVALID_ARG
    assert _shard(lib, qk=9) == tsi.ERR_INVALID_ARG
    assert _shard(lib, B=0) == tsi.OK


def test_merge_rejects_bad_arguments(lib):
    assert lib.tsi_topk_merge(FAKE, FAKE, 2, 0, 8, FAKE, None, None) == tsi.OK
    assert lib.tsi_topk_merge(FAKE, FAKE, 0, 4, 8, FAKE, None, None) == tsi.ERR_INVALID_ARG
    assert lib.tsi_topk_merge(FAKE, FAKE, 1025, 4, 8, FAKE, None, None) == tsi.ERR_UNSUPPORTED
    assert lib.tsi_topk_merge(FAKE, FAKE, 2, 4, 0, FAKE, None, None) == tsi.ERR_UNSUPPORTED
    assert lib.tsi_topk_merge(FAKE, None, 2, 4, 8, FAKE, None, None) == tsi.ERR_INVALID_ARG


# ------------------------------------------------------- the exchange on a gloo group

def _rank_main(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    L, k = 120, 12
    q, kk, w = _int_inputs(L, 2, 4, 3)
    lo, hi = _split(L, [L * r // world for r in range(1, world)])[rank]
    rows = list(range(L))
    sc = torch.full((L, k), float("-inf"), dtype=torch.float64)
    pos = torch.full((L, k), -1, dtype=torch.int64)
    cnt = torch.zeros(L, dtype=torch.int32)
    for t in rows:  # this rank's shard, as tsi_indexer_topk_shard would leave it
        s_, p_ = oracle.shard_topk(q[t], kk[lo:hi], w[t], t, lo, k)
        sc[t, :len(p_)] = torch.from_numpy(s_)
        pos[t, :len(p_)] = torch.from_numpy(p_)
        cnt[t] = len(p_)
    all_sc, all_cnt = tsi.gather_candidates(sc, cnt)
    all_pos, _ = tsi.gather_candidates(pos, cnt)
    ok = True
    ref_idx, _ = oracle.indexer_topk(q[None], kk[None], w[None], k)
    for t in rows:
        lists = [(all_sc[r, t, :all_cnt[r, t]].numpy(), all_pos[r, t, :all_cnt[r, t]].numpy())
                 for r in range(world)]
        _, m = oracle.merge_topk(lists, k)
        n = len(m)
        ok &= bool(np.array_equal(m, ref_idx[t, :n]) and (ref_idx[t, n:] == -1).all())
    dist.barrier()
    dist.destroy_process_group()
    with open(f"{result_path}.{rank}", "w") as f:
        f.write("ok" if ok else "mismatch")


def test_exchange_on_two_gloo_ranks(tmp_path):
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    path = str(tmp_path / "res")
    mp.start_processes(_rank_main, args=(2, port, path), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert open(f"{path}.{r}").read() == "ok"
