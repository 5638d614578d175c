"""GPU parity of the context-parallel indexer: tsi_indexer_topk_shard on every key shard,
then tsi_topk_merge of the lists, equals tsi_indexer_topk over the whole cache bit for bit
(every key's fp32 score is computed the same way in both), and the oracle on integer
inputs.  The shards run one after another on one GPU, standing in for ranks."""
import numpy as np
import pytest
import torch

import oracle
from workloads.gen import draw

pytestmark = pytest.mark.gpu


def _inputs(B, T, S, H_I, d_I, qk, wdt, qdist, wdist, seed):
    dev = "cuda"
    qI = draw((B, T, H_I, d_I), qdist, qk, seed, dev, d_I)
    kI = draw((B, S, d_I), qdist, qk, seed + 1, dev, d_I)
    w = draw((B, T, H_I), wdist, wdt, seed + 2, dev, d_I)
    return qI, kI, w


def _sharded(cuda_lib, qI, kI, w, topk, cuts, kv_len=None):
    B, S = kI.shape[0], kI.shape[1]
    edges = [0] + list(cuts) + [S]
    cands, cnts = [], []
    for lo, hi in zip(edges[:-1], edges[1:]):
        c, n = cuda_lib.indexer_topk_shard(qI, kI[:, lo:hi].contiguous(), w, topk, S, lo,
                                           kv_len=kv_len)
        cands.append(c)
        cnts.append(n)
    cuda_lib.device_status()
    return cuda_lib.topk_merge(torch.stack(cands), torch.stack(cnts), want_score=True)


CASES = [
    # B, T, S, H_I, d_I, qk, cuts, kv_len
    (1, 3000, 3000, 64, 128, "e4m3", (1000, 1129, 2500), None),
    (1, 3000, 3000, 64, 128, "bf16", (1500,), None),
    (2, 300, 1000, 64, 128, "e4m3", (333, 700), [1000, 900]),
    (4, 1, 40000, 64, 128, "e4m3", (12345, 30000), [40000, 20000, 7, 31000]),
    # shards of up to 15000 keys per query row: the two-pass row selection samples them
    (2, 64, 40000, 64, 128, "e4m3", (15000, 26000), [40000, 23456]),
    (1, 700, 700, 4, 32, "f32", (100, 101, 650), None),
    (3, 1, 30000, 4, 32, "f32", (9000,), [30000, 8999, 9001]),
]


@pytest.mark.parametrize("B,T,S,H_I,d_I,qk,cuts,kv", CASES)
def test_shards_merge_to_the_whole_cache(cuda_lib, B, T, S, H_I, d_I, qk, cuts, kv):
    wdt = "f32" if qk == "f32" else "bf16"
    qd, wd = ("int4", "int03") if qk == "f32" else ("int8", "pow2")
    qI, kI, w = _inputs(B, T, S, H_I, d_I, qk, wdt, qd, wd, 7000 + S + T)
    kv_t = None if kv is None else torch.tensor(kv, dtype=torch.int32, device="cuda")
    topk = 2048 if d_I == 128 else 256
    idx_m, sc_m = _sharded(cuda_lib, qI, kI, w, topk, cuts, kv_t)
    idx_w, sc_w = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv_t, want_score=True)
    cuda_lib.device_status()
    assert torch.equal(idx_m.view(-1, topk), idx_w.view(-1, topk))
    assert torch.equal(sc_m.view(-1, topk).view(torch.int32), sc_w.view(-1, topk).view(torch.int32))
    # the oracle on sampled rows (integer inputs: exact)
    rows = sorted({0, B * T - 1} | set(range(0, B * T, max(1, B * T // 7))))
    ref_idx, _ = oracle.indexer_topk(qI.cpu(), kI.cpu(), w.cpu(), topk, rows=rows,
                                     kv_len=None if kv is None else torch.tensor(kv))
    assert np.array_equal(idx_m.view(-1, topk).cpu().numpy()[rows], np.asarray(ref_idx))


def test_merge_of_one_list_ranks_it(cuda_lib):
    qI, kI, w = _inputs(1, 500, 500, 64, 128, "e4m3", "bf16", "int8", "pow2", 77)
    c, n = cuda_lib.indexer_topk_shard(qI, kI, w, 64, 500, 0)
    idx = cuda_lib.topk_merge(c[None], n[None])
    ref = cuda_lib.indexer_topk(qI, kI, w, 64)
    cuda_lib.device_status()
    assert torch.equal(idx, ref.view(-1, 64))


def test_signed_gates_shards_merge_to_the_whole_cache(cuda_lib):
    # gate weights of both signs (powers of two): negative scores through the shards' capped
    # passes, whose raw (score, position) pairs become rank keys before each unit's exact
    # selection; rows of up to 7000 keys per shard take sampled thresholds
    B, T, S, topk = 1, 2000, 12000, 2048
    qI = draw((B, T, 64, 128), "int8", "e4m3", 7101, "cuda", 128)
    kI = draw((B, S, 128), "int8", "e4m3", 7102, "cuda", 128)
    g = torch.Generator(device="cuda")
    g.manual_seed(7103)
    sign = torch.randint(0, 2, (B, T, 64), generator=g, device="cuda").to(torch.float32) * 2 - 1
    w = (draw((B, T, 64), "pow2", "f32", 7104, "cuda") * sign).to(torch.bfloat16)
    idx_m, sc_m = _sharded(cuda_lib, qI, kI, w, topk, (5000,))
    idx_w, sc_w = cuda_lib.indexer_topk(qI, kI, w, topk, want_score=True)
    cuda_lib.device_status()
    assert torch.equal(idx_m.view(-1, topk), idx_w.view(-1, topk))
    assert torch.equal(sc_m.view(-1, topk).view(torch.int32), sc_w.view(-1, topk).view(torch.int32))
    rows = [0, 1, 777, 1500, T - 2, T - 1]
    ref_idx, _ = oracle.indexer_topk(qI.cpu(), kI.cpu(), w.cpu(), topk, rows=rows)
    assert np.array_equal(idx_m.view(-1, topk).cpu().numpy()[rows], np.asarray(ref_idx))
