"""GPU parity of tsi_indexer_topk against the CPU oracle: small and ragged shapes,
decode, prefill chunks, determinism (through the C ABI)."""
import numpy as np
import pytest
import torch

from parity import check_indexer
from workloads.gen import draw

pytestmark = pytest.mark.gpu


def _inputs(B, T, S, H_I, d_I, qk, wdt, qdist, wdist, seed):
    dev = "cuda"
    qI = draw((B, T, H_I, d_I), qdist, qk, seed, dev, d_I)
    kI = draw((B, S, d_I), qdist, qk, seed + 1, dev, d_I)
    w = draw((B, T, H_I), wdist, wdt, seed + 2, dev, d_I)
    return qI, kI, w


def _run_and_check(cuda_lib, B, T, S, H_I, d_I, topk, qk, wdt, qdist, wdist, seed, exact,
                   kv_len=None, rows=None):
    qI, kI, w = _inputs(B, T, S, H_I, d_I, qk, wdt, qdist, wdist, seed)
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device="cuda")
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv, want_score=True)
    cuda_lib.device_status()
    return check_indexer(qI.cpu(), kI.cpu(), w.cpu(), topk, idx.cpu(), sc.cpu(),
                         kv_len=None if kv_len is None else torch.tensor(kv_len), rows=rows,
                         exact=exact)


# Generic (CUDA-core) shapes: integer-valued, so indices and scores are exact.
@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 300])
@pytest.mark.parametrize("topk", [1, 7, 64])
@pytest.mark.parametrize("H_I", [1, 4])
def test_generic_small_integer_exact(cuda_lib, L, topk, H_I):
    _run_and_check(cuda_lib, 1, L, L, H_I, 32, topk, "f32", "f32", "int4", "int03",
                   1000 + L * 10 + topk + H_I, exact=True)


# Tensor-core shapes (H_I = 64, d_I = 128) with ragged key-tile tails.
@pytest.mark.parametrize("qk", ["bf16", "e4m3"])
@pytest.mark.parametrize("L,topk", [(1, 1), (127, 7), (128, 64), (129, 64), (300, 64),
                                    (2047, 2048), (2049, 2048), (4100, 2048), (5000, 100)])
def test_tc_shape_integer_exact(cuda_lib, qk, L, topk):
    _run_and_check(cuda_lib, 1, L, L, 64, 128, topk, qk, "bf16", "int8", "pow2",
                   2000 + L + topk, exact=True)


def test_batch_of_sequences_integer_exact(cuda_lib):
    _run_and_check(cuda_lib, 3, 700, 700, 64, 128, 128, "e4m3", "bf16", "int8", "pow2", 31,
                   exact=True)


def test_prefill_chunk_positions(cuda_lib):
    # T = 300 new rows at the end of a 1000-key cache: row t sits at position 700 + t.
    _run_and_check(cuda_lib, 2, 300, 1000, 64, 128, 256, "bf16", "bf16", "int8", "pow2", 41,
                   exact=True, kv_len=[1000, 900])


@pytest.mark.parametrize("T", [301, 3])
def test_prefill_chunk_positions_e4m3(cuda_lib, T):
    # four query rows per tensor-core unit: T not a multiple of 4 leaves a partial first
    # unit; rows sit at kv_len - T + t (T = 3: a multi-query decode step)
    _run_and_check(cuda_lib, 2, T, 1000, 64, 128, 256, "e4m3", "bf16", "int8", "pow2", 43 + T,
                   exact=True, kv_len=[1000, 905])


def test_decode_ragged_kv_len_integer_exact(cuda_lib):
    # one query per sequence at position kv_len-1; empty, tiny and long caches
    _run_and_check(cuda_lib, 6, 1, 40000, 64, 128, 2048, "e4m3", "bf16", "int8", "pow2", 51,
                   exact=True, kv_len=[0, 1, 5, 2048, 2049, 40000])


@pytest.mark.parametrize("B,kv", [(1, None), (2, [131072, 70001]), (8, None)])
def test_decode_two_stage_merge_integer_exact(cuda_lib, B, kv):
    # a long cache split into many key chunks (64 for one row, 19 per row for eight): the
    # chunk lists are merged in groups of about sqrt(n) lists, then per row
    _run_and_check(cuda_lib, B, 1, 131072, 64, 128, 2048, "e4m3", "bf16", "int8", "pow2",
                   71 + B, exact=True, kv_len=kv)


def test_decode_bf16_integer_exact(cuda_lib):
    # one query per sequence with bf16 operands (the one-row tensor-core units of the bf16
    # format); integers in [-8, 8] are exact in bf16, so the rows match the oracle exactly
    _run_and_check(cuda_lib, 3, 1, 20000, 64, 128, 2048, "bf16", "bf16", "int8", "pow2", 81,
                   exact=True, kv_len=[20000, 7001, 3])


def test_decode_generic_heads_split_merge(cuda_lib):
    # few rows + long cache: keys split over blocks and merged (CUDA-core path)
    _run_and_check(cuda_lib, 4, 1, 30000, 4, 32, 512, "f32", "f32", "int4", "int03", 61,
                   exact=True, kv_len=[30000, 12345, 1, 8193])


@pytest.mark.parametrize("qk,dist", [("bf16", "normal_dI"), ("e4m3", "normal")])
def test_continuous_inputs_near_tie_rule(cuda_lib, qk, dist):
    rec = _run_and_check(cuda_lib, 1, 3000, 3000, 64, 128, 512, qk, "bf16", dist, "uniform",
                         71, exact=False, rows=list(range(0, 3000, 97)) + [2999])
    assert rec > 0.99


def test_repeat_calls_are_bitwise_identical(cuda_lib):
    qI, kI, w = _inputs(1, 5000, 5000, 64, 128, "bf16", "bf16", "normal_dI", "uniform", 81)
    a, sa = cuda_lib.indexer_topk(qI, kI, w, 2048, want_score=True)
    b, sb = cuda_lib.indexer_topk(qI, kI, w, 2048, want_score=True)
    assert torch.equal(a, b) and torch.equal(sa.view(torch.int32), sb.view(torch.int32))


def test_no_keys_gives_padding(cuda_lib):
    qI, kI, w = _inputs(2, 3, 10, 4, 32, "f32", "f32", "int4", "int03", 91)
    kv = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, 5, kv_len=kv, want_score=True)
    idx = idx.cpu()
    assert torch.all(idx[0] == -1)
    # sequence 1 holds 2 keys; rows sit at positions -1, 0, 1
    assert torch.all(idx[1, 0] == -1)
    assert idx[1, 1, 0] == 0 and torch.all(idx[1, 1, 1:] == -1)
    assert sorted(idx[1, 2, :2].tolist()) == [0, 1] and torch.all(idx[1, 2, 2:] == -1)
    assert torch.all(torch.isneginf(sc.cpu()[0]))
