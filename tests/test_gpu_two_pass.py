"""GPU parity of the two-pass tensor-core indexer (tsi_indexer_topk_two_pass: stored scores,
then one block per row) on inputs that drive its row selection off the common path, against
the oracle:

- the keys the row sample reads score low and all others high: the sampled threshold then
  admits far more keys than the row buffer holds, so the row is streamed again through
  the checked selector;
- those keys alone score high: the sampled threshold admits fewer than k keys, so the row
  is streamed again from threshold 0;
- every score equal: the tie rule (lower position first) over rows of 40000 keys;
- sequences of different cached lengths, their rows long enough to be sampled;
- a full-size L = 131072 prefill with integer-valued inputs, checked on the rows at the
  borders of the launch chunks (multiples of 4096 rows from the end) and their neighbours.

Integer-valued e4m3 / bf16 inputs with power-of-two gate weights keep every score exact
in fp32, so indices and scores must match the oracle exactly."""
import numpy as np
import pytest
import torch

from parity import check_indexer
from workloads.gen import draw

pytestmark = pytest.mark.gpu

H, D = 64, 128
TORCH = {"e4m3": torch.float8_e4m3fn, "bf16": torch.bfloat16}


def _check(cuda_lib, qI, kI, w, topk, rows=None):
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, topk, want_score=True, two_pass=True)
    cuda_lib.device_status()
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), topk, idx.cpu(), sc.cpu(), rows=rows, exact=True)
    return idx.cpu(), sc.cpu()


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_all_scores_equal_overflows_the_sampled_threshold(cuda_lib, qk):
    # rows of ~40000 keys: all ties, so the top k are the lowest positions in order
    B, T, S, topk = 1, 9, 40000, 2048
    qI = torch.ones((B, T, H, D), dtype=TORCH[qk], device="cuda")
    kI = torch.ones((B, S, D), dtype=TORCH[qk], device="cuda")
    w = torch.full((B, T, H), 0.25, dtype=torch.bfloat16, device="cuda")
    idx, sc = _check(cuda_lib, qI, kI, w, topk)
    assert torch.equal(idx[0], torch.arange(topk, dtype=torch.int32).expand(T, topk))
    assert torch.all(sc == 64 * 128 * 0.25)


def _sample_contrast(qk, T, S, sampled_value, other_value, seed):
    """Positive integer queries and gate weights; key s is all `sampled_value` when the row
    sample reads it (the first four keys of every 128, rows of <= 163840 keys), else all
    `other_value`."""
    qf = draw((1, T, H, D), "int8", "f32", seed, "cuda").abs()
    qI = torch.where(qf == 0, torch.ones_like(qf), qf).to(TORCH[qk])
    pos = torch.arange(S, device="cuda")
    kval = torch.where((pos % 128) < 4, sampled_value, other_value).to(torch.float32)
    kI = kval.view(1, S, 1).expand(1, S, D).contiguous().to(TORCH[qk])
    w = draw((1, T, H), "pow2", "bf16", seed + 1, "cuda")
    return qI, kI, w


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_sampled_keys_low_overflow_the_row_buffer(cuda_lib, qk):
    T, S, topk = 5, 60000, 2048
    qI, kI, w = _sample_contrast(qk, T, S, 1.0, 4.0, 17)
    idx, _ = _check(cuda_lib, qI, kI, w, topk)
    # the k lowest positions that the sample does not read
    pos = torch.arange(S)
    expect = pos[(pos % 128) >= 4][:topk].to(torch.int32)
    assert torch.equal(idx[0], expect.expand(T, topk))


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_sampled_keys_alone_score_high(cuda_lib, qk):
    T, S, topk = 5, 60000, 2048
    qI, kI, w = _sample_contrast(qk, T, S, 4.0, 1.0, 7)
    idx, _ = _check(cuda_lib, qI, kI, w, topk)
    # every row holds fewer than k high keys: all of them rank first
    for t in range(T):
        p = S - T + t
        n_high = 4 * (p // 128) + min(4, p % 128 + 1)
        assert n_high < topk
        row = idx[0, t]
        assert torch.all((row[:n_high] % 128) < 4) and torch.all((row[n_high:] % 128) >= 4)


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_ragged_sequences_sampled_rows(cuda_lib, qk):
    # per-sequence cache lengths: sampled rows of 12k to 30k keys end where each sequence
    # ends, and a third sequence is shorter than the row buffer
    B, T, S, topk = 3, 64, 30000, 2048
    qI = draw((B, T, H, D), "int8", qk, 31, "cuda", D)
    kI = draw((B, S, D), "int8", qk, 32, "cuda", D)
    w = draw((B, T, H), "pow2", "bf16", 33, "cuda", D)
    kv = torch.tensor([30000, 12345, 4000], dtype=torch.int32, device="cuda")
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv, want_score=True, two_pass=True)
    cuda_lib.device_status()
    rows = sorted({0, T - 1, T, 2 * T - 1, 2 * T, 3 * T - 1} | set(range(5, B * T, 23)))
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), topk, idx.cpu(), sc.cpu(), kv_len=kv.cpu(),
                  rows=np.array(rows), exact=True)


def test_full_size_chunk_borders_integer_exact(cuda_lib):
    # L = 131072 prefill through every launch chunk; rows at multiples of 4096 from the end
    # (the chunk borders of any power-of-two scratch budget) and their neighbours
    T = S = 131072
    topk = 2048
    qI = draw((1, T, H, D), "int8", "e4m3", 901, "cuda", D)
    kI = draw((1, S, D), "int8", "e4m3", 902, "cuda", D)
    w = draw((1, T, H), "pow2", "bf16", 903, "cuda", D)
    borders = [T - 4096 * c for c in (1, 2, 4, 8, 16, 31)]
    rows = sorted({r + d for r in borders for d in (-1, 0)} | {0, 3, T - 1})
    _check(cuda_lib, qI, kI, w, topk, rows=np.array(rows))
