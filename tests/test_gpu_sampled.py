"""GPU parity of the default tensor-core indexer (tsi_indexer_topk) on inputs that defeat
its sampled admission threshold, against the oracle.

With several query rows per sequence the call first scores every 32nd key of each row and
admits, in the full scoring pass, only keys at or above the row's 100th largest sampled
score (for k = 2048).  These inputs make that sample lie:

- the sampled keys score low and all others high: the threshold admits every key, each
  row's selector fills and compacts again and again;
- the sampled keys alone score high: fewer than k keys reach the threshold, so every unit
  is listed and done again from no threshold by the third launch;
- half the rows of each four-row unit see the second pattern and half score every key 0
  (all ties): units that are redone hold rows that were complete;
- every score equal (zero gate weights);
- gate weights of both signs, so that many scores (and some thresholds) are negative.

In the first three, queries and gates are positive integers and a key row holds one
integer value; the signed gates are powers of two over integer queries and keys.  Every
score is exact in fp32 and the oracle's rows must be matched bit for bit.  The same kinds of
input then go through the one-query-per-sequence (decode) path in e4m3, which has no sampled
threshold: key chunks selected in the scoring kernel, merged per row.  A full-size
L = 131072 integer-valued prefill checks sampled rows of the common path.  (Score equation
and k: "GLM-5.2 技术报告速览", §IndexShare; the lower-index tie rule: the reading taken here
of the deterministic top-k of "GLM-5: from Vibe Coding to Agentic Engineering" (Chinese
translation), §3.2.)
"""
import numpy as np
import pytest
import torch

from parity import check_indexer
from workloads.gen import draw

pytestmark = pytest.mark.gpu

H, D = 64, 128
TORCH = {"e4m3": torch.float8_e4m3fn, "bf16": torch.bfloat16}
# enough four-row (e4m3) or two-row (bf16) units to fill the GPU, so each row's keys stay
# in one range and the sampled selection applies; rows are the last T of an S-key cache
T, S, TOPK = 640, 60000, 2048


def _check(cuda_lib, qI, kI, w, rows):
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, TOPK, want_score=True)
    cuda_lib.device_status()
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), TOPK, idx.cpu(), sc.cpu(), rows=np.array(rows),
                  exact=True)
    return idx.cpu()


def _rows():
    return sorted({0, 1, 2, 3, 4, 5, 6, 7, 321, 322, T - 2, T - 1})


def _contrast(qk, sampled_value, other_value, seed, negative_rows=()):
    """Positive integer queries (negated on `negative_rows`) and power-of-two gates; key s
    is all `sampled_value` when the sample reads it (s % 32 == 0), else all `other_value`."""
    qf = draw((1, T, H, D), "int8", "f32", seed, "cuda").abs()
    qf = torch.where(qf == 0, torch.ones_like(qf), qf)
    if len(negative_rows):
        sign = torch.ones(T, device="cuda")
        sign[torch.as_tensor(list(negative_rows), device="cuda")] = -1.0
        qf = qf * sign.view(1, T, 1, 1)
    pos = torch.arange(S, device="cuda")
    kval = torch.where(pos % 32 == 0, sampled_value, other_value).to(torch.float32)
    kI = kval.view(1, S, 1).expand(1, S, D).contiguous().to(TORCH[qk])
    w = draw((1, T, H), "pow2", "bf16", seed + 1, "cuda")
    return qf.to(TORCH[qk]), kI, w


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_sampled_keys_low_admit_every_key(cuda_lib, qk):
    qI, kI, w = _contrast(qk, 1.0, 4.0, 41)
    idx = _check(cuda_lib, qI, kI, w, _rows())
    # every row: the k lowest positions the sample does not read, in order
    pos = torch.arange(S)
    expect = pos[pos % 32 != 0][:TOPK].to(torch.int32)
    assert torch.equal(idx[0], expect.expand(T, TOPK))


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_sampled_keys_alone_high_redo_every_unit(cuda_lib, qk):
    qI, kI, w = _contrast(qk, 4.0, 1.0, 43)
    idx = _check(cuda_lib, qI, kI, w, _rows())
    for t in (0, T // 2, T - 1):
        p = S - T + t
        n_high = p // 32 + 1
        assert n_high < TOPK
        row = idx[0, t]
        assert torch.all(row[:n_high] % 32 == 0) and torch.all(row[n_high:] % 32 != 0)
        assert torch.equal(row[:n_high], torch.arange(0, 32 * n_high, 32, dtype=torch.int32))


def test_units_mixing_redone_and_complete_rows(cuda_lib):
    # rows 4u + 2 and 4u + 3 score every key 0 (a negated query through the ReLU): ties,
    # every key admitted; rows 4u and 4u + 1 come short and send their unit to the third
    # launch, which must reproduce its complete rows exactly
    neg = [t for t in range(T) if t % 4 >= 2]
    qI, kI, w = _contrast("e4m3", 4.0, 1.0, 47, negative_rows=neg)
    idx = _check(cuda_lib, qI, kI, w, _rows())
    ties = torch.arange(TOPK, dtype=torch.int32)
    for t in (2, 3, 322, T - 1):
        assert torch.equal(idx[0, t], ties)


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_all_scores_equal(cuda_lib, qk):
    qI = draw((1, T, H, D), "int8", qk, 51, "cuda", D)
    kI = draw((1, S, D), "int8", qk, 52, "cuda", D)
    w = torch.zeros((1, T, H), dtype=torch.bfloat16, device="cuda")
    idx = _check(cuda_lib, qI, kI, w, _rows())
    assert torch.equal(idx[0], torch.arange(TOPK, dtype=torch.int32).expand(T, TOPK))


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_random_integer_rows(cuda_lib, qk):
    # the common path: thresholds that hold, rows of 59k to 60k keys
    qI = draw((1, T, H, D), "int8", qk, 61, "cuda", D)
    kI = draw((1, S, D), "int8", qk, 62, "cuda", D)
    w = draw((1, T, H), "pow2", "bf16", 63, "cuda", D)
    _check(cuda_lib, qI, kI, w, _rows())


def test_full_size_prefill_integer_exact(cuda_lib):
    # L = 131072 in one call, the benchmark's launch configuration; rows across the range,
    # the longest last
    L = 131072
    qI = draw((1, L, H, D), "int8", "e4m3", 971, "cuda", D)
    kI = draw((1, L, D), "int8", "e4m3", 972, "cuda", D)
    w = draw((1, L, H), "pow2", "bf16", 973, "cuda", D)
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, TOPK, want_score=True)
    cuda_lib.device_status()
    rows = sorted({0, 1, 2047, 2048, 3839, 3840, 3841, 5000, 65535, 65536, 100001, L - 4,
                   L - 3, L - 2, L - 1})
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), TOPK, idx.cpu(), sc.cpu(), rows=np.array(rows),
                  exact=True)


# ---- one query per sequence (decode, e4m3): no sampled threshold; each row's keys are split
# into 19 chunks of 3200 keys that select in the scoring kernel's epilogue (their selectors
# compact when every key is admitted), then the chunk lists are merged in two stages.
def _signed_gates(shape, seed):
    """Powers of two 2^-4 .. 1 with a random sign each: the score equation puts no sign on
    the gate weights, and with signed ones many scores are negative."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    sign = torch.randint(0, 2, shape, generator=g, device="cuda").to(torch.float32) * 2 - 1
    return (draw(shape, "pow2", "f32", seed + 1, "cuda") * sign).to(torch.bfloat16)


@pytest.mark.parametrize("qk", ["e4m3", "bf16"])
def test_signed_gate_weights_integer_exact(cuda_lib, qk):
    # negative scores through the sampled threshold, the raw (score, position) pairs the
    # capped pass appends and their rank keys; every score is a multiple of 2^-4 below 2^20
    # in magnitude, so fp32 holds it exactly in any order of summation
    qI = draw((1, T, H, D), "int8", qk, 181, "cuda", D)
    kI = draw((1, S, D), "int8", qk, 182, "cuda", D)
    w = _signed_gates((1, T, H), 183)
    idx = _check(cuda_lib, qI, kI, w, _rows())
    idx2 = cuda_lib.indexer_topk(qI, kI, w, TOPK, two_pass=True)
    cuda_lib.device_status()
    assert torch.equal(idx, idx2.cpu())


# Adversarial inputs like the ones above, exact against the oracle.  (bf16 requests of one
# query per sequence take the CUDA-core path.)

BD, SD = 8, 60000


def _decode_contrast(qk, sampled_value, other_value, seed, negative_rows=(), kv=None):
    qf = draw((BD, 1, H, D), "int8", "f32", seed, "cuda").abs()
    qf = torch.where(qf == 0, torch.ones_like(qf), qf)
    if len(negative_rows):
        sign = torch.ones(BD, device="cuda")
        sign[torch.as_tensor(list(negative_rows), device="cuda")] = -1.0
        qf = qf * sign.view(BD, 1, 1, 1)
    pos = torch.arange(SD, device="cuda")
    kval = torch.where(pos % 32 == 0, sampled_value, other_value).to(torch.float32)
    kI = kval.view(1, SD, 1).expand(BD, SD, D).contiguous().to(TORCH[qk])
    w = draw((BD, 1, H), "pow2", "bf16", seed + 1, "cuda")
    return qf.to(TORCH[qk]), kI, w


def _check_decode(cuda_lib, qI, kI, w, kv=None):
    kvt = None if kv is None else torch.tensor(kv, dtype=torch.int32, device="cuda")
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, TOPK, kv_len=kvt, want_score=True)
    cuda_lib.device_status()
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), TOPK, idx.cpu(), sc.cpu(), rows=np.arange(BD),
                  exact=True, kv_len=None if kv is None else torch.tensor(kv))
    return idx.cpu()


@pytest.mark.parametrize("qk", ["e4m3"])
def test_decode_sample_low_others_high(cuda_lib, qk):
    # two score values, every other key above the every-32nd ones: full chunk lists, ties
    # inside each score
    qI, kI, w = _decode_contrast(qk, 1.0, 4.0, 141)
    idx = _check_decode(cuda_lib, qI, kI, w)
    pos = torch.arange(SD)
    expect = pos[pos % 32 != 0][:TOPK].to(torch.int32)
    assert torch.equal(idx[:, 0], expect.expand(BD, TOPK))


@pytest.mark.parametrize("qk", ["e4m3"])
def test_decode_sample_high_others_low(cuda_lib, qk):
    # fewer than k keys of the higher score: each row ends in keys of the lower score
    qI, kI, w = _decode_contrast(qk, 4.0, 1.0, 143)
    idx = _check_decode(cuda_lib, qI, kI, w)
    n_high = (SD - 1) // 32 + 1
    assert n_high < TOPK
    row = idx[0, 0]
    assert torch.equal(row[:n_high], torch.arange(0, 32 * n_high, 32, dtype=torch.int32))


def test_decode_rows_mixing_ties_and_short_rows(cuda_lib):
    # rows 1, 4, 6 score every key 0 (ties); ragged caches, one of a single chunk, one tiny
    neg = [1, 4, 6]
    kv = [60000, 41000, 60000, 30001, 2049, 60000, 17, 59999]
    qI, kI, w = _decode_contrast("e4m3", 4.0, 1.0, 147, negative_rows=neg)
    idx = _check_decode(cuda_lib, qI, kI, w, kv=kv)
    assert torch.equal(idx[1, 0], torch.arange(TOPK, dtype=torch.int32))


@pytest.mark.parametrize("qk", ["e4m3"])
def test_decode_all_scores_equal(cuda_lib, qk):
    qI = draw((BD, 1, H, D), "int8", qk, 151, "cuda", D)
    kI = draw((BD, SD, D), "int8", qk, 152, "cuda", D)
    w = torch.zeros((BD, 1, H), dtype=torch.bfloat16, device="cuda")
    idx = _check_decode(cuda_lib, qI, kI, w)
    assert torch.equal(idx[:, 0], torch.arange(TOPK, dtype=torch.int32).expand(BD, TOPK))


@pytest.mark.parametrize("qk", ["e4m3"])
def test_decode_random_integer_rows(cuda_lib, qk):
    # random integer scores over ragged caches
    qI = draw((BD, 1, H, D), "int8", qk, 161, "cuda", D)
    kI = draw((BD, SD, D), "int8", qk, 162, "cuda", D)
    w = draw((BD, 1, H), "pow2", "bf16", 163, "cuda", D)
    _check_decode(cuda_lib, qI, kI, w, kv=[60000, 16384, 16385, 59001, 30000, 1, 2048, 45000])


def test_decode_signed_gate_weights_integer_exact(cuda_lib):
    qI = draw((BD, 1, H, D), "int8", "e4m3", 191, "cuda", D)
    kI = draw((BD, SD, D), "int8", "e4m3", 192, "cuda", D)
    w = _signed_gates((BD, 1, H), 193)
    _check_decode(cuda_lib, qI, kI, w, kv=[60000, 16384, 16385, 59001, 30000, 1, 2048, 45000])


def test_decode_full_size_integer_exact(cuda_lib):
    # the benchmark's decode shape: B = 8 over L = 131072
    L = 131072
    qI = draw((BD, 1, H, D), "int8", "e4m3", 171, "cuda", D)
    kI = draw((BD, L, D), "int8", "e4m3", 172, "cuda", D)
    w = draw((BD, 1, H), "pow2", "bf16", 173, "cuda", D)
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, TOPK, want_score=True)
    cuda_lib.device_status()
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), TOPK, idx.cpu(), sc.cpu(), rows=np.arange(BD),
                  exact=True)
