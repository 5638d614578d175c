"""GPU parity of tsi_indexer_topk (the scores stay in the scoring kernel, which selects each
row's top k in its epilogue from a sampled threshold), its alias tsi_indexer_topk_onchip and
tsi_indexer_topk_two_pass (scores stored, then selected by a second kernel), against each
other and the oracle.  All compute every score the same way and select exactly, so their
indices and scores must agree bit for bit; integer-valued inputs make them exact against
the oracle."""
import numpy as np
import pytest
import torch

from parity import check_indexer
from workloads.gen import draw

pytestmark = pytest.mark.gpu


def _inputs(B, T, S, H_I, d_I, qk, seed):
    wdt, qd, wd = ("f32", "int4", "int03") if qk == "f32" else ("bf16", "int8", "pow2")
    qI = draw((B, T, H_I, d_I), qd, qk, seed, "cuda", d_I)
    kI = draw((B, S, d_I), qd, qk, seed + 1, "cuda", d_I)
    w = draw((B, T, H_I), wd, wdt, seed + 2, "cuda", d_I)
    return qI, kI, w


CASES = [
    # B, T, S, H_I, d_I, qk, topk, kv_len
    (1, 300, 300, 64, 128, "e4m3", 64, None),            # ragged tiles, short rows
    (2, 150, 3000, 64, 128, "bf16", 2048, [3000, 2100]),  # two-row bf16 units, ragged caches
    (1, 4100, 4100, 64, 128, "e4m3", 2048, None),         # rows past k
    (1, 64, 40000, 64, 128, "e4m3", 2048, None),          # long rows (split key ranges)
    (8, 1, 20000, 64, 128, "e4m3", 2048, None),           # one query per sequence
    (1, 700, 700, 4, 32, "f32", 256, None),               # CUDA-core shape
]


@pytest.mark.parametrize("B,T,S,H_I,d_I,qk,topk,kv", CASES)
def test_default_onchip_and_two_pass_agree_with_the_oracle(cuda_lib, B, T, S, H_I, d_I, qk,
                                                           topk, kv):
    qI, kI, w = _inputs(B, T, S, H_I, d_I, qk, 8100 + S + T)
    kv_t = None if kv is None else torch.tensor(kv, dtype=torch.int32, device="cuda")
    a, sa = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv_t, want_score=True)
    b, sb = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv_t, want_score=True, two_pass=True)
    c, sc = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv_t, want_score=True, onchip=True)
    cuda_lib.device_status()
    assert torch.equal(a, b) and torch.equal(a, c)
    assert torch.equal(sa.view(torch.int32), sb.view(torch.int32))
    assert torch.equal(sa.view(torch.int32), sc.view(torch.int32))
    rows = sorted({0, B * T - 1} | set(range(0, B * T, max(1, B * T // 9))))
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), topk, a.cpu(), sa.cpu(),
                  kv_len=None if kv is None else torch.tensor(kv), rows=np.array(rows),
                  exact=True)
