"""tsi_indexer_topk_noalloc against tsi_indexer_topk, through the C ABI.

Some callers cannot allocate device memory while they run: a serving loop whose
device memory is fixed at start-up, or code running inside a custom device
allocator, where a nested cudaMalloc would recurse or synchronize the device.
For them the library keeps the decode scratch (per-split candidate lists) in a
fixed array built into the library instead of a caller workspace.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.  It passes on its own in a fresh
process as well as after the other tests (the array keeps earlier calls'
contents, which must not matter).
"""
import ctypes

import pytest
import torch

import top_selection_indexer_gb300 as tsi
from workloads.gen import draw

pytestmark = pytest.mark.gpu

DT = {torch.float32: tsi.F32, torch.bfloat16: tsi.BF16, torch.float8_e4m3fn: tsi.E4M3}


def _inputs(B, S, H_I, d_I, qk, wdt, qdist, wdist, seed):
    dev = "cuda"
    qI = draw((B, 1, H_I, d_I), qdist, qk, seed, dev, d_I)
    kI = draw((B, S, d_I), qdist, qk, seed + 1, dev, d_I)
    w = draw((B, 1, H_I), wdist, wdt, seed + 2, dev, d_I)
    return qI, kI, w


def _call_noalloc(lib, qI, kI, w, topk, kv_len):
    B, T, H_I, d_I = qI.shape
    S = kI.shape[1]
    idx = torch.full((B, T, topk), -7, dtype=torch.int32, device="cuda")
    score = torch.full((B, T, topk), float("nan"), dtype=torch.float32, device="cuda")
    st = lib.tsi_indexer_topk_noalloc(
        qI.data_ptr(), kI.data_ptr(), w.data_ptr(), DT[qI.dtype], DT[w.dtype], B, T, S, H_I,
        d_I, topk, kv_len.data_ptr(), idx.data_ptr(), score.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == tsi.OK, lib.tsi_last_error()
    return idx, score


# Decode-shaped requests (few rows, long caches): the key range is split across
# blocks, so the built-in scratch is used.  Integer-valued inputs make every partial
# sum exact, so both entry points must agree bit for bit.
CASES = [
    # (B, S, H_I, d_I, qk, w, q dist, w dist, topk, kv_len of call 1, kv_len of call 2)
    (8, 60000, 64, 128, "e4m3", "bf16", "int8", "pow2", 2048,
     [60000, 59999, 30000, 2049, 2048, 100, 1, 0], [40000, 60000, 12345, 8193, 4097, 2, 3000, 777]),
    (4, 50000, 4, 32, "f32", "f32", "int4", "int03", 512,
     [50000, 1, 25000, 9000], [123, 49999, 50000, 4096]),
]


@pytest.mark.parametrize("case", CASES, ids=["e4m3-64x128", "f32-4x32"])
def test_noalloc_matches_regular_entry_point_on_two_calls(cuda_lib, case):
    B, S, H_I, d_I, qk, wdt, qdist, wdist, topk, kv1, kv2 = case
    lib = cuda_lib.load()
    # scratch of the CUDA-core split path (the F32 query selects that path's plan)
    need = lib.tsi_indexer_topk_workspace(B, 1, S, H_I, d_I, topk, tsi.F32)
    assert 0 < need <= lib.tsi_indexer_topk_noalloc_limit()
    calls = []
    for seed, kv in ((11, kv1), (23, kv2)):
        qI, kI, w = _inputs(B, S, H_I, d_I, qk, wdt, qdist, wdist, seed)
        kv_len = torch.tensor(kv, dtype=torch.int32, device="cuda")
        ref_idx, ref_score = cuda_lib.indexer_topk(qI, kI, w, topk, kv_len=kv_len, want_score=True)
        calls.append((qI, kI, w, kv_len, ref_idx, ref_score))
    torch.cuda.synchronize()
    # two no-alloc calls in a row, sharing the built-in scratch
    outs = [_call_noalloc(lib, qI, kI, w, topk, kv_len) for qI, kI, w, kv_len, _, _ in calls]
    cuda_lib.device_status()
    for (_, _, _, _, ref_idx, ref_score), (idx, score) in zip(calls, outs):
        assert torch.equal(idx, ref_idx)
        assert torch.equal(score.view(torch.int32), ref_score.view(torch.int32))


def test_noalloc_rejects_requests_beyond_the_array(cuda_lib):
    lib = cuda_lib.load()
    B, S, topk = 64, 131072, 2048
    need = lib.tsi_indexer_topk_workspace(B, 1, S, 4, 32, topk, tsi.F32)
    assert need > lib.tsi_indexer_topk_noalloc_limit()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    st = lib.tsi_indexer_topk_noalloc(fake, fake, fake, tsi.F32, tsi.F32, B, 1, S, 4, 32, topk,
                                      None, fake, None, None)
    assert st == tsi.ERR_UNSUPPORTED
    assert "scratch" in lib.tsi_last_error().decode()
