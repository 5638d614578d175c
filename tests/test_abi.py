"""The C ABI: the library loads, exports every declared symbol, and rejects bad
arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

import top_selection_indexer_gb300 as tsi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsi.h")

FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsi_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from top_selection_indexer_gb300 import _build

    _build.build()
    return tsi.load()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("tsi_indexer_topk", "tsi_sparse_attn_group", "tsi_indexer_topk_workspace",
              "tsi_sparse_attn_workspace", "tsi_last_error", "tsi_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(tsi.EXPORTS)
    assert lib.tsi_version() >= 100


def _idx(lib, **kw):
    a = dict(qI=FAKE, kI=FAKE, w=FAKE, qk=tsi.E4M3, wdt=tsi.BF16, B=1, T=8, S=8, H_I=64,
             d_I=128, topk=4, kv=None, idx=FAKE, score=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.tsi_indexer_topk(a["qI"], a["kI"], a["w"], a["qk"], a["wdt"], a["B"], a["T"],
                                a["S"], a["H_I"], a["d_I"], a["topk"], a["kv"], a["idx"],
                                a["score"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(topk=0), tsi.ERR_UNSUPPORTED),
    (dict(topk=2049), tsi.ERR_UNSUPPORTED),
    (dict(B=-1), tsi.ERR_INVALID_ARG),
    (dict(qk=7), tsi.ERR_INVALID_ARG),
    (dict(wdt=tsi.E4M3), tsi.ERR_INVALID_ARG),
    (dict(H_I=0), tsi.ERR_INVALID_ARG),
    (dict(H_I=100, d_I=200), tsi.ERR_UNSUPPORTED),
    (dict(idx=None), tsi.ERR_INVALID_ARG),
    (dict(qI=FAKE + 4), tsi.ERR_INVALID_ARG),
    (dict(B=8, T=1, S=131072, topk=2048, ws=None, wsb=0), tsi.ERR_WORKSPACE),
])
def test_indexer_rejects_bad_arguments(lib, kw, status):
    st = _idx(lib, **kw)
    assert st == status, lib.tsi_last_error()
    assert lib.tsi_last_error()


def test_indexer_empty_batch_is_a_noop(lib):
    assert _idx(lib, B=0, qI=None, kI=None, w=None, idx=None) == tsi.OK
    assert _idx(lib, T=0, qI=None, kI=None, w=None, idx=None) == tsi.OK


def test_decode_needs_workspace(lib):
    need = lib.tsi_indexer_topk_workspace(8, 1, 131072, 64, 128, 2048, tsi.E4M3)
    assert need > 0
    st = _idx(lib, B=8, T=1, S=131072, topk=2048, ws=FAKE, wsb=need - 1)
    assert st == tsi.ERR_WORKSPACE


def _scores_bytes(B, T, S, R, budget=8 << 30):
    """Stored scores of the two-pass tensor-core indexer: one chunk of query rows, rows of
    S floats rounded up to 4, the chunk as many rows (a multiple of R) as fit the budget."""
    ld = (S + 3) // 4 * 4
    rows = budget // (B * ld * 4) // R * R
    rows = min(T, max(R, rows))
    return B * rows * ld * 4


def _align(x, a):
    return (x + a - 1) // a * a


def _lists_bytes(slots, topk=2048):
    """One candidate list of topk 8-byte keys per slot, then a count per slot."""
    return _align(slots * topk * 8, 16) + _align(slots * 4, 256)


def _sampled_bytes(B, T, S, qk, R):
    """Scratch of the sampled-threshold selection beside the lists: a threshold per row, the
    short-unit count and list (one entry per unit of R rows), every 32nd key row."""
    off = _align(B * T * 4, 256) + 256
    off = _align(off + B * -(-T // R) * 4, 1024)
    return off + _align(B * -(-S // 32) * (256 if qk == tsi.BF16 else 128), 1024)


@pytest.mark.parametrize("B,T,S,qk,R", [
    (1, 300, 1000, tsi.E4M3, 4),        # all rows in one chunk
    (3, 5, 10, tsi.E4M3, 4),            # rows padded to 12 floats
    (1, 131072, 131072, tsi.E4M3, 4),   # 16384-row chunks: 8 GiB
    (1, 131072, 131071, tsi.BF16, 2),   # padded row, bf16 units of two rows
    (64, 4096, 131072, tsi.E4M3, 4),    # 256-row chunks across 64 sequences
])
def test_two_pass_workspace_holds_one_chunk_of_scores(lib, B, T, S, qk, R):
    need = lib.tsi_indexer_topk_two_pass_workspace(B, T, S, 64, 128, 2048, qk)
    assert need == _scores_bytes(B, T, S, R)
    # key shards select on chip: the caller's lists take the candidates, the workspace
    # holds the sampled selection's scratch only
    assert lib.tsi_indexer_topk_shard_workspace(B, T, S, 64, 128, 2048, qk) == \
        _sampled_bytes(B, T, S, qk, R)


@pytest.mark.parametrize("B,T,S,qk,R", [(1, 131072, 131072, tsi.E4M3, 4),
                                        (2, 3000, 3000, tsi.BF16, 2)])
def test_default_workspace_holds_candidate_lists_and_the_sample(lib, B, T, S, qk, R):
    # the default stores no score: one list per row of every key its selector held (8 B a
    # key, the selector's capacity: 4352 keys for e4m3, 5888 for bf16; these shapes have
    # enough rows to keep each row's keys in one range), a count per row, and the sampled
    # selection's scratch; the on-chip name is the same call
    need = lib.tsi_indexer_topk_workspace(B, T, S, 64, 128, 2048, qk)
    cap = 5888 if qk == tsi.BF16 else 4352
    assert need == _lists_bytes(B * T, cap) + _sampled_bytes(B, T, S, qk, R)
    assert lib.tsi_indexer_topk_onchip_workspace(B, T, S, 64, 128, 2048, qk) == need
    assert need < lib.tsi_indexer_topk_two_pass_workspace(B, T, S, 64, 128, 2048, qk) or \
        T * S < 1 << 24


def test_bf16_decode_takes_the_cuda_core_path(lib):
    # bf16 with one query per sequence: the CUDA-core path's workspace (as for fp32 inputs)
    for S in (4000, 131072):
        assert lib.tsi_indexer_topk_workspace(8, 1, S, 64, 128, 2048, tsi.BF16) == \
            lib.tsi_indexer_topk_workspace(8, 1, S, 64, 128, 2048, tsi.F32)
    # several queries per sequence stay on the tensor cores
    assert lib.tsi_indexer_topk_workspace(1, 4096, 4096, 64, 128, 2048, tsi.BF16) != \
        lib.tsi_indexer_topk_workspace(1, 4096, 4096, 64, 128, 2048, tsi.F32)


def test_decode_workspace_holds_candidate_lists(lib):
    # one query per sequence: key-range candidate lists (8 B a key) and counts, no scores
    need = lib.tsi_indexer_topk_workspace(8, 1, 131072, 64, 128, 2048, tsi.E4M3)
    assert need >= 8 * 2048 * 8 * 2  # at least two key ranges per row
    assert need < 8 * 131072 * 4     # far below one row of stored scores per sequence


def _attn(lib, n=1, **kw):
    P = ctypes.c_void_p * n
    a = dict(q=P(*[FAKE] * n), k=P(*[FAKE] * n), v=None, B=1, T=4, S=4, H=64, Hkv=1,
             Dqk=576, Dv=512, scale=1 / 24, idx=FAKE, topk=4, kv=None, out=P(*[FAKE] * n),
             ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.tsi_sparse_attn_group(n, a["q"], a["k"], a["v"], a["B"], a["T"], a["S"], a["H"],
                                     a["Hkv"], a["Dqk"], a["Dv"], a["scale"], a["idx"],
                                     a["topk"], a["kv"], a["out"], a["ws"], a["wsb"],
                                     a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(topk=0), tsi.ERR_UNSUPPORTED),
    (dict(topk=4096), tsi.ERR_UNSUPPORTED),
    (dict(H=6, Hkv=4), tsi.ERR_INVALID_ARG),
    (dict(Dqk=1024), tsi.ERR_UNSUPPORTED),
    (dict(Dqk=256, Dv=512), tsi.ERR_UNSUPPORTED),  # value from key needs Dv <= Dqk
    (dict(scale=float("inf")), tsi.ERR_INVALID_ARG),
    (dict(idx=None), tsi.ERR_INVALID_ARG),
    (dict(idx=FAKE + 8), tsi.ERR_INVALID_ARG),
    (dict(B=-2), tsi.ERR_INVALID_ARG),
])
def test_attn_rejects_bad_arguments(lib, kw, status):
    st = _attn(lib, **kw)
    assert st == status, lib.tsi_last_error()


def test_attn_null_layer_pointer(lib):
    P = ctypes.c_void_p * 2
    assert _attn(lib, n=2, q=P(FAKE, None)) == tsi.ERR_INVALID_ARG


def test_attn_zero_layers_is_a_noop(lib):
    assert _attn(lib, n=1, B=0) == tsi.OK
