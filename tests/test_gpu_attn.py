"""GPU parity of tsi_sparse_attn_group against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from parity import check_attn
from workloads.gen import draw

pytestmark = pytest.mark.gpu


def _rand_idx(B, T, S, topk, kv_len, seed, pad_frac=0.0):
    """Random causal index rows in arbitrary order, -1 padded past min(k, p+1)."""
    g = np.random.default_rng(seed)
    idx = -np.ones((B, T, topk), dtype=np.int32)
    for b in range(B):
        n_len = S if kv_len is None else kv_len[b]
        for t in range(T):
            p = n_len - T + t
            n = max(0, min(topk, p + 1))
            if n and pad_frac:
                n = max(1, int(n * (1 - pad_frac)))
            if n > 0:
                idx[b, t, :n] = g.choice(p + 1, size=n, replace=False)
    return torch.from_numpy(idx)


def _run(cuda_lib, B, T, S, H, Hkv, Dqk, Dv, topk, v_from_k, n_layers, seed, kv_len=None,
         pad_frac=0.0, rows=None):
    dev = "cuda"
    qs = [draw((B, T, H, Dqk), "normal", "bf16", seed + 10 * l, dev) for l in range(n_layers)]
    ks = [draw((B, S, Hkv, Dqk), "normal", "bf16", seed + 10 * l + 1, dev)
          for l in range(n_layers)]
    vs = None if v_from_k else [draw((B, S, Hkv, Dv), "normal", "bf16", seed + 10 * l + 2, dev)
                                for l in range(n_layers)]
    idx = _rand_idx(B, T, S, topk, kv_len, seed, pad_frac)
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=dev)
    scale = 1.0 / Dqk ** 0.5
    outs = cuda_lib.sparse_attn_group(qs, ks, vs, idx.to(dev), scale, kv_len=kv, Dv=Dv)
    cuda_lib.device_status()
    if rows is None:
        rows = np.arange(B * T)
    rows = np.asarray(rows)
    assert rows.min() >= 0 and rows.max() < B * T, "sampled rows out of range"
    sel = torch.as_tensor(rows)
    for l in range(n_layers):
        check_attn(qs[l].reshape(B * T, H, Dqk)[sel.to(dev)].cpu(), ks[l].cpu(),
                   None if vs is None else vs[l].cpu(), idx.reshape(B * T, topk)[sel], scale,
                   outs[l].reshape(B * T, H, Dv)[sel.to(dev)].cpu(), rows, T, Dv,
                   kv_len=None if kv_len is None else torch.tensor(kv_len))
    return outs


def test_mha_small_group(cuda_lib):
    _run(cuda_lib, 1, 200, 200, 4, 4, 64, 64, 64, False, 4, 100)


def test_gqa_heads(cuda_lib):
    _run(cuda_lib, 2, 50, 50, 8, 2, 32, 16, 16, False, 2, 200)


@pytest.mark.parametrize("L,topk", [(1, 1), (130, 64), (300, 64), (2100, 2048)])
def test_mqa_latent_prefill(cuda_lib, L, topk):
    rows = np.unique(np.r_[0, min(1, L - 1), np.linspace(0, L - 1, 24).astype(int), L - 1])
    _run(cuda_lib, 1, L, L, 64, 1, 576, 512, topk, True, 1, 300 + L, rows=rows)


def test_mqa_latent_padding_and_empty_rows(cuda_lib):
    _run(cuda_lib, 3, 40, 600, 64, 1, 576, 512, 256, True, 1, 400, kv_len=[600, 30, 0],
         pad_frac=0.3)


def test_mqa_latent_decode_split(cuda_lib):
    # decode: few rows, each over up to 2048 keys (split along the index list + combine)
    _run(cuda_lib, 8, 1, 20000, 64, 1, 576, 512, 2048, True, 2, 500,
         kv_len=[20000, 19000, 3000, 2048, 2049, 100, 1, 20000])


def test_layers_share_index_but_not_outputs(cuda_lib):
    outs = _run(cuda_lib, 1, 64, 64, 4, 4, 64, 64, 16, False, 4, 600)
    for l in range(1, 4):
        assert not torch.equal(outs[0], outs[l])


@pytest.mark.parametrize("topk", [65, 129, 1000])
def test_mqa_latent_ragged_half_tiles(cuda_lib, topk):
    # the tensor-core kernel takes keys 64 at a time: a last half-tile with 1, 1 or 40 keys,
    # padding anywhere in the rows, two sequences of different lengths
    rows = np.unique(np.r_[0, 1, np.linspace(0, 399, 20).astype(int), 199, 200, 399])
    _run(cuda_lib, 2, 200, 1500, 64, 1, 576, 512, topk, True, 1, 700 + topk,
         kv_len=[1500, 700], pad_frac=0.2, rows=rows)


def test_mqa_latent_decode_one_half_tile_per_split(cuda_lib):
    # four rows of 128 keys: every row splits into two CTAs of one 64-key half-tile each
    _run(cuda_lib, 4, 1, 5000, 64, 1, 576, 512, 128, True, 2, 800,
         kv_len=[5000, 129, 64, 2000])
