"""GPU parity on the five workloads, at their full sizes, in the launch
configuration the benchmark times (one IndexShare group per test).

The oracle checks every row the CPU can score in seconds (all rows at L <= 1024,
a stratified sample beyond), plus properties on every row (padding, causality,
uniqueness via the checker's structural asserts on the sampled rows and a global
range check here)."""
import numpy as np
import pytest
import torch

from parity import check_attn, check_indexer, stratified_rows
from workloads import get_config, make_attn_inputs, make_indexer_inputs

pytestmark = pytest.mark.gpu


def _global_index_properties(idx, T, S, topk):
    """Every row: n = min(k, p+1) valid, distinct, causal entries, then -1 padding."""
    B = idx.shape[0]
    t = torch.arange(T, device=idx.device).view(1, T, 1)
    p = (S - T) + t
    n = torch.clamp(p + 1, max=topk)
    pos = torch.arange(topk, device=idx.device).view(1, 1, topk)
    valid = pos < n
    assert torch.all(idx[~valid.expand(B, T, topk)] == -1)
    vi = torch.where(valid, idx, torch.zeros_like(idx))
    assert torch.all((vi >= 0) & (vi <= p))
    srt, _ = torch.sort(torch.where(valid, idx, -1 - pos), dim=-1)
    assert torch.all(srt[..., 1:] != srt[..., :-1]), "duplicate index in a row"


def _group(cuda_lib, cfg, group, idx_rows, attn_rows, exact):
    qI, kI, w = make_indexer_inputs(cfg, group, "cuda")
    idx, sc = cuda_lib.indexer_topk(qI, kI, w, cfg.topk, want_score=True)
    cuda_lib.device_status()
    if cfg.B == 1 and cfg.T == cfg.S:
        _global_index_properties(idx, cfg.T, cfg.S, cfg.topk)
    rec = check_indexer(qI.cpu(), kI.cpu(), w.cpu(), cfg.topk, idx.cpu(), sc.cpu(),
                        rows=idx_rows, exact=exact)
    del qI, kI, w
    if cfg.n_layers == 0:
        return rec
    sel = torch.as_tensor(np.asarray(attn_rows))
    for l0 in range(cfg.group):
        layer = group * cfg.group + l0
        Q, K, V = make_attn_inputs(cfg, layer, "cuda")
        out = cuda_lib.sparse_attn_group([Q], [K], None if V is None else [V], idx, cfg.scale,
                                         Dv=cfg.Dv)[0]
        cuda_lib.device_status()
        rows_T = cfg.B * cfg.T
        check_attn(Q.reshape(rows_T, cfg.H, cfg.Dqk)[sel.cuda()].cpu(), K.cpu(),
                   None if V is None else V.cpu(),
                   idx.reshape(rows_T, cfg.topk)[sel.cuda()].cpu(), cfg.scale,
                   out.reshape(rows_T, cfg.H, cfg.Dv)[sel.cuda()].cpu(), attn_rows, cfg.T,
                   cfg.Dv)
        del Q, K, V, out
    torch.cuda.empty_cache()
    return rec


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.empty_cache()


def test_config1_tiny_group(cuda_lib):
    cfg = get_config(1)
    _group(cuda_lib, cfg, 0, np.arange(cfg.T), np.arange(cfg.T), exact=True)


def test_config2_indexer_int_e4m3_exact(cuda_lib):
    cfg = get_config(2)
    rows = stratified_rows(cfg.T, 160, cfg.topk, extra=range(cfg.T - 8, cfg.T))
    _group(cuda_lib, cfg, 0, rows, None, exact=True)


def test_config3_group_bf16(cuda_lib):
    cfg = get_config(3)
    rows = stratified_rows(cfg.T, 260, cfg.topk)
    arows = stratified_rows(cfg.T, 66, cfg.topk)
    assert len(rows) >= 256 and len(arows) >= 64
    rec = _group(cuda_lib, cfg, 0, rows, arows, exact=False)
    assert rec > 0.99


@pytest.mark.parametrize("group", [0, 1, 2, 3])
def test_config4_group_e4m3_full_size(cuda_lib, group):
    # every IndexShare group of the 16-layer stack: 256 stratified indexer rows and 64
    # attention rows per layer, the sample shifted per group so the groups cover different rows
    cfg = get_config(4)
    shift = 997 * group
    rows = [(r + shift) % cfg.T if 0 < r < cfg.T - 2 else r
            for r in stratified_rows(cfg.T, 260, cfg.topk)]
    arows = [(r + shift) % cfg.T if 0 < r < cfg.T - 2 else r
             for r in stratified_rows(cfg.T, 66, cfg.topk)]
    rows, arows = sorted(set(rows)), sorted(set(arows))
    assert len(rows) >= 256 and len(arows) >= 64
    rec = _group(cuda_lib, cfg, group, rows, arows, exact=False)
    assert rec > 0.99


def test_config5_decode(cuda_lib):
    cfg = get_config(5)
    rows = np.arange(cfg.B * cfg.T)
    rec = _group(cuda_lib, cfg, 0, rows, rows, exact=False)
    assert rec > 0.99
