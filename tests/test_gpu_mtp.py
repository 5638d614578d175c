"""MTP with IndexShare ("GLM 5.2: Built for Long Horizon Tasks" §5.3: the first MTP step
runs the indexer and later steps reuse its top-k indices; §5.2: the config's
index_share_for_mtp_iteration).  Decode with the tensor-core kernels: step 1 selects the
keys of its query at position kv_len - 1; draft step j (a query at kv_len - 1 + j over a
cache j tokens longer) attends over step 1's index rows with its own Q and latent.  Each
step is checked against the oracle on the same index rows."""
import numpy as np
import pytest
import torch

import oracle
from parity import check_attn, check_indexer
from workloads import get_config, make_indexer_inputs
from workloads.gen import draw

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("steps", [3])
def test_mtp_steps_reuse_first_step_indices(cuda_lib, steps):
    cfg = get_config(4)
    B, S, k = 4, 20000, cfg.topk
    kv0 = [20000 - steps, 7000, 2049, 900]  # cache lengths at step 1 (room for the drafts)
    dev = "cuda"
    icfg = cfg.with_(B=B, T=1, S=S)
    qI, kI, w = make_indexer_inputs(icfg, 0, dev)
    kv1 = torch.tensor(kv0, dtype=torch.int32, device=dev)
    idx1, sc1 = cuda_lib.indexer_topk(qI, kI, w, k, kv_len=kv1, want_score=True)
    cuda_lib.device_status()
    check_indexer(qI.cpu(), kI.cpu(), w.cpu(), k, idx1.cpu(), sc1.cpu(),
                  kv_len=torch.tensor(kv0), exact=False)
    # one latent cache per layer (the MTP layer) long enough for every draft step
    K = draw((B, S, 1, cfg.Dqk), "normal", "bf16", 4242, dev)
    for j in range(steps):
        kv_j = [n + j for n in kv0]
        Q = draw((B, 1, cfg.H, cfg.Dqk), "normal", "bf16", 5000 + j, dev)
        kv = torch.tensor(kv_j, dtype=torch.int32, device=dev)
        out = cuda_lib.sparse_attn_group([Q], [K], None, idx1, cfg.scale, kv_len=kv, Dv=cfg.Dv)[0]
        cuda_lib.device_status()
        rows = np.arange(B)
        check_attn(Q.reshape(B, cfg.H, cfg.Dqk).cpu(), K.cpu(), None,
                   idx1.reshape(B, k).cpu(), cfg.scale, out.reshape(B, cfg.H, cfg.Dv).cpu(),
                   rows, 1, cfg.Dv, kv_len=torch.tensor(kv_j))
        # the reused rows hold positions of step 1 only: every one is below step j's length
        ids = idx1.reshape(B, k).cpu().numpy()
        for b in range(B):
            sel = ids[b][ids[b] >= 0]
            assert sel.size == min(k, kv0[b]) and sel.max() < kv_j[b] - j


def test_mtp_reuse_equals_fresh_selection_when_indexer_agrees(cuda_lib):
    # if the draft step's own indexer would pick the same set (same indexer query, the
    # newest key scoring lowest), reuse and recomputation give the same attention
    cfg = get_config(4)
    B, S, k = 2, 5000, 64
    dev = "cuda"
    icfg = cfg.with_(B=B, T=1, S=S)
    qI, kI, w = make_indexer_inputs(icfg, 1, dev)
    kv0 = torch.tensor([3000, 4000], dtype=torch.int32, device=dev)
    idx1 = cuda_lib.indexer_topk(qI, kI, w, k, kv_len=kv0)
    # the draft step's cache: one more key per sequence, all-zero so that it scores 0
    kI2 = kI.clone()
    for bb, n in enumerate(kv0.tolist()):
        kI2.view(torch.uint8)[bb, n] = 0  # e4m3 zero is the all-zero byte
    kv1 = kv0 + 1
    idx2 = cuda_lib.indexer_topk(qI, kI2, w, k, kv_len=kv1)
    cuda_lib.device_status()
    a = np.sort(idx1.reshape(B, k).cpu().numpy(), axis=1)
    b = np.sort(idx2.reshape(B, k).cpu().numpy(), axis=1)
    ref_i, _ = oracle.indexer_topk(qI.cpu(), kI2.cpu(), w.cpu(), k, kv_len=kv1.cpu())
    # scores are w . ReLU(q . k) >= 0 with the uniform gate: the new key scores 0 and loses
    # every tie to lower positions, so with at least k positive scores the set is unchanged
    assert (np.sort(np.asarray(ref_i).reshape(B, k), axis=1) >= 0).all()
    assert np.array_equal(a, b)
