"""Parity checks of the CUDA path against the CPU oracle (helpers for the GPU tests).

Index rule (indexer + top-k):
  * integer-valued inputs: every partial sum is an exact fp32 number, so the GPU's
    index rows and scores must equal the oracle's bit for bit;
  * other inputs: fp32 accumulation may reorder near-ties.  Every index that is in
    one row but not the other must have an oracle score within delta of the
    oracle's k-th score, delta_s = 2^-15 * sum_j |w_j| sum_d |q_jd k_sd| (the
    worst-case fp32 summation bound gamma_n for n = d_I + H_I + 1 <= 193 terms is
    below 2^-16 of that magnitude sum; doubled for the tensor core's accumulation
    order).  GPU scores must match the oracle's within the same delta, and the row
    must be in rank order.
Attention rule: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| per element, the oracle run
on the GPU's own index rows, so selection near-ties do not enter the tolerance.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

DELTA_EXP = -15
ATOL, RTOL = 2e-2, 1e-2


def stratified_rows(T, n, topk, extra=()):
    """Row sample: row 0, rows around k, the last rows, and an even spread."""
    rows = {0, T - 1, T - 2, T // 2}
    for r in (topk - 2, topk - 1, topk, topk + 1):
        if 0 <= r < T:
            rows.add(r)
    rows.update(int(x) for x in np.linspace(0, T - 1, max(n - len(rows), 2)))
    rows.update(extra)
    return sorted(r for r in rows if 0 <= r < T)


def _abs64(x):
    # magnitudes for the tolerance only (torch's exact widening casts)
    return np.abs(x.double().numpy())


def check_indexer(qI, kI, w, topk, idx_gpu, score_gpu=None, kv_len=None, rows=None,
                  exact=False):
    """Compare GPU idx [B,T,k] (+ scores) with the oracle on the given flattened rows.

    All tensors on the CPU.  Returns the mean recall |gpu & oracle| / |oracle|.
    """
    B, T, H_I, d_I = qI.shape
    S = kI.shape[1]
    if rows is None:
        rows = np.arange(B * T)
    rows = np.asarray(rows, dtype=np.int64)
    idx_o, sc_o = oracle.indexer_topk(qI, kI, w, topk, kv_len=kv_len, rows=rows)
    g_idx = idx_gpu.reshape(B * T, topk)[torch.as_tensor(rows)].numpy()
    g_sc = None if score_gpu is None else \
        score_gpu.reshape(B * T, topk)[torch.as_tensor(rows)].double().numpy()
    full = {}
    if not exact:  # full oracle score rows, computed in parallel (ctypes drops the GIL)
        def one(row):
            b, t = int(row) // T, int(row) % T
            n_len = S if kv_len is None else max(0, min(int(kv_len[b]), S))
            return row, oracle.indexer_scores(qI[b, t], kI[b], w[b, t], n_len - T + t)
        with ThreadPoolExecutor(max_workers=oracle.n_threads_default()) as ex:
            full = dict(ex.map(one, [int(x) for x in rows]))
    recalls = []
    kabs = {}
    for r, row in enumerate(rows):
        b, t = int(row) // T, int(row) % T
        n_len = S if kv_len is None else max(0, min(int(kv_len[b]), S))
        p = n_len - T + t
        n = max(0, min(topk, p + 1))
        gi, oi = g_idx[r], idx_o[r]
        # structure: n valid entries then -1 padding, unique, causal
        assert np.all(gi[n:] == -1), f"row {row}: padding"
        assert np.all((gi[:n] >= 0) & (gi[:n] <= p)), f"row {row}: out-of-range index"
        assert len(set(gi[:n].tolist())) == n, f"row {row}: duplicate index"
        if exact:
            np.testing.assert_array_equal(gi, oi, err_msg=f"row {row}")
            if g_sc is not None:
                np.testing.assert_array_equal(g_sc[r, :n], sc_o[r, :n], err_msg=f"row {row}")
            recalls.append(1.0)
            continue
        if n == p + 1:  # every causal key is selected: the set is fixed
            assert set(gi[:n].tolist()) == set(range(n)), f"row {row}: short row set"
        I = full[int(row)]
        if b not in kabs:
            kabs[b] = _abs64(kI[b])
        mag = (_abs64(w[b, t]) @ _abs64(qI[b, t])) @ kabs[b][:p + 1].T
        delta = np.ldexp(mag, DELTA_EXP)
        kth = sc_o[r, n - 1] if n > 0 else 0.0
        kth_pos = oi[n - 1] if n > 0 else 0
        diff = set(gi[:n].tolist()) ^ set(oi[:n].tolist())
        for s in diff:
            assert abs(I[s] - kth) <= delta[s] + delta[kth_pos], \
                f"row {row}: index {s} score {I[s]} vs k-th {kth} (delta {delta[s]})"
        if g_sc is not None and n > 0:
            err = np.abs(g_sc[r, :n] - I[gi[:n]])
            assert np.all(err <= delta[gi[:n]]), f"row {row}: score error {err.max()}"
            # rank order of the GPU row: score desc, then index asc
            s_, i_ = g_sc[r, :n], gi[:n]
            ok = (s_[:-1] > s_[1:]) | ((s_[:-1] == s_[1:]) & (i_[:-1] < i_[1:]))
            assert np.all(ok), f"row {row}: not in rank order"
        recalls.append(1.0 - len(set(oi[:n].tolist()) - set(gi[:n].tolist())) / max(n, 1))
    return float(np.mean(recalls)) if recalls else 1.0


def check_attn(q_rows, K, V, idx_rows, scale, out_rows, rows, T, Dv, kv_len=None):
    """Compare GPU O rows with the oracle run on the GPU's own index rows.

    q_rows [n,H,Dqk], idx_rows [n,k], out_rows [n,H,Dv]: the sampled flattened rows
    ``rows`` (b*T+t); K [B,S,Hkv,Dqk], V [B,S,Hkv,Dv] or None.  CPU tensors.
    """
    rows = np.asarray(rows, dtype=np.int64)
    ref = oracle.sparse_attn(q_rows, K, V, idx_rows, scale, T, rows, Dv=Dv, kv_len=kv_len)
    got = out_rows.double().numpy()
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} elements outside tolerance; "
                           f"max err {err.max():.3e}")
    return float(err.max())
