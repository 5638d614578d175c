"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes part of the oracle to something independent: the number
formats' own definitions (checked against torch's casts), closed forms,
special cases that reduce to a library routine (numpy matmul, torch.topk,
torch SDPA), brute force on tiny inputs and invariants stated by the pages.
Chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from top_selection_indexer_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _randint(g, lo, hi, shape, dtype=torch.float32):
    return torch.randint(lo, hi + 1, shape, generator=g).to(dtype)


# ------------------------------------------------------------------ number formats


def test_decode_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    x = codes.view(torch.float8_e4m3fn)
    ours = oracle.decode(x)
    ref = x.to(torch.float32).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_bf16_all_codes_match_torch():
    codes = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    x = codes.view(torch.bfloat16)
    ours = oracle.decode(x)
    ref = x.to(torch.float32).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------------------------ indexer score


def _scores(qI, kI, w, b, t, p):
    return oracle.indexer_scores(qI[b, t], kI[b], w[b, t], p)


def test_score_nonnegative_operands_reduce_to_matmul():
    # q >= 0 and k >= 0 make every ReLU the identity, so
    # I[s] = sum_j w_j (q_j . k_s) = ((w^T Q) K^T)[s]: a plain matrix product.
    g = torch.Generator().manual_seed(1)
    H_I, d_I, S = 5, 12, 40
    q = torch.rand(1, 1, H_I, d_I, generator=g)
    k = torch.rand(1, S, d_I, generator=g)
    w = torch.rand(1, 1, H_I, generator=g) * 3 - 1  # any sign
    got = _scores(q, k, w, 0, 0, S - 1)
    ref = (w[0, 0].double().numpy() @ q[0, 0].double().numpy()) @ k[0].double().numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_score_relu_odd_part_is_linear():
    # ReLU(x) - ReLU(-x) = x, so I(q) - I(-q) = sum_j w_j q_j . k_s, a matmul.
    g = torch.Generator().manual_seed(2)
    H_I, d_I, S = 7, 16, 50
    q = torch.randn(1, 1, H_I, d_I, generator=g)
    k = torch.randn(1, S, d_I, generator=g)
    w = torch.randn(1, 1, H_I, generator=g)
    diff = _scores(q, k, w, 0, 0, S - 1) - _scores(-q, k, w, 0, 0, S - 1)
    ref = (w[0, 0].double().numpy() @ q[0, 0].double().numpy()) @ k[0].double().numpy().T
    np.testing.assert_allclose(diff, ref, rtol=1e-12, atol=1e-12)
    # and the even part is |x|: I(q) + I(-q) = sum_j w_j |q_j . k_s|
    summ = _scores(q, k, w, 0, 0, S - 1) + _scores(-q, k, w, 0, 0, S - 1)
    ref2 = np.abs(q[0, 0].double().numpy() @ k[0].double().numpy().T).T @ w[0, 0].double().numpy()
    np.testing.assert_allclose(summ, ref2, rtol=1e-12, atol=1e-12)


def test_score_one_hot_head_and_unit_query():
    # Only head j0 gated (weight c), its query the unit vector e_d0:
    # I[s] = c * max(0, k[s, d0]).
    g = torch.Generator().manual_seed(3)
    H_I, d_I, S, j0, d0, c = 6, 9, 30, 4, 7, 2.5
    q = torch.randn(1, 1, H_I, d_I, generator=g)
    q[0, 0, j0] = 0
    q[0, 0, j0, d0] = 1
    w = torch.zeros(1, 1, H_I)
    w[0, 0, j0] = c
    k = torch.randn(1, S, d_I, generator=g)
    got = _scores(q, k, w, 0, 0, S - 1)
    ref = c * np.maximum(0.0, k[0, :, d0].double().numpy())
    np.testing.assert_array_equal(got, ref)


def test_score_row_is_causal_length():
    g = torch.Generator().manual_seed(4)
    q = torch.randn(1, 1, 2, 4, generator=g)
    k = torch.randn(1, 10, 4, generator=g)
    w = torch.ones(1, 1, 2)
    assert _scores(q, k, w, 0, 0, 6).shape == (7,)
    assert _scores(q, k, w, 0, 0, -1).shape == (0,)


# ------------------------------------------------------------------ top-k


def _brute_rank_select(I, k):
    """Rank by counting: s has rank #{s': I[s'] > I[s] or (I[s'] == I[s] and s' < s)}."""
    n = len(I)
    out = -np.ones(k, dtype=np.int64)
    for s in range(n):
        rank = 0
        for s2 in range(n):
            if I[s2] > I[s] or (I[s2] == I[s] and s2 < s):
                rank += 1
        if rank < k:
            out[rank] = s
    return out


@pytest.mark.parametrize("L,k,H_I", [(1, 1, 1), (2, 7, 4), (63, 7, 1), (64, 64, 4),
                                     (65, 7, 4), (127, 1, 4), (300, 64, 1)])
def test_topk_matches_brute_force_with_ties(L, k, H_I):
    g = torch.Generator().manual_seed(100 + L + k + H_I)
    d_I = 4
    # small integers: many exactly tied scores
    q = _randint(g, -2, 2, (1, L, H_I, d_I))
    kk = _randint(g, -2, 2, (1, L, d_I))
    w = _randint(g, 0, 2, (1, L, H_I))
    rows = sorted(set([0, min(1, L - 1), L // 2, max(0, L - 2), L - 1]))
    idx, sc = oracle.indexer_topk(q, kk, w, k, rows=rows)
    for r, t in enumerate(rows):
        I = _scores(q, kk, w, 0, t, t)
        ref = _brute_rank_select(I, k)
        np.testing.assert_array_equal(idx[r], ref)
        n = min(k, t + 1)
        np.testing.assert_array_equal(sc[r, :n], I[ref[:n]])
        assert np.all(np.isneginf(sc[r, n:]))


def test_topk_short_rows_select_every_causal_key():
    # Rows with p + 1 <= k select exactly {0..p} (causal rule).
    g = torch.Generator().manual_seed(5)
    L, k = 40, 16
    q = torch.randn(1, L, 3, 8, generator=g)
    kk = torch.randn(1, L, 8, generator=g)
    w = torch.rand(1, L, 3, generator=g)
    idx, _ = oracle.indexer_topk(q, kk, w, k)
    for t in range(k):
        assert sorted(idx[t, :t + 1].tolist()) == list(range(t + 1))
        assert np.all(idx[t, t + 1:] == -1)
    for t in range(k, L):
        assert np.all((idx[t] >= 0) & (idx[t] <= t))
        assert len(set(idx[t].tolist())) == k


def test_topk_zero_gate_gives_lowest_indices():
    # w == 0: every score is 0, the tie rule picks 0..min(k,p+1)-1 in order.
    g = torch.Generator().manual_seed(6)
    L, k = 50, 20
    q = torch.randn(1, L, 4, 8, generator=g)
    kk = torch.randn(1, L, 8, generator=g)
    w = torch.zeros(1, L, 4)
    idx, sc = oracle.indexer_topk(q, kk, w, k)
    for t in range(L):
        n = min(k, t + 1)
        np.testing.assert_array_equal(idx[t, :n], np.arange(n))
        assert np.all(sc[t, :n] == 0.0)


def test_topk_distinct_scores_match_torch_topk():
    # With distinct scores among the top k+1 the selection is torch.topk's
    # (sorted=True) output.
    g = torch.Generator().manual_seed(7)
    L, k, H_I, d_I = 400, 37, 4, 16
    q = torch.randn(1, L, H_I, d_I, generator=g)
    kk = torch.randn(1, L, d_I, generator=g)
    w = torch.rand(1, L, H_I, generator=g)
    rows = [50, 199, 399]
    idx, _ = oracle.indexer_topk(q, kk, w, k, rows=rows)
    for r, t in enumerate(rows):
        I = torch.from_numpy(_scores(q, kk, w, 0, t, t))
        top = torch.sort(I, descending=True).values[:k + 1]
        assert len(torch.unique(top)) == k + 1
        ref = torch.topk(I, k, sorted=True).indices.numpy()
        np.testing.assert_array_equal(idx[r], ref)


def test_topk_equal_scores_prefer_lower_index():
    # Duplicate key rows give bit-identical scores; the lower position must win.
    g = torch.Generator().manual_seed(8)
    L, k = 32, 3
    q = torch.randn(1, L, 2, 4, generator=g)
    kk = torch.randn(1, L, 4, generator=g)
    w = torch.rand(1, L, 2, generator=g)
    t = L - 1
    I = _scores(q, kk, w, 0, t, t)
    best = int(np.argmax(I))
    kk[0, 25] = kk[0, best]
    kk[0, 29] = kk[0, best]
    kk[0, 3] = kk[0, best]
    idx, _ = oracle.indexer_topk(q, kk, w, k, rows=[t])
    assert idx[0].tolist() == sorted({best, 3, 25, 29})[:3]


def test_topk_decode_row_uses_kv_len():
    # T = 1 query per sequence sits at position kv_len[b] - 1 and sees keys 0..kv_len-1.
    g = torch.Generator().manual_seed(9)
    B, S, k = 3, 60, 8
    q = torch.randn(B, 1, 2, 8, generator=g)
    kk = torch.randn(B, S, 8, generator=g)
    w = torch.rand(B, 1, 2, generator=g)
    kv_len = torch.tensor([60, 5, 33], dtype=torch.int32)
    idx, _ = oracle.indexer_topk(q, kk, w, k, kv_len=kv_len)
    for b in range(B):
        I = _scores(q, kk, w, b, 0, int(kv_len[b]) - 1)
        np.testing.assert_array_equal(idx[b], _brute_rank_select(I, k))


def test_topk_negative_zero_equals_zero():
    # -0.0 and +0.0 are equal scores, so the tie rule decides between them.
    q = torch.zeros(1, 4, 1, 2)
    q[0, :, 0, 0] = 1.0
    kk = torch.zeros(1, 4, 2)
    kk[0, :, 0] = torch.tensor([-1.0, 0.0, -2.0, 0.0])  # ReLU gives +0 for every key
    w = torch.tensor([[[-1.0], [-1.0], [-1.0], [-1.0]]]).reshape(1, 4, 1)  # w * 0 = -0
    idx, sc = oracle.indexer_topk(q, kk, w, 4, rows=[3])
    np.testing.assert_array_equal(idx[0], [0, 1, 2, 3])


# ------------------------------------------------------------------ sparse attention


def _sdpa_rows(Q, K, V, mask, scale):
    """torch SDPA in float64 for one sequence: Q [T,H,D], K/V [S,H,*], mask [T,S] bool."""
    import torch.nn.functional as F

    q = Q.double().permute(1, 0, 2).unsqueeze(0)
    k = K.double().permute(1, 0, 2).unsqueeze(0)
    v = V.double().permute(1, 0, 2).unsqueeze(0)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_attn_single_key_returns_its_value():
    g = torch.Generator().manual_seed(10)
    S, H, D = 20, 3, 8
    Q = torch.randn(1, H, D, generator=g).to(torch.bfloat16)
    K = torch.randn(1, S, 1, D, generator=g).to(torch.bfloat16)
    V = torch.randn(1, S, 1, 5, generator=g).to(torch.bfloat16)
    idx = np.full((1, 6), -1, dtype=np.int32)
    idx[0, 2] = 13
    out = oracle.sparse_attn(Q, K, V, idx, 0.3, 1, [0])
    for h in range(H):
        np.testing.assert_array_equal(out[0, h], V[0, 13, 0].double().numpy())


def test_attn_full_selection_is_causal_sdpa():
    # k >= p+1 with every causal key selected: textbook causal attention.
    g = torch.Generator().manual_seed(11)
    L, H, D, Dv = 24, 4, 16, 12
    Q = torch.randn(1, L, H, D, generator=g).to(torch.bfloat16)
    K = torch.randn(1, L, H, D, generator=g).to(torch.bfloat16)
    V = torch.randn(1, L, H, Dv, generator=g).to(torch.bfloat16)
    topk = 32
    idx = -np.ones((L, topk), dtype=np.int32)
    for t in range(L):
        idx[t, :t + 1] = np.arange(t + 1)[::-1]
    out = oracle.sparse_attn(Q.reshape(L, H, D), K, V, idx, 0.25, L, np.arange(L))
    mask = torch.tril(torch.ones(L, L, dtype=torch.bool))
    ref = _sdpa_rows(Q[0], K[0], V[0], mask, 0.25)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_attn_sparse_equals_dense_under_topk_mask_mqa_latent():
    # Sparse attention over the index set == dense attention with -inf outside it
    # ("GLM 5.2: Built for Long Horizon Tasks", discussion §3).  MQA latent: one
    # key head shared by all query heads, value = first Dv dims of the key.
    g = torch.Generator().manual_seed(12)
    L, H, Dqk, Dv, topk = 40, 4, 24, 16, 9
    Q = torch.randn(1, L, H, Dqk, generator=g).to(torch.bfloat16)
    K = torch.randn(1, L, 1, Dqk, generator=g).to(torch.bfloat16)
    idx = -np.ones((L, topk), dtype=np.int32)
    mask = torch.zeros(L, L, dtype=torch.bool)
    rs = np.random.default_rng(0)
    for t in range(L):
        n = min(topk, t + 1)
        sel = rs.choice(t + 1, size=n, replace=False)
        idx[t, :n] = sel
        mask[t, sel] = True
    out = oracle.sparse_attn(Q.reshape(L, H, Dqk), K, None, idx, 0.2, L, np.arange(L), Dv=Dv)
    Kx = K[0].expand(L, H, Dqk)
    Vx = K[0, :, :, :Dv].expand(L, H, Dv)
    ref = _sdpa_rows(Q[0], Kx, Vx, mask, 0.2)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_attn_grouped_heads_share_consecutive_kv_heads():
    # H query heads over Hkv key/value heads: query head h reads kv head h // (H/Hkv)
    # (the MQA latent is Hkv = 1, MHA is Hkv = H).  Checked against torch SDPA with
    # the kv heads repeated.
    g = torch.Generator().manual_seed(16)
    L, H, Hkv, D, Dv = 16, 6, 2, 8, 4
    Q = torch.randn(1, L, H, D, generator=g).to(torch.bfloat16)
    K = torch.randn(1, L, Hkv, D, generator=g).to(torch.bfloat16)
    V = torch.randn(1, L, Hkv, Dv, generator=g).to(torch.bfloat16)
    idx = -np.ones((L, L), dtype=np.int32)
    for t in range(L):
        idx[t, :t + 1] = np.arange(t + 1)
    out = oracle.sparse_attn(Q.reshape(L, H, D), K, V, idx, 0.4, L, np.arange(L))
    rep = H // Hkv
    ref = _sdpa_rows(Q[0], K[0].repeat_interleave(rep, dim=1), V[0].repeat_interleave(rep, dim=1),
                     torch.tril(torch.ones(L, L, dtype=torch.bool)), 0.4)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_attn_index_order_does_not_matter():
    g = torch.Generator().manual_seed(13)
    L, H, D, topk = 30, 2, 8, 10
    Q = torch.randn(1, H, D, generator=g).to(torch.bfloat16)
    K = torch.randn(1, L, 1, D, generator=g).to(torch.bfloat16)
    sel = np.array([3, 17, 29, 0, 8, 11, 12, -1, 25, -1], dtype=np.int32)
    a = oracle.sparse_attn(Q, K, None, sel[None], 0.5, 1, [0], Dv=D)
    b = oracle.sparse_attn(Q, K, None, sel[::-1].copy()[None], 0.5, 1, [0], Dv=D)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_attn_empty_row_is_zero():
    Q = torch.ones(1, 2, 4, dtype=torch.bfloat16)
    K = torch.ones(1, 5, 1, 4, dtype=torch.bfloat16)
    out = oracle.sparse_attn(Q, K, None, np.full((1, 3), -1, np.int32), 1.0, 1, [0], Dv=4)
    assert np.all(out == 0.0)


# ------------------------------------------------------------------ IndexShare


def test_indexshare_identical_indexers_equal_per_layer_dsa():
    # A group whose 4 layers hold identical indexer inputs: sharing the Full
    # layer's index set is the same computation as 4 independent DSA layers.
    g = torch.Generator().manual_seed(14)
    L, H_I, d_I, topk, H, D = 48, 3, 8, 6, 2, 8
    qI = torch.randn(1, L, H_I, d_I, generator=g)
    kI = torch.randn(1, L, d_I, generator=g)
    w = torch.rand(1, L, H_I, generator=g)
    layers = []
    for _ in range(4):
        layers.append((torch.randn(1, L, H, D, generator=g).to(torch.bfloat16),
                       torch.randn(1, L, 1, D, generator=g).to(torch.bfloat16), None))
    ind = [(qI, kI, w)] * 4
    i_sh, o_sh = oracle.dsa_group(ind, layers, topk, 0.3, Dv=D, share=True)
    i_ds, o_ds = oracle.dsa_group(ind, layers, topk, 0.3, Dv=D, share=False)
    for l in range(4):
        np.testing.assert_array_equal(i_sh[l], i_ds[l])
        np.testing.assert_array_equal(o_sh[l], o_ds[l])
    # The Shared layers attend over exactly the Full layer's index rows...
    for l in range(1, 4):
        np.testing.assert_array_equal(i_sh[l], i_sh[0])
    # ...and their outputs still differ, because each layer has its own Q/K/V.
    assert not np.allclose(o_sh[1], o_sh[2])


def test_indexshare_shared_layers_ignore_their_own_indexers():
    g = torch.Generator().manual_seed(15)
    L, topk = 40, 5
    ind = [(torch.randn(1, L, 2, 4, generator=g), torch.randn(1, L, 4, generator=g),
            torch.rand(1, L, 2, generator=g)) for _ in range(4)]
    layers = [(torch.randn(1, L, 2, 4, generator=g).to(torch.bfloat16),
               torch.randn(1, L, 1, 4, generator=g).to(torch.bfloat16), None) for _ in range(4)]
    i_sh, _ = oracle.dsa_group(ind, layers, topk, 0.5, Dv=4, share=True)
    i_ds, _ = oracle.dsa_group(ind, layers, topk, 0.5, Dv=4, share=False)
    np.testing.assert_array_equal(i_sh[0], i_ds[0])
    assert any(not np.array_equal(i_sh[0], i_ds[l]) for l in range(1, 4))


# ------------------------------------------------------------------ accounting


def test_pair_counts_match_pages_closed_forms():
    gold = json.load(open(os.path.join(GOLDEN, "pair_counts.json")))
    L, k, tol = gold["L"], gold["k"], gold["relative_tolerance"]
    assert accounting.causal_pairs(1, L, L) == L * (L + 1) // 2
    assert abs(accounting.causal_pairs(1, L, L) / gold["causal_pairs_approx"] - 1) < tol
    assert abs(accounting.selected_pairs(1, L, L, k) / gold["selected_pairs_approx"] - 1) < tol
    assert accounting.causal_pairs(1, 1, L) == gold["decode_candidates_approx"]
    assert accounting.selected_pairs(1, 1, L, k) == gold["decode_selected"]


@pytest.mark.parametrize("T,S,k,kv", [(5, 9, 3, None), (1, 9, 4, [7]), (10, 10, 4, None),
                                      (3, 5, 10, [2]), (7, 7, 1, None), (4, 6, 2, [0])])
def test_pair_counts_brute_force(T, S, k, kv):
    n = S if kv is None else kv[0]
    ps = range(n - T, n)
    assert accounting.causal_pairs(1, T, S, kv) == sum(max(0, p + 1) for p in ps)
    assert accounting.selected_pairs(1, T, S, k, kv) == sum(min(k, max(0, p + 1)) for p in ps)


def test_cost_model_indexshare_ratio():
    # With C_A = 0 the IndexShare/DSA ratio is r; with r = 1 they coincide.
    assert accounting.cost_indexshare(8, 100, 4, 1.0, 0.0, 0.25) == \
        pytest.approx(0.25 * accounting.cost_dsa(8, 100, 4, 1.0, 0.0))
    assert accounting.cost_indexshare(8, 100, 4, 1.0, 3.0, 1.0) == \
        accounting.cost_dsa(8, 100, 4, 1.0, 3.0)
