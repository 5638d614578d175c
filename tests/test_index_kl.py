"""Group-centroid KL target ("GLM-5.2 技术报告速览" §IndexShare, "少数层挑，其余层复用":
pbar_t = 1/(m+1) sum_j p^(l+j)_t, the indexer fitted to it by KL): the oracle pinned to
closed forms, textbook special cases, a finite-difference derivative and brute force, plus
the host-side argument checks of the C ABI (no GPU needed)."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import top_selection_indexer_gb300 as tsi


def _basis_keys(B, S, D):
    """K[b, s] = e_s (s < D): every key has its own coordinate, exactly representable."""
    k = torch.zeros(B, S, D)
    for s in range(min(S, D)):
        k[:, s, s] = 1.0
    return k.bfloat16()


def _kl(q_layers, k_layers, idx, score, scale, kv_len=None, T=None):
    n = idx.shape[0]
    T = n if T is None else T
    return oracle.index_kl([q.bfloat16() for q in q_layers], k_layers, idx,
                           torch.as_tensor(score, dtype=torch.float64), scale, T,
                           np.arange(n), kv_len=kv_len)


# ----------------------------------------------------------------------- closed forms

def test_one_hot_heads_give_head_counts():
    # head h of layer l puts all its weight on key pi_l(h) (logit 40 against 0): the layer's
    # head-averaged distribution is the share of heads pointing at each key, and the
    # centroid is the mean of those shares over the layers
    H, n, D, scale, A = 6, 5, 8, 0.5, 80.0
    K = _basis_keys(1, n, D)
    pis = [[0, 0, 3, 1, 3, 3], [4, 2, 2, 2, 0, 1]]
    qs = []
    for pi in pis:
        q = torch.zeros(1, H, D)
        for h, s in enumerate(pi):
            q[0, h, s] = A
        qs.append(q)
    idx = torch.tensor([[3, -1, 0, 4, 1, 2, -1]], dtype=torch.int32)
    score = np.zeros((1, 7))
    out = _kl(qs, [K, K], idx, score, scale)
    for i, s in enumerate(idx[0].tolist()):
        want = 0.0 if s < 0 else sum(pi.count(s) for pi in pis) / (len(pis) * H)
        assert abs(out["pbar"][0, i] - want) < 1e-12
    for l, pi in enumerate(pis):
        for i, s in enumerate(idx[0].tolist()):
            want = 0.0 if s < 0 else pi.count(s) / H
            assert abs(out["p"][l, 0, i] - want) < 1e-12


def test_two_level_softmax_closed_form():
    # Q[h] = a_h e_0 over basis keys: head h's logits are scale*a_h on key 0 and 0 on the
    # other n-1 keys, so softmax = (e^x, 1, ..., 1) / (e^x + n - 1) and lse = ln(e^x + n - 1)
    H, n, D, scale = 4, 6, 8, 0.75
    a = [1.0, 2.0, -1.5, 0.25]
    q = torch.zeros(1, H, D)
    for h in range(H):
        q[0, h, 0] = a[h]
    K = _basis_keys(1, n, D)
    idx = torch.tensor([[5, 0, 2, 1, 4, 3]], dtype=torch.int32)
    out = _kl([q], [K], idx, np.zeros((1, n)), scale)
    x = np.array(a) * scale
    z = np.exp(x) + n - 1
    np.testing.assert_allclose(out["lse"][0, 0], np.log(z), rtol=0, atol=1e-13)
    want_key0 = np.mean(np.exp(x) / z)
    want_other = np.mean(1.0 / z)
    for i, s in enumerate(idx[0].tolist()):
        assert abs(out["pbar"][0, i] - (want_key0 if s == 0 else want_other)) < 1e-14
    assert abs(out["pbar"].sum() - 1.0) < 1e-14


def test_kl_vanishes_when_the_indexer_matches_the_centroid():
    # Gibbs: KL(p || q) = 0 iff q = p.  Scores ln(pbar) + c (any c) reproduce pbar exactly.
    H, n, D, scale = 4, 6, 8, 0.75
    a = [1.0, 2.0, -1.5, 0.25]
    q = torch.zeros(1, H, D)
    for h in range(H):
        q[0, h, 0] = a[h]
    K = _basis_keys(1, n, D)
    idx = torch.tensor([[0, 1, 2, 3, 4, 5]], dtype=torch.int32)
    x = np.array(a) * scale
    z = np.exp(x) + n - 1
    pbar = np.array([np.mean(np.exp(x) / z)] + [np.mean(1.0 / z)] * (n - 1))
    out = _kl([q], [K], idx, np.log(pbar)[None] + 3.0, scale)
    assert abs(out["loss"][0]) < 1e-13
    assert np.abs(out["grad"]).max() < 1e-14
    # and any other scores give a positive divergence
    out2 = _kl([q], [K], idx, np.log(pbar)[None] + np.linspace(0, 0.3, n)[None], scale)
    assert out2["loss"][0] > 1e-4


def test_uniform_attention_against_scipy_entropy():
    # identical keys: every head is uniform over the selected keys, so pbar = 1/n and the
    # loss is the relative entropy of the uniform distribution to softmax(I)
    scipy_stats = pytest.importorskip("scipy.stats")
    scipy_special = pytest.importorskip("scipy.special")
    g = torch.Generator().manual_seed(3)
    H, n, D = 4, 9, 16
    K = torch.randn(1, 1, D, generator=g).expand(1, n, D).contiguous().bfloat16()
    qs = [torch.randn(1, H, D, generator=g) for _ in range(3)]
    idx = torch.randperm(n, generator=g).to(torch.int32)[None]
    score = torch.randn(1, n, generator=g).double().numpy() * 2
    out = _kl(qs, [K] * 3, idx, score, 0.3)
    np.testing.assert_allclose(out["pbar"][0], np.full(n, 1.0 / n), rtol=0, atol=1e-14)
    want = scipy_stats.entropy(np.full(n, 1.0 / n), scipy_special.softmax(score[0]))
    assert abs(out["loss"][0] - want) < 1e-12


# --------------------------------------------------------------- derivative and brute force

def _random_case(seed, G=3, H=5, n=11, D=12, S=16, n_pad=3):
    g = torch.Generator().manual_seed(seed)
    qs = [torch.randn(1, H, D, generator=g).bfloat16() for _ in range(G)]
    ks = [torch.randn(1, S, D, generator=g).bfloat16() for _ in range(G)]
    sel = torch.randperm(S, generator=g)[:n].to(torch.int32)
    idx = torch.cat([sel, torch.full((n_pad,), -1, dtype=torch.int32)])[None]
    score = torch.randn(1, n + n_pad, generator=g).double().numpy()
    return qs, ks, idx, score


def test_grad_is_the_derivative_of_the_loss():
    qs, ks, idx, score = _random_case(5)
    scale = 0.4
    base = _kl(qs, ks, idx, score, scale)
    eps = 1e-6
    for i in range(idx.shape[1]):
        sp, sm = score.copy(), score.copy()
        sp[0, i] += eps
        sm[0, i] -= eps
        fd = (_kl(qs, ks, idx, sp, scale)["loss"][0] - _kl(qs, ks, idx, sm, scale)["loss"][0]) / (2 * eps)
        assert abs(fd - base["grad"][0, i]) < 1e-8, (i, fd, base["grad"][0, i])


def test_brute_force_tiny():
    # every sum written out with math.exp / math.log, one term at a time
    G, H, n, D = 2, 2, 3, 3
    g = torch.Generator().manual_seed(11)
    qs = [torch.randn(1, H, D, generator=g).bfloat16() for _ in range(G)]
    ks = [torch.randn(1, 5, D, generator=g).bfloat16() for _ in range(G)]
    idx = torch.tensor([[4, 1, 2]], dtype=torch.int32)
    score = [[0.3, -1.2, 2.0]]
    scale = 0.9
    out = _kl(qs, ks, idx, np.array(score), scale)
    pbar = [0.0] * n
    for l in range(G):
        Q = qs[l].double()[0]
        Kl = ks[l].double()[0]
        for h in range(H):
            logits = []
            for i in range(n):
                s = int(idx[0, i])
                dot = 0.0
                for d in range(D):
                    dot += float(Q[h, d]) * float(Kl[s, d])
                logits.append(scale * dot)
            z = sum(math.exp(x) for x in logits)
            for i in range(n):
                pbar[i] += math.exp(logits[i]) / z / (H * G)
    zq = sum(math.exp(x) for x in score[0])
    loss = 0.0
    for i in range(n):
        qi = math.exp(score[0][i]) / zq
        loss += pbar[i] * math.log(pbar[i] / qi)
    np.testing.assert_allclose(out["pbar"][0], pbar, rtol=1e-12, atol=0)
    assert abs(out["loss"][0] - loss) < 1e-12


# -------------------------------------------------------------------------- invariants

def test_padding_and_out_of_range_entries_are_not_keys():
    qs, ks, idx, score = _random_case(7, n_pad=0)
    kv = torch.tensor([13])  # keys 13.. of the 16-key cache are past the sequence's end
    full = _kl(qs, ks, idx, score, 0.4, kv_len=kv)
    keep = [(i, s) for i, s in enumerate(idx[0].tolist()) if 0 <= s < 13]
    idx2 = torch.tensor([[s for _, s in keep]], dtype=torch.int32)
    score2 = score[:, [i for i, _ in keep]]
    comp = _kl(qs, ks, idx2, score2, 0.4, kv_len=kv)
    assert abs(full["loss"][0] - comp["loss"][0]) < 1e-13
    for j, (i, _) in enumerate(keep):
        assert abs(full["pbar"][0, i] - comp["pbar"][0, j]) < 1e-15
        assert abs(full["grad"][0, i] - comp["grad"][0, j]) < 1e-15
    dropped = [i for i in range(idx.shape[1]) if i not in dict(keep)]
    assert dropped and all(full["pbar"][0, i] == 0 and full["grad"][0, i] == 0 for i in dropped)


def test_permuting_the_index_row_permutes_the_outputs():
    qs, ks, idx, score = _random_case(8)
    perm = np.random.default_rng(0).permutation(idx.shape[1])
    a = _kl(qs, ks, idx, score, 0.4)
    b = _kl(qs, ks, idx[:, perm], score[:, perm], 0.4)
    assert abs(a["loss"][0] - b["loss"][0]) < 1e-13
    np.testing.assert_allclose(a["pbar"][0, perm], b["pbar"][0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(a["grad"][0, perm], b["grad"][0], rtol=0, atol=1e-15)


def test_centroid_is_the_mean_of_the_single_layer_distributions():
    qs, ks, idx, score = _random_case(9, G=3)
    group = _kl(qs, ks, idx, score, 0.4)
    singles = [_kl([qs[l]], [ks[l]], idx, score, 0.4)["pbar"] for l in range(3)]
    np.testing.assert_allclose(group["pbar"], sum(singles) / 3, rtol=0, atol=1e-15)
    assert abs(group["pbar"].sum() - 1.0) < 1e-13
    assert group["loss"][0] >= 0


def test_row_without_keys():
    qs, ks, _, _ = _random_case(10)
    idx = torch.full((1, 6), -1, dtype=torch.int32)
    out = _kl(qs, ks, idx, np.zeros((1, 6)), 0.4)
    assert out["loss"][0] == 0 and not out["pbar"].any() and not out["grad"].any()
    assert np.isneginf(out["lse"]).all()


# ------------------------------------------------------------------ host-side ABI checks

FAKE = 0x10000


@pytest.fixture(scope="module")
def lib():
    from top_selection_indexer_gb300 import _build

    _build.build()
    return tsi.load()


def _call(lib, **kw):
    a = dict(n=4, B=1, T=8, S=100, H=64, D=576, topk=64, loss=FAKE, grad=None, pbar=None,
             score=FAKE, lse=FAKE)
    a.update(kw)
    P = ctypes.c_void_p * max(a["n"], 1)
    ptrs = P(*([FAKE] * max(a["n"], 1)))
    lse = None if a["lse"] is None else P(*([a["lse"]] * max(a["n"], 1)))
    return lib.tsi_index_kl(a["n"], ptrs, ptrs, lse, a["B"], a["T"], a["S"], a["H"], a["D"],
                            0.1, FAKE, a["score"], a["topk"], None, a["loss"], a["grad"],
                            a["pbar"], None)


def test_index_kl_rejects_bad_arguments(lib):
    assert _call(lib, n=0) == tsi.ERR_INVALID_ARG
    assert _call(lib, n=9) == tsi.ERR_INVALID_ARG
    assert _call(lib, topk=0) == tsi.ERR_UNSUPPORTED
    assert _call(lib, topk=2049) == tsi.ERR_UNSUPPORTED
    assert _call(lib, H=32) == tsi.ERR_UNSUPPORTED
    assert _call(lib, D=512) == tsi.ERR_UNSUPPORTED
    assert _call(lib, loss=None) == tsi.ERR_INVALID_ARG
    assert _call(lib, score=None) == tsi.ERR_INVALID_ARG
    assert _call(lib, lse=None) == tsi.ERR_INVALID_ARG
    assert _call(lib, grad=FAKE + 4) == tsi.ERR_INVALID_ARG
    assert _call(lib, lse=FAKE + 8) == tsi.ERR_INVALID_ARG
    assert _call(lib, B=0) == tsi.OK


def test_given_log_partitions_rescale_each_head():
    # normalising with lse + c_h instead of the exact lse scales head h's probabilities by
    # exp(-c_h): with one head per layer the layer's distribution scales by exactly that
    qs, ks, idx, score = _random_case(12, G=2, H=1)
    exact = _kl(qs, ks, idx, score, 0.4)
    c = np.array([0.5, -0.25])
    given = oracle.index_kl([q.bfloat16() for q in qs], ks, idx, torch.as_tensor(score),
                            0.4, 1, np.arange(1), lse=exact["lse"] + c[:, None, None])
    for l in range(2):
        np.testing.assert_allclose(given["p"][l], exact["p"][l] * np.exp(-c[l]), rtol=1e-13,
                                   atol=0)
    np.testing.assert_allclose(given["lse"], exact["lse"], rtol=0, atol=0)
