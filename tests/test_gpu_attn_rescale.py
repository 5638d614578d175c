"""GPU parity of the sparse attention when the online softmax must rescale.

The tensor-core attention keeps a running maximum per head and refreshes it only when a
logit exceeds it by 2^16 (log2 units, about 11 nats); the output accumulated so far is
then rescaled in place.  With N(0, 1) activations and the 1/sqrt(576) scale the logits of a
row spread over about one nat, so the other tests never take that branch after a row's
first keys.  Here the logits spread over tens of nats and rise along each index row:

  * Q[t, h] = sigma_h (0.95 base_t + 0.31 noise_th), sigma_h cycling over {1, 4, 16}: the
    heads share a direction, so one key order makes every head's logits rise, but only the
    sigma = 16 heads (logit std 16 nats) overrun the margin; the others keep alpha = 1, so a
    rescale factor applied to the wrong head changes their output by O(1);
  * prefill rows hold their keys in ascending order of base_t . K[s] (the running maximum
    climbs through the row: several refreshes per head);
  * decode rows put the row's lower-half keys in even 64-key half-tiles and its upper-half
    keys in odd ones, so each CTA of the split (two half-tiles here) refreshes inside its
    range and the combine merges partials whose maxima lie far apart.

The test first checks, from the inputs alone, that the branch is taken (the kernel's refresh
rule replayed in fp64 on the sampled rows), then compares outputs and log-partitions with the
oracle at the attention tolerance, and the group-centroid KL target fed by those
log-partitions.  Softmax over the selected positions: "GLM 5.2: Built for Long Horizon
Tasks", discussion §3; the shared index set: "GLM-5.2 技术报告速览", §IndexShare.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_attn
from workloads.gen import draw

pytestmark = pytest.mark.gpu

H, D, DV = 64, 576, 512
SCALE = 1.0 / D ** 0.5
LOG2E = 1.4426950408889634
MARGIN = 16.0  # the kernel's refresh margin in log2 units
SIGMAS = np.array([1.0, 4.0, 16.0])
# The attention's log-partition sums the bf16-rounded probabilities that multiply V; each is
# within a relative 2^-8 of the exact one (8 significant bits, round to nearest), so the sum
# is too and ln of it within ln(1 + 2^-8) < 3.9e-3.  With one key dominating a head (logit
# spreads of tens of nats here) that bound is reached; the fp32 logits add < 1e-4.
LSE_ATOL = 4e-3


def _q(B, T, seed, dev):
    """Q with a shared direction per row and a per-head scale (see the module docstring);
    also returns the shared direction (float32, CPU) that orders the keys."""
    base = draw((B, T, 1, D), "normal", "f32", seed, "cpu")
    noise = draw((B, T, H, D), "normal", "f32", seed + 1, "cpu")
    sig = torch.tensor(SIGMAS[np.arange(H) % len(SIGMAS)], dtype=torch.float32).view(1, 1, H, 1)
    q = (sig * (0.95 * base + 0.31 * noise)).to(torch.bfloat16)
    return q.to(dev), base[:, :, 0]


def _rows(B, T, S, topk, kv_len, base, K, seed, mode, pad_frac=0.0):
    """Index rows: a random causal key set per row, ordered by the shared direction's logit
    (ascending, or lower/upper halves interleaved by half-tile), -1 padding at the end."""
    g = np.random.default_rng(seed)
    idx = -np.ones((B, T, topk), dtype=np.int32)
    Kf = K.float()
    for b in range(B):
        n_len = S if kv_len is None else kv_len[b]
        for t in range(T):
            p = n_len - T + t
            n = max(0, min(topk, p + 1))
            if n and pad_frac:
                n = max(1, int(n * (1 - pad_frac)))
            if n == 0:
                continue
            keys = g.choice(p + 1, size=n, replace=False)
            z = (Kf[b, torch.as_tensor(keys)].reshape(n, D) @ base[b, t]).numpy()
            keys = keys[np.argsort(z, kind="stable")]
            if mode == "interleave":
                lo, hi = keys[: n // 2], keys[n // 2:]
                out = []
                for j in range(0, max(len(lo), len(hi)), 64):
                    out += list(lo[j:j + 64]) + list(hi[j:j + 64])
                keys = np.array(out, dtype=np.int64)
            idx[b, t, :n] = keys
    return torch.from_numpy(idx)


def _refreshes(q_rows, K, idx_rows, b_of_row, halves_per_split):
    """Number of (row, head, half-tile) events where the kernel's rule rescales the output
    accumulated so far: a half-tile (not the first of its CTA's range) whose largest logit
    exceeds the running maximum by more than the margin."""
    events = 0
    for r in range(q_rows.shape[0]):
        row = idx_rows[r].numpy()
        q = q_rows[r].double().numpy()  # [H, D]
        kb = K[b_of_row[r]].double().numpy().reshape(-1, D)
        n_half = (len(row) + 63) // 64
        for h0 in range(0, n_half, halves_per_split):
            m = np.full(H, -np.inf)
            for j, hf in enumerate(range(h0, min(n_half, h0 + halves_per_split))):
                ent = row[64 * hf: 64 * hf + 64]
                ent = ent[ent >= 0]
                if len(ent) == 0:
                    continue
                z = (kb[ent] @ q.T).max(axis=0) * SCALE * LOG2E  # [H]
                need = z > m + MARGIN
                if j > 0:
                    events += int(need.sum())
                m = np.where(need, z, m)
    return events


def _plan_halves_per_split(rows, topk, sms=152):
    """Half-tiles per CTA of a row, as the library plans it for `rows` query rows."""
    nh = (topk + 63) // 64
    ns = 1
    if 0 < rows < sms:
        ns = min(nh, (sms + rows - 1) // rows)
    return (nh + ns - 1) // ns


def _check_group(cuda_lib, B, T, S, topk, kv_len, mode, seed, rows, n_layers=2, pad_frac=0.0,
                 min_events=1):
    dev = "cuda"
    qs, bases = [], []
    for l in range(n_layers):
        q, base = _q(B, T, seed + 10 * l, dev)
        qs.append(q)
        bases.append(base)
    ks = [draw((B, S, 1, D), "normal", "bf16", seed + 10 * l + 5, dev) for l in range(n_layers)]
    # the index rows follow layer 0's direction (the Full layer); the Shared layer reuses
    # them, and its own direction is correlated with nothing: a mix of orders
    idx = _rows(B, T, S, topk, kv_len, bases[0], ks[0].cpu(), seed + 7, mode, pad_frac)
    kv = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=dev)
    outs, lses = cuda_lib.sparse_attn_group(qs, ks, None, idx.to(dev), SCALE, kv_len=kv, Dv=DV,
                                            want_lse=True)
    cuda_lib.device_status()
    rows = np.asarray(rows)
    sel = torch.as_tensor(rows)
    q0_rows = qs[0].reshape(B * T, H, D)[sel.to(dev)].cpu()
    idx_rows = idx.reshape(B * T, topk)[sel]
    hps = _plan_halves_per_split(B * T, topk)
    ev = _refreshes(q0_rows, ks[0].cpu(), idx_rows, rows // T, hps)
    assert ev >= min_events, f"the inputs take the rescale branch only {ev} times"
    kv_cpu = None if kv_len is None else torch.tensor(kv_len)
    for l in range(n_layers):
        check_attn(qs[l].reshape(B * T, H, D)[sel.to(dev)].cpu(), ks[l].cpu(), None, idx_rows,
                   SCALE, outs[l].reshape(B * T, H, DV)[sel.to(dev)].cpu(), rows, T, DV,
                   kv_len=kv_cpu)
    # log-partitions of every layer, then the KL target fed by them
    q_rows = [q.reshape(B * T, H, D)[sel.to(dev)].cpu() for q in qs]
    k_cpu = [k.cpu() for k in ks]
    zero = torch.zeros(len(rows), topk)
    ref = oracle.index_kl(q_rows, k_cpu, idx_rows, zero, SCALE, T, rows, kv_len=kv_cpu)
    got_lse = np.stack([lse.reshape(B * T, H).cpu().double().numpy()[rows] for lse in lses])
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isfinite(got_lse), fin)
    np.testing.assert_allclose(got_lse[fin], ref["lse"][fin], rtol=0, atol=LSE_ATOL)
    g = torch.Generator(device="cpu").manual_seed(seed + 9)
    sc = torch.randn(idx.shape, generator=g) * 2
    sc = torch.where(idx >= 0, sc, torch.full_like(sc, float("-inf"))).to(dev)
    loss, pbar = cuda_lib.index_kl(qs, [k.view(B, S, D) for k in ks], lses, idx.to(dev), sc,
                                   SCALE, kv_len=kv, want_pbar=True)
    cuda_lib.device_status()
    # the oracle handed the kernel's own log-partitions: the KL kernel's error alone
    ref2 = oracle.index_kl(q_rows, k_cpu, idx_rows, sc.reshape(B * T, topk)[sel.to(dev)].cpu(),
                           SCALE, T, rows, kv_len=kv_cpu, lse=got_lse)
    pb = pbar.reshape(B * T, topk).cpu().double().numpy()[rows]
    np.testing.assert_allclose(pb, ref2["pbar"], rtol=2e-4, atol=1e-9)
    ls = loss.reshape(-1).cpu().double().numpy()[rows]
    assert np.all(np.abs(ls - ref2["loss"]) <= 5e-4 * np.maximum(1.0, np.abs(ref2["loss"])))


def test_rescale_prefill_rows(cuda_lib):
    # one sequence of 2100 rows: rows beyond 2048 keys hold 32 full half-tiles
    T = 2100
    rows = np.unique(np.r_[0, 1, 63, 64, 65, 200, np.linspace(0, T - 1, 20).astype(int), T - 1])
    _check_group(cuda_lib, 1, T, T, 2048, None, "ascending", 31000, rows, min_events=100)


@pytest.mark.parametrize("topk,pad_frac", [(65, 0.0), (129, 0.2), (1000, 0.2)])
def test_rescale_ragged_half_tiles(cuda_lib, topk, pad_frac):
    # a last half-tile of one key (k = 65: that key alone overruns the margin), padding,
    # two sequences of different lengths
    rows = np.unique(np.r_[0, 1, np.linspace(0, 399, 16).astype(int), 199, 200, 399])
    _check_group(cuda_lib, 2, 200, 1500, topk, [1500, 700], "ascending", 32000 + topk, rows,
                 pad_frac=pad_frac, min_events=20)


def test_rescale_decode_split_rows(cuda_lib):
    # eight decode rows (two half-tiles per CTA), each CTA's second half-tile far above its
    # first; one row shorter than k
    kv = [20000, 19000, 3000, 2048, 2049, 1500, 4096, 20000]
    _check_group(cuda_lib, 8, 1, 20000, 2048, kv, "interleave", 33000, np.arange(8),
                 min_events=500)
