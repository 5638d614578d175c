"""Work accounting for the DSA indexer + top-k + sparse attention path.

Closed forms used by the benchmark to turn times into rates and roofline
fractions (pure host arithmetic, no kernels):

* causal pairs of a prefill: sum over query rows of (p_t + 1) keys, p_t the
  row's position -- "GLM 5.2: Built for Long Horizon Tasks", discussion §2
  (about 5e11 candidate pairs at L = 1M);
* selected pairs: sum of min(k, p_t + 1) -- same passage (about 2.05e9 at
  L = 1M, k = 2048);
* the DSA / IndexShare cost model T_DSA ~ N C_I L^2 + N C_A L k and
  T_IndexShare ~ r N C_I L^2 + N C_A L k -- same page, discussion §3.
"""


def query_positions(T: int, kv_len: int):
    """Positions p_t of the T query rows of a sequence holding kv_len keys."""
    return range(kv_len - T, kv_len)


def causal_pairs(B: int, T: int, S: int, kv_len=None) -> int:
    """Number of (query, key) pairs with key <= query position, over all rows."""
    total = 0
    for b in range(B):
        n = S if kv_len is None else max(0, min(int(kv_len[b]), S))
        lo = n - T  # position of row 0
        # sum_{t=0}^{T-1} max(0, lo + t + 1)
        first = max(0, -lo)  # first row with a non-negative key count
        if first >= T:
            continue
        a = lo + first + 1
        z = lo + T
        total += (a + z) * (z - a + 1) // 2
    return total


def selected_pairs(B: int, T: int, S: int, topk: int, kv_len=None) -> int:
    """Number of selected keys: sum over rows of min(k, p_t + 1)."""
    total = 0
    for b in range(B):
        n = S if kv_len is None else max(0, min(int(kv_len[b]), S))
        lo = n - T  # row t holds c_t = lo + t + 1 keys
        c_lo, c_hi = max(1, lo + 1), lo + T
        if c_hi < 1:
            continue
        m = min(c_hi, topk)
        if m >= c_lo:  # rows with 1 <= c <= k contribute c
            total += (c_lo + m) * (m - c_lo + 1) // 2
        total += max(0, c_hi - max(topk, c_lo - 1)) * topk  # rows with c > k contribute k
    return total


def indexer_flops(pairs: int, H_I: int, d_I: int) -> int:
    """Tensor-core FLOPs of the indexer: 2 * H_I * d_I per causal pair."""
    return 2 * H_I * d_I * pairs


def indexer_bytes(rows: int, S_total_keys: int, H_I: int, d_I: int, qk_bytes: int,
                  w_bytes: int, topk: int) -> int:
    """Algorithmic HBM bytes of indexer + top-k: q, w, keys read once, idx written."""
    return rows * H_I * d_I * qk_bytes + rows * H_I * w_bytes + S_total_keys * d_I * qk_bytes \
        + rows * topk * 4


def attn_bytes(valid_k: int, rows: int, H: int, Hkv: int, Dqk: int, Dv: int, topk: int,
               v_from_k: bool, elem: int = 2) -> int:
    """Algorithmic bytes of one sparse-attention layer.

    Each selected key row is gathered once per query row (K, plus V when it is a
    separate tensor), Q is read and O written once, the index row is read once.
    """
    kv_row = Hkv * (Dqk if v_from_k else Dqk + Dv) * elem
    return valid_k * kv_row + rows * H * Dqk * elem + rows * H * Dv * elem + rows * topk * 4


def attn_flops(valid_k: int, H: int, Dqk: int, Dv: int) -> int:
    """FLOPs of one sparse-attention layer: 2*(Dqk + Dv) per (selected key, head)."""
    return 2 * valid_k * H * (Dqk + Dv)


def cost_dsa(N: int, L: int, k: int, C_I: float, C_A: float) -> float:
    """Prefill cost model of per-layer DSA: N C_I L^2 + N C_A L k."""
    return N * C_I * L * L + N * C_A * L * k


def cost_indexshare(N: int, L: int, k: int, C_I: float, C_A: float, r: float) -> float:
    """Prefill cost model with IndexShare (Full-layer ratio r): r N C_I L^2 + N C_A L k."""
    return r * N * C_I * L * L + N * C_A * L * k


def index_kl_bytes(valid_k: int, rows: int, n_layers: int, H: int, Dqk: int, topk: int,
                   grad: bool = True, pbar: bool = False, elem: int = 2) -> int:
    """Algorithmic bytes of the group-centroid KL target over one group of n_layers layers
    ("GLM-5.2 技术报告速览" §IndexShare: pbar_t = 1/(m+1) sum_j p^(l+j)_t).

    Per layer every selected key row (Dqk elements) is gathered once per query row and the
    row's queries (H x Dqk) and log-partitions (H fp32) are read once; the index row and its
    scores are read once, the loss (and the gradient / centroid rows) written once.
    """
    per_layer = valid_k * Dqk * elem + rows * H * Dqk * elem + rows * H * 4
    outs = rows * 4 + (rows * topk * 4 if grad else 0) + (rows * topk * 4 if pbar else 0)
    return n_layers * per_layer + rows * topk * 8 + outs


def index_kl_flops(valid_k: int, n_layers: int, H: int, Dqk: int) -> int:
    """Tensor-core FLOPs of the recomputed logits: 2 * Dqk per (selected key, head, layer)."""
    return 2 * valid_k * H * Dqk * n_layers
