"""CPU oracle (ctypes wrapper around ``tsi_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it and shares no code with it.

Every function computes in double precision from the stored bit patterns of its
inputs; see the C file's header for the passages each function follows.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsi_oracle.c")
_LIB = os.path.join(_HERE, "libtsi_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"f32": 0, "bf16": 1, "e4m3": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no machine-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.tsio_decode.argtypes = [vp, i64, i32]
            lib.tsio_decode.restype = dbl
            lib.tsio_decode_n.argtypes = [vp, i64, i32, vp]
            lib.tsio_decode_n.restype = None
            lib.tsio_indexer_topk.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                              vp, i64, vp, vp, vp, vp, i32]
            lib.tsio_indexer_topk.restype = i32
            lib.tsio_indexer_scores.argtypes = [vp, vp, vp, i32, i32, i32, i32, i64, vp]
            lib.tsio_indexer_scores.restype = i64
            lib.tsio_sparse_attn.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                             dbl, vp, i32, vp, i64, vp, vp, vp, i32]
            lib.tsio_sparse_attn.restype = i32
            _lib = lib
    return _lib


def _as_bytes_array(x):
    """Return (numpy array with the tensor's raw storage, dtype name)."""
    import torch

    if isinstance(x, np.ndarray):
        if x.dtype == np.float32:
            return np.ascontiguousarray(x), "f32"
        raise TypeError("numpy inputs must be float32; pass torch tensors for bf16/e4m3")
    x = x.detach().to("cpu").contiguous()
    if x.dtype == torch.float32:
        return x.numpy(), "f32"
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy(), "bf16"
    if x.dtype == torch.float8_e4m3fn:
        return x.view(torch.uint8).numpy(), "e4m3"
    raise TypeError(f"unsupported dtype {x.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def n_threads_default() -> int:
    return max(1, os.cpu_count() or 1)


def decode(x) -> np.ndarray:
    """Decode every stored element of ``x`` to float64 (oracle's own decoder)."""
    arr, dt = _as_bytes_array(x)
    flat = np.ascontiguousarray(arr.reshape(-1))
    out = np.empty(flat.size, dtype=np.float64)
    _load().tsio_decode_n(_ptr(flat), flat.size, DTYPE_CODE[dt], _ptr(out))
    return out.reshape(arr.shape)


def _rows_arrays(B, T, rows):
    if rows is None:
        rb = np.repeat(np.arange(B, dtype=np.int32), T)
        rt = np.tile(np.arange(T, dtype=np.int32), B)
    else:
        rows = np.asarray(rows, dtype=np.int64).reshape(-1)
        rb = (rows // max(T, 1)).astype(np.int32)
        rt = (rows % max(T, 1)).astype(np.int32)
    return np.ascontiguousarray(rb), np.ascontiguousarray(rt)


def _take_rows(x, sel):
    """x[sel] on the CPU, also for float8 (gathered through a same-size integer view)."""
    import torch

    x = x.detach().to("cpu")
    if x.dtype == torch.float8_e4m3fn:
        return x.view(torch.uint8)[sel].view(torch.float8_e4m3fn)
    return x[sel]


def indexer_topk(qI, kI, w, topk, kv_len=None, rows=None, n_threads=None):
    """Top-k of I[t,s] = sum_j w[t,j] ReLU(qI[t,j].kI[s]) over s <= p_t.

    qI [B,T,H_I,d_I], kI [B,S,d_I], w [B,T,H_I]; ``rows`` lists flattened query
    rows b*T+t (default: all).  Returns (idx int32 [n,topk], score float64
    [n,topk]) in rank order (score desc, index asc), padded with -1 / -inf.
    """
    import torch

    B, T, H_I, d_I = qI.shape
    rb, rt = _rows_arrays(B, T, rows)
    flat = rb.astype(np.int64) * T + rt
    q_rows = qI.reshape(B * T, H_I, d_I)
    w_rows = w.reshape(B * T, H_I)
    if rows is not None:
        sel = torch.as_tensor(flat)
        if int(sel.min()) < 0 or int(sel.max()) >= B * T:
            raise IndexError("rows out of range")
        q_rows = _take_rows(q_rows, sel)
        w_rows = _take_rows(w_rows, sel)
    return indexer_topk_rows(q_rows, kI, w_rows, topk, T, flat, kv_len, n_threads)


def indexer_topk_rows(q_rows, kI, w_rows, topk, T, rows, kv_len=None, n_threads=None):
    """Like ``indexer_topk`` with query-side tensors already compacted to ``rows``."""
    import torch

    B, S, d_I = kI.shape
    n, H_I = q_rows.shape[0], q_rows.shape[1]
    rb, rt = _rows_arrays(B, T, rows)
    assert rb.size == n
    q_arr, qdt = _as_bytes_array(q_rows)
    k_arr, kdt = _as_bytes_array(kI)
    w_arr, wdt = _as_bytes_array(w_rows)
    assert qdt == kdt
    kv = None if kv_len is None else np.ascontiguousarray(
        torch.as_tensor(kv_len).to("cpu", torch.int32).numpy())
    idx = np.empty((n, topk), dtype=np.int32)
    sc = np.empty((n, topk), dtype=np.float64)
    rc = _load().tsio_indexer_topk(_ptr(q_arr), _ptr(k_arr), _ptr(w_arr), DTYPE_CODE[qdt],
                                   DTYPE_CODE[wdt], B, T, S, H_I, d_I, topk, _ptr(kv), n,
                                   _ptr(rb), _ptr(rt), _ptr(idx), _ptr(sc),
                                   n_threads or n_threads_default())
    if rc != 0:
        raise RuntimeError(f"oracle indexer_topk failed ({rc})")
    return idx, sc


def indexer_scores(q_row, k_seq, w_row, p):
    """All scores I[s], s = 0..p, of one query row (q_row [H_I,d_I], k_seq [S,d_I])."""
    H_I, d_I = q_row.shape
    q_arr, qdt = _as_bytes_array(q_row)
    k_arr, kdt = _as_bytes_array(k_seq)
    w_arr, wdt = _as_bytes_array(w_row)
    assert qdt == kdt
    out = np.empty(max(int(p) + 1, 1), dtype=np.float64)
    n = _load().tsio_indexer_scores(_ptr(q_arr), _ptr(k_arr), _ptr(w_arr), DTYPE_CODE[qdt],
                                    DTYPE_CODE[wdt], H_I, d_I, int(p), _ptr(out))
    if n < 0:
        raise RuntimeError("oracle indexer_scores failed")
    return out[:n]


def sparse_attn(q_rows, k, v, idx_rows, scale, T, rows, Dv=None, kv_len=None, n_threads=None):
    """O[r,h,:] = softmax over row r's selected keys of scale*Q.K, applied to V.

    q_rows [n,H,Dqk] (compacted to ``rows``, flattened b*T+t), k [B,S,Hkv,Dqk],
    v [B,S,Hkv,Dv] or None (then the value is the first ``Dv`` dims of k),
    idx_rows [n,topk] (entries outside [0, kv_len[b]) are not keys).
    Returns float64 [n,H,Dv].
    """
    import torch

    B, S, Hkv, Dqk = k.shape
    n, H, Dqk2 = q_rows.shape
    assert Dqk2 == Dqk
    if v is not None:
        Dv = v.shape[-1]
    if Dv is None:
        raise ValueError("Dv required when v is None")
    rb, rt = _rows_arrays(B, T, rows)
    assert rb.size == n
    q_arr, qdt = _as_bytes_array(q_rows)
    k_arr, kdt = _as_bytes_array(k)
    v_arr = None
    if v is not None:
        v_arr, vdt = _as_bytes_array(v)
        assert vdt == kdt
    assert qdt == kdt
    idx = np.ascontiguousarray(torch.as_tensor(idx_rows).to("cpu", torch.int32).numpy())
    topk = idx.shape[-1]
    assert idx.shape[0] == n
    kv = None if kv_len is None else np.ascontiguousarray(
        torch.as_tensor(kv_len).to("cpu", torch.int32).numpy())
    out = np.empty((n, H, Dv), dtype=np.float64)
    rc = _load().tsio_sparse_attn(_ptr(q_arr), _ptr(k_arr), _ptr(v_arr), DTYPE_CODE[qdt], B, T, S,
                                  H, Hkv, Dqk, Dv, float(scale), _ptr(idx), topk, _ptr(kv), n,
                                  _ptr(rb), _ptr(rt), _ptr(out), n_threads or n_threads_default())
    if rc != 0:
        raise RuntimeError(f"oracle sparse_attn failed ({rc})")
    return out


def dsa_group(indexer_inputs, layers, topk, scale, Dv=None, kv_len=None, share=True,
              n_threads=None):
    """One IndexShare group (1 Full + Shared layers) or, with share=False, per-layer DSA.

    indexer_inputs: list of (qI, kI, w); with share=True only element 0 (the Full
    layer's indexer) is used and its index rows serve every layer ("GLM-5.2
    技术报告速览" §IndexShare: Shared layers inherit the nearest Full layer's index
    set; each layer still attends with its own Q/K/V).  With share=False layer l
    selects with indexer_inputs[l] (plain DSA).  layers: list of (Q, K, V) with
    Q [B,T,H,Dqk].  Returns (list of idx [B*T,topk], list of O float64 [B*T,H,Dv]).
    """
    idxs, outs = [], []
    full_idx = None
    for l, (Q, K, V) in enumerate(layers):
        if share:
            if full_idx is None:
                qI, kI, w = indexer_inputs[0]
                full_idx, _ = indexer_topk(qI, kI, w, topk, kv_len, n_threads=n_threads)
            idx = full_idx
        else:
            qI, kI, w = indexer_inputs[l]
            idx, _ = indexer_topk(qI, kI, w, topk, kv_len, n_threads=n_threads)
        B, T, H, Dqk = Q.shape
        rows = np.arange(B * T)
        outs.append(sparse_attn(Q.reshape(B * T, H, Dqk), K, V, idx, scale, T, rows, Dv=Dv,
                                kv_len=kv_len, n_threads=n_threads))
        idxs.append(idx)
    return idxs, outs


def index_share_layers(n_layers, freq=4, skip_offset=0, pattern=None):
    """Anchor layer of every layer of an IndexShare stack.

    "GLM 5.2: Built for Long Horizon Tasks" §5.2: the model config sets index_topk_freq,
    index_skip_topk_offset and index_topk_pattern, and after the offset the layer types
    repeat full, shared, shared, shared.  "GLM-5.2 技术报告速览" §IndexShare: a Shared
    layer inherits the index set of the nearest Full layer before it.  Reading (the pages
    do not spell out the layers before the offset): they keep their own indexer (Full).
    An explicit pattern ('F' / 'S' per layer) replaces freq and offset.
    """
    if pattern is not None:
        if len(pattern) != n_layers or any(c not in "FS" for c in pattern):
            raise ValueError("pattern must have one 'F' or 'S' per layer")
        kinds = list(pattern)
    else:
        kinds = []
        for layer in range(n_layers):
            if layer < skip_offset:
                kinds.append("F")
            else:
                kinds.append("F" if (layer - skip_offset) % freq == 0 else "S")
    anchors = []
    for layer, kind in enumerate(kinds):
        if kind == "F":
            anchors.append(layer)
        elif not anchors:
            raise ValueError("layer 0 must be a Full layer")
        else:
            anchors.append(anchors[-1])
    return anchors


def topk_overlap(idx_a, idx_b):
    """Per-row |S_a ∩ S_b| and |S_a| of two [rows, k] index arrays (entries < 0 are padding).

    "GLM-5.2 技术报告速览" §IndexShare: the pairwise overlap of the per-layer top-k index
    sets.  Written as plain set intersection, one row at a time.
    """
    a = np.asarray(idx_a).reshape(-1, np.asarray(idx_a).shape[-1])
    b = np.asarray(idx_b).reshape(a.shape)
    inter = np.zeros(a.shape[0], dtype=np.int64)
    card = np.zeros(a.shape[0], dtype=np.int64)
    for r in range(a.shape[0]):
        sa = {int(x) for x in a[r] if x >= 0}
        sb = {int(x) for x in b[r] if x >= 0}
        inter[r] = len(sa & sb)
        card[r] = len(sa)
    return inter, card


def shard_topk(q_row, k_shard, w_row, p, key_offset, topk):
    """Top-k of one query row over one key shard, as (scores, positions) in rank order.

    The shard holds keys key_offset .. key_offset + len(k_shard) - 1 of the whole cache;
    the row at position p keeps the keys s <= p among them ("GLM 5.2: Built for Long
    Horizon Tasks", discussion §4: the context split over ranks).  Rank order is score
    descending, position ascending; positions are those of the whole cache.
    """
    n_local = min(len(k_shard), int(p) + 1 - int(key_offset))
    if n_local <= 0:
        return np.zeros(0), np.zeros(0, dtype=np.int64)
    sc = indexer_scores(q_row, k_shard[:n_local], w_row, n_local - 1)
    pos = np.arange(n_local, dtype=np.int64) + int(key_offset)
    order = np.lexsort((pos, -sc))[:topk]
    return sc[order], pos[order]


def merge_topk(lists, topk):
    """Top-k of the union of candidate lists [(scores, positions), ...], rank order: the
    plain definition (concatenate, order by score descending then position ascending)."""
    if not lists:
        return np.zeros(0), np.zeros(0, dtype=np.int64)
    sc = np.concatenate([np.asarray(l[0], dtype=np.float64) for l in lists])
    pos = np.concatenate([np.asarray(l[1], dtype=np.int64) for l in lists])
    order = np.lexsort((pos, -sc))[:topk]
    return sc[order], pos[order]


def _logsumexp(x, axis=-1):
    """ln sum exp(x) along ``axis`` in float64 (-inf for an empty or all -inf slice)."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[axis] == 0:
        return np.full(np.delete(x.shape, axis), -np.inf)
    m = np.max(x, axis=axis, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore"):
        out = np.log(np.sum(np.exp(x - m_safe), axis=axis, keepdims=True)) + m_safe
    return np.squeeze(out, axis=axis)


def index_kl(q_layers, k_layers, idx_rows, score_rows, scale, T, rows, kv_len=None, lse=None):
    """Group-centroid KL target of a Full layer's indexer, per query row.

    "GLM-5.2 技术报告速览" §IndexShare, subsection "少数层挑，其余层复用": the Full
    layer's indexer is fitted, by KL, to the centroid of the head-averaged main-attention
    distributions of the layers it serves,

        pbar_t = 1/(m+1) * sum_{j=0..m} p^(l+j)_t,

    p^(l+j)_t being layer l+j's attention distribution of query t averaged over heads and
    m the number of Shared layers.  Reading taken here (the page leaves the key set and the
    KL direction to the sparse-attention setting it builds on): every distribution lives on
    the row's selected keys S_t (the entries of idx inside [0, kv_len[b])), the only keys
    the main attention of the group sees, and the loss is KL(pbar_t || q_t) with
    q_t = softmax over S_t of the indexer scores I[t, s].

    q_layers   list of [n, H, Dqk] query rows of each layer of the group (compacted to
               ``rows``, flattened b*T + t), Full layer first
    k_layers   list of [B, S, Dqk] (or [B, S, 1, Dqk]) key caches of the same layers
    idx_rows   [n, topk] the group's shared index rows; score_rows [n, topk] the indexer
               scores I[t, idx[t, i]] in the same order
    lse        optional [G, n, H]: log-partitions to normalise with instead of the exact
               ones (to check a kernel that is handed another implementation's values)
    Returns a dict of float64 arrays:
        lse   [G, n, H]  ln sum_{s in S_t} exp(scale * Q[t,h] . K[s])  (-inf: no key)
        p     [G, n, topk] head-averaged attention of each layer, 0 at padding
        pbar  [n, topk]   the centroid
        q     [n, topk]   the indexer distribution
        loss  [n]         KL(pbar_t || q_t), 0 for a row with no key
        grad  [n, topk]   d loss_t / d I[t, idx[t, i]] = q - pbar (pbar sums to one), 0 at
                          padding
    Library steps: float64 matmul for the logits; everything else is written out.
    """
    import torch

    G = len(q_layers)
    assert G >= 1 and len(k_layers) == G
    idx = np.asarray(torch.as_tensor(idx_rows).to("cpu", torch.int64).numpy())
    n, topk = idx.shape
    sc = np.asarray(torch.as_tensor(score_rows).to("cpu", torch.float64).numpy()).reshape(n, topk)
    k_shapes = [tuple(k.shape) for k in k_layers]
    B, S = k_shapes[0][0], k_shapes[0][1]
    rb, _ = _rows_arrays(B, T, rows)
    kv = None if kv_len is None else np.asarray(torch.as_tensor(kv_len).to("cpu").numpy())
    # decode each layer's queries once; keys once per layer when small, else per row
    qd = [decode(q).reshape(n, q.shape[-2], q.shape[-1]) for q in q_layers]
    H = qd[0].shape[1]
    small = all(int(np.prod(s)) <= (1 << 24) for s in k_shapes)
    kd = [decode(k).reshape(B, S, -1) for k in k_layers] if small else None
    out = {
        "lse": np.full((G, n, H), -np.inf),
        "p": np.zeros((G, n, topk)),
        "pbar": np.zeros((n, topk)),
        "q": np.zeros((n, topk)),
        "loss": np.zeros(n),
        "grad": np.zeros((n, topk)),
    }
    for r in range(n):
        b = int(rb[r])
        length = S if kv is None else int(kv[b])
        valid = (idx[r] >= 0) & (idx[r] < length)
        if not valid.any():
            continue
        sel = idx[r][valid]
        for l in range(G):
            if kd is not None:
                keys = kd[l][b, sel]
            else:
                kl = k_layers[l].reshape(B, S, -1)
                keys = decode(_take_rows(kl[b], torch.as_tensor(sel)))
            logits = scale * (qd[l][r] @ keys.T)  # [H, |S_t|]
            lse_l = _logsumexp(logits, axis=1)  # [H]
            lse_given = None if lse is None else np.asarray(lse[l][r], dtype=np.float64)
            lse_use = lse_l if lse_given is None else lse_given
            probs = np.exp(logits - lse_use[:, None])  # softmax of every head over S_t
            out["lse"][l, r] = lse_l
            out["p"][l, r, valid] = probs.mean(axis=0)  # average over the H heads
        pbar = out["p"][:, r, :].sum(axis=0) / G  # centroid of the group's layers
        out["pbar"][r] = pbar
        i_valid = sc[r][valid]
        log_q = i_valid - _logsumexp(i_valid)
        q = np.exp(log_q)
        out["q"][r, valid] = q
        pv = pbar[valid]
        pos = pv > 0
        out["loss"][r] = np.sum(pv[pos] * (np.log(pv[pos]) - log_q[pos]))
        out["grad"][r, valid] = q - pv
    return out
