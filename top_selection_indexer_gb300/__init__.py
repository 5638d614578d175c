"""GB300-native DSA lightning indexer + top-k + IndexShare sparse attention.

Thin ctypes binding over ``libtsi.so`` (see ``include/tsi.h``): it checks that
tensors are CUDA and contiguous, allocates outputs / workspace with torch when
the caller passes none, and forwards device pointers and sizes.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.
"""
import ctypes
import os
import threading

from . import accounting  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsi.so")
_lib = None
_lock = threading.Lock()

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_ASSERT = \
    range(7)
F32, BF16, E4M3 = 0, 1, 2
MAX_TOPK = 2048

EXPORTS = ("tsi_indexer_topk_workspace", "tsi_indexer_topk", "tsi_indexer_topk_onchip_workspace",
           "tsi_indexer_topk_onchip", "tsi_indexer_topk_two_pass_workspace",
           "tsi_indexer_topk_two_pass", "tsi_sparse_attn_workspace",
           "tsi_sparse_attn_group", "tsi_device_status", "tsi_last_error", "tsi_version",
           "tsi_launch_count", "tsi_indexer_topk_noalloc", "tsi_indexer_topk_noalloc_limit",
           "tsi_indexer_topk_path", "tsi_sparse_attn_path", "tsi_index_share_layers",
           "tsi_topk_overlap", "tsi_indexer_topk_shard_workspace", "tsi_indexer_topk_shard",
           "tsi_topk_merge", "tsi_sparse_attn_group_lse", "tsi_index_kl",
           "tsi_selftest_wait_timeout")


class TSIError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"status {status}: {msg}")
        self.status = status


def load():
    """Load libtsi.so; raises if it has not been built (no silent fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
            lib.tsi_indexer_topk_workspace.argtypes = [i32] * 7
            lib.tsi_indexer_topk_workspace.restype = sz
            lib.tsi_indexer_topk.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                             vp, vp, vp, vp, sz, vp]
            lib.tsi_indexer_topk.restype = i32
            lib.tsi_indexer_topk_onchip_workspace.argtypes = [i32] * 7
            lib.tsi_indexer_topk_onchip_workspace.restype = sz
            lib.tsi_indexer_topk_onchip.argtypes = lib.tsi_indexer_topk.argtypes
            lib.tsi_indexer_topk_onchip.restype = i32
            lib.tsi_indexer_topk_two_pass_workspace.argtypes = [i32] * 7
            lib.tsi_indexer_topk_two_pass_workspace.restype = sz
            lib.tsi_indexer_topk_two_pass.argtypes = lib.tsi_indexer_topk.argtypes
            lib.tsi_indexer_topk_two_pass.restype = i32
            lib.tsi_sparse_attn_workspace.argtypes = [i32] * 8
            lib.tsi_sparse_attn_workspace.restype = sz
            lib.tsi_sparse_attn_group.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                  i32, f32, vp, i32, vp, vp, vp, sz, vp]
            lib.tsi_sparse_attn_group.restype = i32
            lib.tsi_device_status.argtypes = [vp]
            lib.tsi_device_status.restype = i32
            lib.tsi_last_error.argtypes = []
            lib.tsi_last_error.restype = ctypes.c_char_p
            lib.tsi_version.argtypes = []
            lib.tsi_version.restype = i32
            lib.tsi_launch_count.argtypes = []
            lib.tsi_launch_count.restype = ctypes.c_uint64
            lib.tsi_indexer_topk_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                     i32, i32, vp, vp, vp, vp]
            lib.tsi_indexer_topk_noalloc.restype = i32
            lib.tsi_indexer_topk_path.argtypes = [i32, i32, i32]
            lib.tsi_indexer_topk_path.restype = i32
            lib.tsi_sparse_attn_path.argtypes = [i32] * 5
            lib.tsi_sparse_attn_path.restype = i32
            lib.tsi_indexer_topk_noalloc_limit.argtypes = []
            lib.tsi_indexer_topk_noalloc_limit.restype = sz
            lib.tsi_index_share_layers.argtypes = [i32, i32, i32, ctypes.c_char_p, vp]
            lib.tsi_index_share_layers.restype = i32
            lib.tsi_topk_overlap.argtypes = [vp, vp, i32, i32, vp, vp, vp]
            lib.tsi_topk_overlap.restype = i32
            lib.tsi_indexer_topk_shard_workspace.argtypes = [i32] * 7
            lib.tsi_indexer_topk_shard_workspace.restype = sz
            lib.tsi_indexer_topk_shard.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32,
                                                   ctypes.c_int64, i32, i32, i32, i32, vp, vp,
                                                   vp, vp, sz, vp]
            lib.tsi_indexer_topk_shard.restype = i32
            lib.tsi_topk_merge.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
            lib.tsi_topk_merge.restype = i32
            lib.tsi_sparse_attn_group_lse.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, i32,
                                                      i32, i32, f32, vp, i32, vp, vp, vp, vp, sz,
                                                      vp]
            lib.tsi_sparse_attn_group_lse.restype = i32
            lib.tsi_index_kl.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp,
                                         i32, vp, vp, vp, vp, vp]
            lib.tsi_index_kl.restype = i32
            lib.tsi_selftest_wait_timeout.argtypes = [vp]
            lib.tsi_selftest_wait_timeout.restype = i32
            _lib = lib
    return _lib


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().tsi_launch_count())


def indexer_path(qk_dtype, H_I, d_I) -> int:
    """1: tensor-core kernel, 0: CUDA-core kernel, -1: unsupported."""
    return load().tsi_indexer_topk_path(qk_dtype, H_I, d_I)


def attn_path(H, Hkv, Dqk, Dv, v_from_k) -> int:
    """1: tensor-core kernel, 0: CUDA-core kernel, -1: unsupported."""
    return load().tsi_sparse_attn_path(H, Hkv, Dqk, Dv, int(bool(v_from_k)))


def last_error() -> str:
    return load().tsi_last_error().decode()


def _check(st):
    if st != OK:
        raise TSIError(st, last_error())


def _dtype_code(t):
    import torch

    code = {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3}.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


def _dev(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def indexer_topk_workspace(B, T, S, H_I, d_I, topk, qk_dtype, onchip=False,
                           two_pass=False) -> int:
    lib = load()
    fn = lib.tsi_indexer_topk_two_pass_workspace if two_pass else \
        lib.tsi_indexer_topk_onchip_workspace if onchip else lib.tsi_indexer_topk_workspace
    return fn(B, T, S, H_I, d_I, topk, qk_dtype)


def indexer_topk(qI, kI, w, topk, kv_len=None, idx=None, score=None, workspace=None,
                 stream=None, want_score=False, onchip=False, two_pass=False):
    """Top-k key positions of the lightning-indexer score (``tsi_indexer_topk``: no score
    leaves the scoring kernel; ``onchip`` calls ``tsi_indexer_topk_onchip``, the same;
    ``two_pass`` calls ``tsi_indexer_topk_two_pass``: the same results from scores stored
    for a second, selecting kernel).

    qI [B,T,H_I,d_I], kI [B,S,d_I] (f32/bf16/e4m3), w [B,T,H_I] (f32/bf16),
    kv_len [B] int32 or None.  Returns idx [B,T,topk] int32 (and score float32
    when ``want_score`` or ``score`` is given).
    """
    import torch

    B, T, H_I, d_I = qI.shape
    S = kI.shape[1]
    if idx is None:
        idx = torch.empty((B, T, topk), dtype=torch.int32, device=qI.device)
    if score is None and want_score:
        score = torch.empty((B, T, topk), dtype=torch.float32, device=qI.device)
    code = _dtype_code(qI)
    if _dtype_code(kI) != code:
        raise TypeError("qI and kI must share a dtype")
    need = indexer_topk_workspace(B, T, S, H_I, d_I, topk, code, onchip, two_pass)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=qI.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load()
    fn = lib.tsi_indexer_topk_two_pass if two_pass else \
        lib.tsi_indexer_topk_onchip if onchip else lib.tsi_indexer_topk
    _check(fn(
        _dev(qI, "qI"), _dev(kI, "kI"), _dev(w, "w"), code, _dtype_code(w), B, T, S, H_I, d_I,
        topk, _dev(kv_len, "kv_len"), _dev(idx, "idx"), _dev(score, "score"),
        _dev(workspace, "workspace"), ws_bytes, _stream_handle(stream)))
    return (idx, score) if score is not None else idx


def sparse_attn_workspace(B, T, S, H, Hkv, Dqk, Dv, topk) -> int:
    return load().tsi_sparse_attn_workspace(B, T, S, H, Hkv, Dqk, Dv, topk)


def sparse_attn_group(qs, ks, vs, idx, scale, kv_len=None, outs=None, workspace=None,
                      stream=None, Dv=None, want_lse=False, lses=None):
    """Sparse attention of every layer of one IndexShare group over the shared ``idx``.

    qs: list of Q [B,T,H,Dqk] bf16; ks: list of K [B,S,Hkv,Dqk] bf16; vs: list of
    V [B,S,Hkv,Dv] bf16, or None (value = first ``Dv`` dims of K).  Returns the
    list of O [B,T,H,Dv] bf16; with ``want_lse`` (or ``lses`` given) also the list of
    per-head log-partitions [B,T,H] fp32 (tsi_sparse_attn_group_lse).
    """
    import torch

    n = len(qs)
    B, T, H, Dqk = qs[0].shape
    S, Hkv = ks[0].shape[1], ks[0].shape[2]
    if vs is not None:
        Dv = vs[0].shape[-1]
    if Dv is None:
        raise ValueError("Dv is required when the value comes from the key")
    topk = idx.shape[-1]
    if outs is None:
        outs = [torch.empty((B, T, H, Dv), dtype=torch.bfloat16, device=qs[0].device)
                for _ in range(n)]
    need = sparse_attn_workspace(B, T, S, H, Hkv, Dqk, Dv, topk)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=qs[0].device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    for name, lst in (("q", qs), ("k", ks), ("out", outs)) + ((("v", vs),) if vs else ()):
        for t in lst:
            if t.dtype != torch.bfloat16:
                raise TypeError(f"{name} tensors must be bfloat16")
    P = ctypes.c_void_p * n
    qp = P(*[_dev(t, "q") for t in qs])
    kp = P(*[_dev(t, "k") for t in ks])
    vp = P(*[_dev(t, "v") for t in vs]) if vs is not None else None
    op = P(*[_dev(t, "out") for t in outs])
    if want_lse or lses is not None:
        if lses is None:
            lses = [torch.empty((B, T, H), dtype=torch.float32, device=qs[0].device)
                    for _ in range(n)]
        for t in lses:
            if t.dtype != torch.float32:
                raise TypeError("lse tensors must be float32")
        lp = P(*[_dev(t, "lse") for t in lses])
        _check(load().tsi_sparse_attn_group_lse(
            n, qp, kp, vp, B, T, S, H, Hkv, Dqk, Dv, float(scale), _dev(idx, "idx"), topk,
            _dev(kv_len, "kv_len"), op, lp, _dev(workspace, "workspace"), ws_bytes,
            _stream_handle(stream)))
        return outs, lses
    _check(load().tsi_sparse_attn_group(
        n, qp, kp, vp, B, T, S, H, Hkv, Dqk, Dv, float(scale), _dev(idx, "idx"), topk,
        _dev(kv_len, "kv_len"), op, _dev(workspace, "workspace"), ws_bytes,
        _stream_handle(stream)))
    return outs


def index_kl(qs, ks, lses, idx, score, scale, kv_len=None, want_grad=False, want_pbar=False,
             loss=None, grad=None, pbar=None, stream=None):
    """Group-centroid KL target of the Full layer's indexer over the group's layers
    (tsi_index_kl).

    qs: list of Q [B,T,64,576] bf16 (Full layer first); ks: list of latent caches
    [B,S,576] or [B,S,1,576] bf16; lses: the layers' [B,T,64] fp32 log-partitions
    (``sparse_attn_group(..., want_lse=True)``); idx [B,T,topk] int32 the shared index
    rows; score [B,T,topk] fp32 the indexer scores of those entries.  Returns loss [B,T]
    fp32, followed by grad and / or pbar [B,T,topk] fp32 when asked for.
    """
    import torch

    n = len(qs)
    B, T, H, Dqk = qs[0].shape
    S = ks[0].shape[1]
    topk = idx.shape[-1]
    dev = qs[0].device
    for name, lst, dt in (("q", qs, torch.bfloat16), ("k", ks, torch.bfloat16),
                          ("lse", lses, torch.float32)):
        if len(lst) != n:
            raise ValueError(f"{name}: {len(lst)} tensors for {n} layers")
        for t in lst:
            if t.dtype != dt:
                raise TypeError(f"{name} tensors must be {dt}")
    if score.dtype != torch.float32:
        raise TypeError("score must be float32")
    if loss is None:
        loss = torch.empty((B, T), dtype=torch.float32, device=dev)
    if want_grad and grad is None:
        grad = torch.empty((B, T, topk), dtype=torch.float32, device=dev)
    if want_pbar and pbar is None:
        pbar = torch.empty((B, T, topk), dtype=torch.float32, device=dev)
    P = ctypes.c_void_p * n
    qp = P(*[_dev(t, "q") for t in qs])
    kp = P(*[_dev(t, "k") for t in ks])
    lp = P(*[_dev(t, "lse") for t in lses])
    _check(load().tsi_index_kl(
        n, qp, kp, lp, B, T, S, H, Dqk, float(scale), _dev(idx, "idx"), _dev(score, "score"),
        topk, _dev(kv_len, "kv_len"), _dev(loss, "loss"), _dev(grad, "grad"),
        _dev(pbar, "pbar"), _stream_handle(stream)))
    out = (loss,)
    if want_grad or grad is not None:
        out += (grad,)
    if want_pbar or pbar is not None:
        out += (pbar,)
    return out[0] if len(out) == 1 else out


def selftest_wait_timeout(stream=None):
    """Launch the failure-path self-test (tsi_selftest_wait_timeout): a bounded device
    wait that runs out; device_status() afterwards raises TSIError(ERR_TIMEOUT)."""
    _check(load().tsi_selftest_wait_timeout(_stream_handle(stream)))


def device_status(stream=None):
    """Synchronize and read / clear the device error word (raises on a set flag)."""
    _check(load().tsi_device_status(_stream_handle(stream)))


def index_share_layers(n_layers, freq=4, skip_offset=0, pattern=None):
    """Anchor layer per layer of an IndexShare stack (tsi_index_share_layers): the layer
    whose indexer gives layer l its index rows, l itself for a Full layer."""
    out = (ctypes.c_int32 * max(n_layers, 1))()
    pat = None if pattern is None else pattern.encode()
    _check(load().tsi_index_share_layers(n_layers, freq, skip_offset, pat,
                                         ctypes.cast(out, ctypes.c_void_p)))
    return [int(out[i]) for i in range(n_layers)]


def topk_overlap(idx_a, idx_b, inter=None, card_a=None, stream=None):
    """Per-row |S_a ∩ S_b| and |S_a| of two [rows, topk] int32 index buffers
    (tsi_topk_overlap).  Returns (inter, card_a), int32 tensors of length rows."""
    import torch

    if idx_a.shape != idx_b.shape or idx_a.dtype != torch.int32 or idx_b.dtype != torch.int32:
        raise ValueError("idx_a and idx_b must be int32 tensors of one shape")
    topk = idx_a.shape[-1]
    rows = idx_a.numel() // topk if topk else 0
    if inter is None:
        inter = torch.empty(rows, dtype=torch.int32, device=idx_a.device)
    if card_a is None:
        card_a = torch.empty(rows, dtype=torch.int32, device=idx_a.device)
    _check(load().tsi_topk_overlap(_dev(idx_a, "idx_a"), _dev(idx_b, "idx_b"), rows, topk,
                                   _dev(inter, "inter"), _dev(card_a, "card_a"),
                                   _stream_handle(stream)))
    return inter, card_a


def indexer_topk_shard(qI, kI, w, topk, S_total, key_offset, kv_len=None, cand=None,
                       cand_cnt=None, workspace=None, stream=None):
    """One key shard of a context-parallel indexer (``tsi_indexer_topk_shard``).

    kI [B, S_shard, d_I] holds keys key_offset .. key_offset+S_shard-1 of a cache of
    S_total keys.  Returns (cand [B*T, topk] uint64 rank keys, unordered, with positions of
    the whole cache; cand_cnt [B*T] int32).
    """
    import torch

    B, T, H_I, d_I = qI.shape
    S = kI.shape[1]
    rows = B * T
    if cand is None:
        cand = torch.empty((rows, topk), dtype=torch.int64, device=qI.device)
    if cand_cnt is None:
        cand_cnt = torch.empty(rows, dtype=torch.int32, device=qI.device)
    code = _dtype_code(qI)
    if _dtype_code(kI) != code:
        raise TypeError("qI and kI must share a dtype")
    need = load().tsi_indexer_topk_shard_workspace(B, T, S, H_I, d_I, topk, code)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=qI.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().tsi_indexer_topk_shard(
        _dev(qI, "qI"), _dev(kI, "kI"), _dev(w, "w"), code, _dtype_code(w), B, T, S_total,
        key_offset, S, H_I, d_I, topk, _dev(kv_len, "kv_len"), _dev(cand, "cand"),
        _dev(cand_cnt, "cand_cnt"), _dev(workspace, "workspace"), ws_bytes,
        _stream_handle(stream)))
    return cand, cand_cnt


def topk_merge(cand, cand_cnt, idx=None, score=None, want_score=False, stream=None):
    """Top-k rows from candidate lists (``tsi_topk_merge``): cand [n_lists, rows, topk]
    uint64 rank keys, cand_cnt [n_lists, rows] int32.  Returns idx [rows, topk] int32 (and
    the scores with ``want_score``)."""
    import torch

    n_lists, rows, topk = cand.shape
    if idx is None:
        idx = torch.empty((rows, topk), dtype=torch.int32, device=cand.device)
    if score is None and want_score:
        score = torch.empty((rows, topk), dtype=torch.float32, device=cand.device)
    _check(load().tsi_topk_merge(_dev(cand, "cand"), _dev(cand_cnt, "cand_cnt"), n_lists, rows,
                                 topk, _dev(idx, "idx"), _dev(score, "score"),
                                 _stream_handle(stream)))
    return (idx, score) if score is not None else idx


def gather_candidates(cand, cand_cnt, group=None):
    """The exchange step of the context-parallel indexer: all-gather every rank's candidate
    lists into [world, rows, topk] / [world, rows] (torch.distributed: NCCL between GPUs)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    parts_c = [torch.empty_like(cand) for _ in range(world)]
    parts_n = [torch.empty_like(cand_cnt) for _ in range(world)]
    dist.all_gather(parts_c, cand.contiguous(), group=group)
    dist.all_gather(parts_n, cand_cnt.contiguous(), group=group)
    return torch.stack(parts_c), torch.stack(parts_n)


def cp_indexer_topk(qI, kI_shard, w, topk, S_total, key_offset, kv_len=None, group=None,
                    want_score=False):
    """Context-parallel indexer + top-k: this rank's shard, the all-gather of every rank's
    lists, the merge.  Every rank gets the rows of tsi_indexer_topk over the whole cache."""
    cand, cnt = indexer_topk_shard(qI, kI_shard, w, topk, S_total, key_offset, kv_len=kv_len)
    all_c, all_n = gather_candidates(cand, cnt, group)
    return topk_merge(all_c, all_n, want_score=want_score)
