"""Seeded synthetic inputs (torch generators only; no arithmetic of the method).

Seed rule: ``seed = 0x7351 + 1000*config + 10*layer + tensor_id`` with tensor
ids qI=0, kI=1, w=2, Q=3, K/latent=4, V=5.  Indexer tensors of a group use the
layer index of that group's Full layer.

Distributions (the workloads' recipes):
  int4      uniform integers in [-4, 4]
  int8      uniform integers in [-8, 8] (exact in e4m3)
  normal_dI N(0, 1/d_I)
  normal    N(0, 1)
  int03     uniform integers in [0, 3]
  pow2      2^U{-4..0}
  uniform   U(0, 1)
Casting to the stored dtype rounds to nearest even (torch's casts).
"""
import torch

TORCH_DTYPE = {
    "f32": torch.float32,
    "bf16": torch.bfloat16,
    "e4m3": torch.float8_e4m3fn,
}

TENSOR_ID = {"qI": 0, "kI": 1, "w": 2, "Q": 3, "K": 4, "V": 5}


def seed_for(cfg_id: int, layer: int, tensor: str) -> int:
    return 0x7351 + 1000 * cfg_id + 10 * layer + TENSOR_ID[tensor]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw(shape, dist: str, dtype: str, seed: int, device, d_I: int = 128,
         chunk_elems: int = 1 << 28) -> torch.Tensor:
    """Draw a tensor of ``shape`` from ``dist`` and store it as ``dtype``.

    Large tensors are drawn in chunks along the first dimension so that the
    float32 staging buffer stays small.
    """
    out = torch.empty(shape, dtype=TORCH_DTYPE[dtype], device=device)
    g = _gen(seed, device)
    flat = out.view(-1)
    n = flat.numel()
    for lo in range(0, n, chunk_elems):
        hi = min(n, lo + chunk_elems)
        m = hi - lo
        if dist == "int4":
            x = torch.randint(-4, 5, (m,), generator=g, device=device).to(torch.float32)
        elif dist == "int8":
            x = torch.randint(-8, 9, (m,), generator=g, device=device).to(torch.float32)
        elif dist == "int03":
            x = torch.randint(0, 4, (m,), generator=g, device=device).to(torch.float32)
        elif dist == "pow2":
            e = torch.randint(-4, 1, (m,), generator=g, device=device).to(torch.float32)
            x = torch.exp2(e)
        elif dist == "uniform":
            x = torch.rand((m,), generator=g, device=device, dtype=torch.float32)
        elif dist == "normal":
            x = torch.randn((m,), generator=g, device=device, dtype=torch.float32)
        elif dist == "normal_dI":
            x = torch.randn((m,), generator=g, device=device, dtype=torch.float32)
            x.mul_((1.0 / d_I) ** 0.5)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        flat[lo:hi] = x.to(out.dtype)
        del x
    return out


def make_indexer_inputs(cfg, group: int = 0, device="cpu"):
    """qI [B,T,H_I,d_I], kI [B,S,d_I], w [B,T,H_I] for one IndexShare group."""
    layer = group * cfg.group
    qI = draw((cfg.B, cfg.T, cfg.H_I, cfg.d_I), cfg.qk_dist, cfg.qk_dtype,
              seed_for(cfg.id, layer, "qI"), device, cfg.d_I)
    kI = draw((cfg.B, cfg.S, cfg.d_I), cfg.qk_dist, cfg.qk_dtype,
              seed_for(cfg.id, layer, "kI"), device, cfg.d_I)
    w = draw((cfg.B, cfg.T, cfg.H_I), cfg.w_dist, cfg.w_dtype,
             seed_for(cfg.id, layer, "w"), device, cfg.d_I)
    return qI, kI, w


def make_attn_inputs(cfg, layer: int, device="cpu", with_q: bool = True):
    """Q [B,T,H,Dqk] bf16, K [B,S,Hkv,Dqk] bf16, V [B,S,Hkv,Dv] bf16 or None.

    For the MQA latent (v_from_k) the value is the first Dv dims of K, so no
    separate V tensor is drawn.
    """
    Q = None
    if with_q:
        Q = draw((cfg.B, cfg.T, cfg.H, cfg.Dqk), "normal", "bf16",
                 seed_for(cfg.id, layer, "Q"), device)
    K = draw((cfg.B, cfg.S, cfg.Hkv, cfg.Dqk), "normal", "bf16",
             seed_for(cfg.id, layer, "K"), device)
    V = None
    if not cfg.v_from_k:
        V = draw((cfg.B, cfg.S, cfg.Hkv, cfg.Dv), "normal", "bf16",
                 seed_for(cfg.id, layer, "V"), device)
    return Q, K, V
