"""The five synthetic workloads of the DSA indexer + top-k + IndexShare path.

Shapes follow the pages' workloads (a 30B and a 744B GLM model at 100K-1M
context, "GLM-5.2 技术报告速览" §IndexShare; MLA 576-d latent with d_c=512,
d_r=64, H=64, "GLM 5.2: Built for Long Horizon Tasks" discussion §3).  No
dataset or weights are involved: every tensor is drawn from a seeded
distribution (see ``gen.py``).
"""
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Config:
    id: int
    name: str
    # batch / query rows / cached keys per sequence
    B: int
    T: int
    S: int
    # lightning indexer
    H_I: int
    d_I: int
    topk: int
    qk_dtype: str  # 'f32' | 'bf16' | 'e4m3'
    w_dtype: str  # 'f32' | 'bf16'
    qk_dist: str  # 'int4' | 'int8' | 'normal_dI' | 'normal'
    w_dist: str  # 'int03' | 'pow2' | 'uniform'
    # sparse attention (n_layers = 0: indexer + top-k only)
    n_layers: int
    H: int = 64
    Hkv: int = 1
    Dqk: int = 576
    Dv: int = 512
    v_from_k: bool = True  # MQA latent: value = first Dv dims of the key row
    group: int = 4  # IndexShare: 1 Full + (group-1) Shared layers

    @property
    def n_groups(self) -> int:
        return max(1, self.n_layers // self.group) if self.n_layers else 1

    @property
    def scale(self) -> float:
        return 1.0 / (self.Dqk ** 0.5)

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


CONFIGS = {
    1: Config(1, "tiny-group-L1024", B=1, T=1024, S=1024, H_I=4, d_I=32, topk=64,
              qk_dtype="f32", w_dtype="f32", qk_dist="int4", w_dist="int03",
              n_layers=4, H=4, Hkv=4, Dqk=64, Dv=64, v_from_k=False),
    2: Config(2, "indexer-only-L8192-e4m3-int", B=1, T=8192, S=8192, H_I=64, d_I=128,
              topk=2048, qk_dtype="e4m3", w_dtype="bf16", qk_dist="int8", w_dist="pow2",
              n_layers=0),
    3: Config(3, "group-L32768-bf16", B=1, T=32768, S=32768, H_I=64, d_I=128, topk=2048,
              qk_dtype="bf16", w_dtype="bf16", qk_dist="normal_dI", w_dist="uniform",
              n_layers=4),
    4: Config(4, "prefill-L131072-16layers-e4m3", B=1, T=131072, S=131072, H_I=64, d_I=128,
              topk=2048, qk_dtype="e4m3", w_dtype="bf16", qk_dist="normal", w_dist="uniform",
              n_layers=16),
    5: Config(5, "decode-B8-S131072", B=8, T=1, S=131072, H_I=64, d_I=128, topk=2048,
              qk_dtype="e4m3", w_dtype="bf16", qk_dist="normal", w_dist="uniform",
              n_layers=4),
}


def get_config(i: int) -> Config:
    return CONFIGS[i]
