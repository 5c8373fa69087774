"""Named workload shapes for MiniMax Sparse Attention (MSA).

The talk pages describe the method (an index branch of 4 index query heads against
1 index key head, per-KV-head block top-k, exact attention over the chosen blocks)
but fix no sizes; the shapes below are the synthetic workloads this library is
measured and tested on.  Every config has 4 KV heads, 4 index query heads (one
per KV head) and one shared index key head.
"""
from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class MsaConfig:
    name: str
    mode: str            # "prefill" or "decode"
    dtype: str           # "f32" or "bf16"
    batch: int
    seq: int             # prefill: T tokens; decode: cache length L (query at L-1)
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    index_dim: int
    block_size: int
    top_k: int
    q_tile: int          # 64 for prefill selection tiles, 1 for decode
    seed: int
    input_scale: float   # multiplies the N(0,1) draws
    n_plants: int        # planted blocks per KV head
    plant_alpha: float   # strength of the planted index-key direction
    description: str = field(default="", compare=False)

    @property
    def seq_q(self) -> int:
        return self.seq if self.mode == "prefill" else 1

    @property
    def seq_k(self) -> int:
        return self.seq

    @property
    def group(self) -> int:
        return self.n_heads_q // self.n_heads_kv

    @property
    def n_tiles(self) -> int:
        return -(-self.seq_q // self.q_tile)

    @property
    def n_blocks(self) -> int:
        return -(-self.seq_k // self.block_size)

    def with_(self, **kw) -> "MsaConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": MsaConfig(
        "tiny", "prefill", "f32", 1, 1024, 16, 4, 64, 64, 64, 4, 64, 0, 1.0, 3, 3.0,
        "fp32 prefill T=1024, 16/4 heads, d=dI=64, block 64, k=4"),
    "p32k": MsaConfig(
        "p32k", "prefill", "bf16", 1, 32768, 32, 4, 128, 128, 128, 16, 64, 1,
        128 ** -0.5, 8, 2.0,
        "bf16 prefill T=32768, 32/4 heads, d=dI=128, block 128, k=16"),
    "p128k": MsaConfig(
        "p128k", "prefill", "bf16", 1, 131072, 64, 4, 128, 128, 128, 32, 64, 2,
        128 ** -0.5, 16, 2.0,
        "bf16 prefill T=131072, 64/4 heads, d=dI=128, block 128, k=32"),
    "d1m": MsaConfig(
        "d1m", "decode", "bf16", 8, 1 << 20, 64, 4, 128, 128, 128, 64, 1, 3, 1.0, 32, 2.0,
        "bf16 decode, batch 8 x 1,048,576-token cache, 64/4 heads, block 128, k=64"),
    "p1m": MsaConfig(
        "p1m", "prefill", "bf16", 1, 1 << 20, 64, 4, 128, 128, 128, 64, 64, 4, 1.0, 64, 2.0,
        "bf16 prefill T=1,048,576, 64/4 heads, d=dI=128, block 128, k=64"),
}


def get_config(name: str) -> MsaConfig:
    return CONFIGS[name]
