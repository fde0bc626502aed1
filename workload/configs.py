"""The five seeded synthetic workloads of the FASA decode step.

Each workload is named by what it is and carries its sizes.  The shapes are
those of the attention layers the FASA pages evaluate on (Llama-3-8B,
Qwen2.5-7B, Mistral-7B: 128-dim heads with grouped KV heads), with synthetic
values standing in for model activations: pre-RoPE q/k ~ N(0, 1) with a few
"outlier" frequency chunks scaled x8 per KV head, v ~ N(0, 1).
"""

from dataclasses import dataclass, field
from typing import Optional


@dataclass(frozen=True)
class Config:
    name: str
    dtype: str            # "f32" or "bf16": storage type of q, K, V, K_dom
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rope_theta: float
    context: int          # cache capacity T_max (and the length when not ragged)
    n_tip: int            # dominant FCs per KV head
    budget: int           # N_fac, the token budget of the top-k
    n_outlier: int        # outlier FCs per KV head (scaled x8 in pre-RoPE q/k)
    layers: int = 1
    ragged: Optional[tuple] = None   # (lo, hi): per-sequence length ~ U{lo..hi}
    seed: int = 0
    # per-KV-head dominant-FC counts (each <= n_tip, the table's row length)
    n_tip_per_head: Optional[tuple] = None
    # per-layer token budgets (each <= budget, which sizes the workspace)
    budget_per_layer: Optional[tuple] = None

    def head_n_tip(self, h: int) -> int:
        return self.n_tip if self.n_tip_per_head is None else self.n_tip_per_head[h]

    def layer_budget(self, layer: int) -> int:
        return self.budget if self.budget_per_layer is None else self.budget_per_layer[layer]

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_fc(self) -> int:
        return self.head_dim // 2

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_(self, **kw) -> "Config":
        d = dict(self.__dict__)
        d.update(kw)
        return Config(**d)


def _seed(i: int) -> int:
    return 0xFA5A0000 + i


CONFIGS = {
    # Parity-scale case: fp32, one layer, GQA 2, 64-dim heads.
    "tiny_fp32_ctx1k": Config(
        name="tiny_fp32_ctx1k", dtype="f32", batch=1, n_q_heads=4, n_kv_heads=2,
        head_dim=64, rope_theta=1e4, context=1024, n_tip=8, budget=64,
        n_outlier=2, seed=_seed(1)),
    # Llama-3-8B-shaped decode attention at 32K context (the headline).
    "llama3_8b_ctx32k": Config(
        name="llama3_8b_ctx32k", dtype="bf16", batch=1, n_q_heads=32, n_kv_heads=8,
        head_dim=128, rope_theta=5e5, context=32768, n_tip=16, budget=256,
        n_outlier=4, seed=_seed(2)),
    # Qwen2.5-7B-shaped long-CoT decode: batch 8, GQA 7, budget 18.9% of 16K.
    "qwen25_7b_b8_ctx16k": Config(
        name="qwen25_7b_b8_ctx16k", dtype="bf16", batch=8, n_q_heads=28, n_kv_heads=4,
        head_dim=128, rope_theta=1e6, context=16384, n_tip=16, budget=3097,
        n_outlier=4, seed=_seed(3)),
    # Mistral-7B-shaped 32-layer decode step, batch 32, ragged 4K..32K.
    "mistral_7b_l32_b32_ragged": Config(
        name="mistral_7b_l32_b32_ragged", dtype="bf16", batch=32, n_q_heads=32,
        n_kv_heads=8, head_dim=128, rope_theta=1e6, context=32768, n_tip=12,
        budget=256, n_outlier=4, layers=32, ragged=(4096, 32768), seed=_seed(4)),
    # Llama-3-8B-shaped 128K stress, batch 4.
    "llama3_8b_b4_ctx128k": Config(
        name="llama3_8b_b4_ctx128k", dtype="bf16", batch=4, n_q_heads=32, n_kv_heads=8,
        head_dim=128, rope_theta=5e5, context=131072, n_tip=8, budget=2048,
        n_outlier=4, seed=_seed(5)),
    # Variants the pages describe (per-head N_tip, the Oracle upper bound,
    # per-layer budgets), each a first-class workload of its own:
    # Llama-3-8B 32K with per-KV-head N_tip of 4..28 (mean 16, as uniform 16).
    "llama3_8b_ctx32k_ragged_ntip": Config(
        name="llama3_8b_ctx32k_ragged_ntip", dtype="bf16", batch=1, n_q_heads=32, n_kv_heads=8,
        head_dim=128, rope_theta=5e5, context=32768, n_tip=28, budget=256,
        n_outlier=4, seed=_seed(2), n_tip_per_head=(4, 8, 12, 16, 16, 20, 24, 28)),
    # Llama-3-8B 32K with every FC dominant: TIP scores are the full logits
    # (the pages' "Oracle" selection, run through the same kernels).
    "llama3_8b_ctx32k_oraclek": Config(
        name="llama3_8b_ctx32k_oraclek", dtype="bf16", batch=1, n_q_heads=32, n_kv_heads=8,
        head_dim=128, rope_theta=5e5, context=32768, n_tip=64, budget=256,
        n_outlier=4, seed=_seed(2)),
    # The Mistral-7B 32-layer step with pyramid budgets: 384 at the first
    # layer down to 128 at the last (mean 256, as the uniform workload).
    "mistral_7b_l32_b32_pyramid": Config(
        name="mistral_7b_l32_b32_pyramid", dtype="bf16", batch=32, n_q_heads=32,
        n_kv_heads=8, head_dim=128, rope_theta=1e6, context=32768, n_tip=12,
        budget=384, n_outlier=4, layers=32, ragged=(4096, 32768), seed=_seed(4),
        budget_per_layer=tuple(int(round(384 - 256 * l / 31)) for l in range(32))),
}

# Order used by tests: the pages' workloads from smallest to largest.
CONFIG_ORDER = ["tiny_fp32_ctx1k", "llama3_8b_ctx32k", "qwen25_7b_b8_ctx16k",
                "mistral_7b_l32_b32_ragged", "llama3_8b_b4_ctx128k"]


def get_config(name: str) -> Config:
    return CONFIGS[name]
