"""Model shapes of the five synthetic workloads and their input recipe.

Shapes follow the pages' models: the 2B dense coder of the Kog post
("3k tokens/s per request", section on the 2B example at FP16) and the
Ling-3.0-flash MoE of the DGX Spark article (section "model and baseline
configuration": hidden 2560, 512 routed experts top-8 plus 1 shared,
moe_intermediate 768, vocabulary 157184, 42 layers). Attention in every
config is GQA with head dim 128 (the MoE stack replaces Ling's KDA/MLA layers
by GQA 20/4).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_q: int = 0            # query heads (0: no attention block)
    n_kv: int = 0           # key/value heads
    head_dim: int = 128
    ffn: int = 0            # dense SwiGLU width (0: no dense FFN)
    n_experts: int = 0      # routed experts (0: no MoE FFN)
    top_k: int = 0
    moe_inter: int = 0
    n_shared: int = 0
    vocab: int = 0          # 0: no LM head
    kv_prefill: int = 0     # cached positions before the first decode step
    lm_head_dtype: str = "bf16"   # "bf16" | "fp8"
    kv_dtype: str = "bf16"        # "bf16" | "fp8" (e4m3 codes with a scale per layer, K/V and kv head)
    attn_window: int = 0          # > 0: every query attends to the last attn_window positions only
    embedding: bool = False       # True: the step starts from E[token]; False: from a given hidden
    final_norm: bool = True       # RMSNorm before the LM head
    steps: int = 1                # greedy decode steps of the workload
    verify: int = 1               # tokens per verify window (1 = plain decode)
    rms_eps: float = 1e-6
    rope_base: float = 1e4
    w_std: float = 0.02

    @property
    def qkv_rows(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    @property
    def attn(self) -> bool:
        return self.n_q > 0

    @property
    def moe(self) -> bool:
        return self.n_experts > 0

    def with_(self, **kw) -> "ModelShape":
        return replace(self, **kw)


def dense_layer_shape() -> ModelShape:
    """One dense decoder layer + LM head, batch 1 (hidden 1024, GQA 8/2, FFN 2816, vocab 32000, 256 cached)."""
    return ModelShape("dense_layer_lmhead", n_layers=1, hidden=1024, n_q=8, n_kv=2, ffn=2816,
                      vocab=32000, kv_prefill=256)


def dense_2b_shape() -> ModelShape:
    """2B-class dense decoder: 28 layers, hidden 2560, GQA 20/4, FFN 6912, vocab 32768, 4096 cached, 256 steps."""
    return ModelShape("dense_2b", n_layers=28, hidden=2560, n_q=20, n_kv=4, ffn=6912, vocab=32768,
                      kv_prefill=4096, embedding=True, steps=256)


def moe_layer_shape(verify: int = 1) -> ModelShape:
    """One MoE FFN block (pre-norm + residual): 512 routed experts top-8 + 1 shared, intermediate 768, MXFP4."""
    return ModelShape("moe_layer", n_layers=1, hidden=2560, n_experts=512, top_k=8, moe_inter=768,
                      n_shared=1, verify=verify)


def lm_head_shape(dtype: str = "bf16", verify: int = 1) -> ModelShape:
    """Bare LM-head GEMV + argmax: hidden 2560 to vocab 157184, bf16 or FP8-e4m3 per-row scale."""
    return ModelShape("lm_head", n_layers=0, hidden=2560, vocab=157184, lm_head_dtype=dtype,
                      final_norm=False, verify=verify)


def moe_stack_shape(verify: int = 1) -> ModelShape:
    """42-layer MoE stack: GQA 20/4, 32768 cached, MoE 512 top-8 + shared (MXFP4), FP8 head 157184x2560."""
    return ModelShape("moe_stack", n_layers=42, hidden=2560, n_q=20, n_kv=4, n_experts=512, top_k=8,
                      moe_inter=768, n_shared=1, vocab=157184, kv_prefill=32768, lm_head_dtype="fp8",
                      embedding=True, steps=512, verify=verify)


CONFIGS = {
    "dense_layer_lmhead": dense_layer_shape,
    "dense_2b": dense_2b_shape,
    "moe_layer": moe_layer_shape,
    "lm_head": lm_head_shape,
    "moe_stack": moe_stack_shape,
}
