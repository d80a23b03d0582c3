"""Decoder shapes of the synthetic workloads.

The three shapes are those of the workloads the pages measure on: a tiny
random decoder for exhaustive checks, Qwen2.5-1.5B (the model behind every
28-field and 255-choice number on the pages) and Qwen2.5-7B for batched
serving.
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    rms_eps: float
    rope_theta: float
    tied_embedding: bool
    dtype: str          # "f32" or "bf16": the precision the weights are drawn in

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


_SHAPES = {
    # 2 layers, d=64, 4 query / 2 KV heads of dim 16, SwiGLU 172, vocab 512, fp32.
    "tiny": ModelConfig("tiny", 2, 64, 4, 2, 16, 172, 512, 1e-6, 1e4, True, "f32"),
    # 2 layers, d=768, 6 query / 2 KV heads of dim 128 (the production head
    # size), SwiGLU 1024, vocab 512, fp32: small enough for exhaustive oracle
    # checks of the head-dim-128 kernels.
    "tiny-h128": ModelConfig("tiny-h128", 2, 768, 6, 2, 128, 1024, 512, 1e-6, 1e4, True, "f32"),
    # Qwen2.5-1.5B shape, bf16, tied embedding.
    "1.5b": ModelConfig("1.5b", 28, 1536, 12, 2, 128, 8960, 151936, 1e-6, 1e6, True, "bf16"),
    # Qwen2.5-7B shape, bf16, untied LM head.
    "7b": ModelConfig("7b", 28, 3584, 28, 4, 128, 18944, 152064, 1e-6, 1e6, False, "bf16"),
}

# Which decoder each numbered workload runs on (1-based, in the order the
# workloads are listed: tiny reference, 28-field triage, 255-choice router,
# long document, batched serving).
CONFIG_MODEL = {1: "tiny", 2: "1.5b", 3: "1.5b", 4: "1.5b", 5: "7b"}


def model_config(name: str) -> ModelConfig:
    return _SHAPES[name]
