"""The five synthetic workloads of the batch-one Qwen3-0.6B-shape decoder.

Dimensions are the public Qwen3-0.6B configuration as printed in "M1 - Load the
weights" (dimension table: V 151936, H 1024, L 28, d 128, 16 query / 8 KV heads,
I 3072) and "Scalar-Native Qwen3 Reference Runtime" section 2 (RMSNorm eps 1e-6,
tied embeddings).  RoPE base theta = 1e6 is the Qwen3 value.  All weights are
random-init (no checkpoint), K/V fills and prompts are seeded uniform/normal draws.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n_layers: int = 28
    hidden: int = 1024
    n_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    intermediate: int = 3072
    vocab: int = 151936
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    weight_format: str = "bf16"      # "bf16" | "int8_g32"
    act_format: str = "f32"          # "f32" | "q8": projection inputs quantized per 32-block (int8 weights)
    kv_format: str = "f32"           # K/V cache element type: "f32" (the reference's) | "bf16"
    prompt_len: int = 0              # prefill tokens
    kv_prefill: int = 0              # positions imported into the K/V cache instead of a prompt
    decode_steps: int = 0
    notes: str = field(default="", compare=False)

    @property
    def max_ctx(self) -> int:
        return self.kv_prefill + self.prompt_len + self.decode_steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        "tiny", seed=1, n_layers=2, vocab=8192, prompt_len=8, decode_steps=8,
        notes="2 layers, vocab 8192; 8-token prompt + 8 greedy decode steps"),
    "qwen3_0p6b_decode": Workload(
        "qwen3_0p6b_decode", seed=2, prompt_len=128, decode_steps=384,
        notes="full 0.6B shape; 128-token prompt + 384 greedy decode steps"),
    "qwen3_0p6b_prefill2048": Workload(
        "qwen3_0p6b_prefill2048", seed=3, prompt_len=2048, decode_steps=16,
        notes="full 0.6B shape; 2048-token prompt + 16 decode steps"),
    "qwen3_0p6b_ctx32k": Workload(
        "qwen3_0p6b_ctx32k", seed=4, kv_prefill=32768, decode_steps=64, kv_format="bf16",
        notes="full 0.6B shape; K/V cache pre-filled to 32768 positions with N(0,1) bf16, 64 decode steps"),
    "qwen3_0p6b_int8": Workload(
        "qwen3_0p6b_int8", seed=5, weight_format="int8_g32", prompt_len=256, decode_steps=768,
        notes="full 0.6B shape, int8 group-32 projections/MLP; 256-token prompt + 768 decode steps"),
}
