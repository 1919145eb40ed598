"""Expected tensor set of a Qwen3 checkpoint, derived from the config dims.

TEST INFRASTRUCTURE (part of the oracle).  "M1 - Load the weights", section
"Deriving what should be there": globals embed_tokens [V,H], model.norm [H] and an
optional tied lm_head [V,H], plus the 11-tensor block repeated per layer with
weights stored [out, in].  Stored count sums every file tensor; the logical count
counts a tied lm_head once.
"""
from __future__ import annotations


def expected_tensors(vocab, hidden, n_layers, n_heads, n_kv_heads, head_dim, intermediate, tied_copy=True):
    H, V, d, I = hidden, vocab, head_dim, intermediate
    out = [("model.embed_tokens.weight", (V, H))]
    for l in range(n_layers):
        p = f"model.layers.{l}."
        out += [
            (p + "input_layernorm.weight", (H,)),
            (p + "self_attn.q_proj.weight", (n_heads * d, H)),
            (p + "self_attn.k_proj.weight", (n_kv_heads * d, H)),
            (p + "self_attn.v_proj.weight", (n_kv_heads * d, H)),
            (p + "self_attn.q_norm.weight", (d,)),
            (p + "self_attn.k_norm.weight", (d,)),
            (p + "self_attn.o_proj.weight", (H, n_heads * d)),
            (p + "post_attention_layernorm.weight", (H,)),
            (p + "mlp.gate_proj.weight", (I, H)),
            (p + "mlp.up_proj.weight", (I, H)),
            (p + "mlp.down_proj.weight", (H, I)),
        ]
    out.append(("model.norm.weight", (H,)))
    if tied_copy:
        out.append(("lm_head.weight", (V, H)))
    return out


def numel(shape) -> int:
    n = 1
    for s in shape:
        n *= s
    return n


def param_counts(tensors):
    """(stored, logical, embedding) parameter counts; a tied lm_head is counted once in logical."""
    stored = sum(numel(s) for _, s in tensors)
    emb = numel(dict(tensors)["model.embed_tokens.weight"])
    tied = sum(numel(s) for n, s in tensors if n == "lm_head.weight")
    return stored, stored - tied, emb


def kv_cache_bytes(n_layers, n_kv_heads, head_dim, ctx, bytes_per_elem) -> int:
    """K and V planes [L][Hkv][C][d]: 2 * L * Hkv * d * C * bytes."""
    return 2 * n_layers * n_kv_heads * head_dim * ctx * bytes_per_elem
