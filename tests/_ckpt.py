"""Writers of synthetic safetensors / SLM2 checkpoint bytes for the loader tests (test helper).

Layout ("M1 - Load the weights", section "The safetensors format"): [u64 little-endian N]
[N bytes of JSON][blob]; the header is padded with spaces so the blob starts on an 8-byte
boundary, and every tensor starts on an 8-byte boundary of the file.
"""
from __future__ import annotations

import json
import struct

import numpy as np

Q8_BLOCK = 34  # fp16 scale + 32 int8 codes


def q8_blocks(codes: np.ndarray, scales_bits: np.ndarray) -> bytes:
    """SLM2 Q8_0 bytes of a matrix from int8 codes [out, in] and fp16 scale bits [out, in/32]."""
    c = np.ascontiguousarray(codes, dtype=np.int8).reshape(-1, 32)
    s = np.ascontiguousarray(scales_bits, dtype=np.uint16).reshape(-1)
    out = np.empty((c.shape[0], Q8_BLOCK), np.uint8)
    out[:, :2] = s.view(np.uint8).reshape(-1, 2)
    out[:, 2:] = c.view(np.uint8)
    return out.tobytes()


def build(entries, metadata=None, header_text=None, align=True, size_only=False):
    """entries: [(name, dtype, shape, payload bytes or byte count)] -> file bytes (or
    (prefix + header bytes, file size) when size_only).  header_text overrides the JSON."""
    header = {}
    if metadata is not None:
        header["__metadata__"] = metadata
    off = 0
    for name, dt, shape, payload in entries:
        n = payload if isinstance(payload, int) else len(payload)
        if align and off % 8:
            off += 8 - off % 8
        header[name] = {"dtype": dt, "shape": list(shape), "data_offsets": [off, off + n]}
        off += n
    text = header_text if header_text is not None else json.dumps(header, separators=(",", ":"))
    raw = text.encode()
    if align and (8 + len(raw)) % 8:
        raw += b" " * (8 - (8 + len(raw)) % 8)
    prefix = struct.pack("<Q", len(raw)) + raw
    if size_only:
        return prefix, len(prefix) + off
    blob = bytearray(off)
    for name, dt, shape, payload in entries:
        if isinstance(payload, int):
            continue
        b, e = header[name]["data_offsets"]
        blob[b:e] = payload
    return prefix + bytes(blob)


def model_entries(wl, w, q8=False, f32_norms=False, head=True, head_bytes=None):
    """Checkpoint entries of a seeded model (qw_inputs.make_weights) under the Qwen3 names."""
    def vec(a):
        if f32_norms:
            return "F32", (np.asarray(a, np.uint32) << 16).astype(np.uint32).tobytes()
        return "BF16", np.ascontiguousarray(a, np.uint16).tobytes()

    out = [("model.embed_tokens.weight", "BF16", w["embed"].shape, w["embed"].tobytes())]
    names = {"q": "self_attn.q_proj", "k": "self_attn.k_proj", "v": "self_attn.v_proj", "o": "self_attn.o_proj",
             "gate": "mlp.gate_proj", "up": "mlp.up_proj", "down": "mlp.down_proj"}
    for l, lw in enumerate(w["layers"]):
        p = f"model.layers.{l}."
        for key, nm in (("input_norm", "input_layernorm"), ("post_norm", "post_attention_layernorm"),
                        ("q_norm", "self_attn.q_norm"), ("k_norm", "self_attn.k_norm")):
            dt, b = vec(lw[key])
            out.append((p + nm + ".weight", dt, lw[key].shape, b))
        for m, nm in names.items():
            if q8:
                out.append((p + nm + ".weight", "Q8_0", lw[m].shape, q8_blocks(lw[m + "_q8"], lw[m + "_s"])))
            else:
                out.append((p + nm + ".weight", "BF16", lw[m].shape, lw[m].tobytes()))
    dt, b = vec(w["final_norm"])
    out.append(("model.norm.weight", dt, w["final_norm"].shape, b))
    if head:
        out.append(("lm_head.weight", "BF16", w["embed"].shape, head_bytes or w["embed"].tobytes()))
    return out
