"""Seeded synthetic inputs for the batch-one Qwen3 decoder (weights, prompts, K/V fills).

This package is shared by the CPU oracle and the CUDA path *as input data only*: it
draws random numbers and lays them out as tensors, and holds none of the decoder's
arithmetic.  The generator is PCG32 as frozen in "Portable WebAssembly Runtime
Architecture for TinyRustLM", section "Deterministic sampling contract"; normal
deviates come from Box-Muller on consecutive 24-bit uniforms.

Tensor layout follows "M1 - Load the weights" (the 11-tensor block shape table):
every matrix is stored [out, in] row-major; the lm_head is tied to the embedding.
Stream ids are the tensor's index in the checkpoint order (embed = 0, then 11 per
layer, then the final norm), the seed is the workload's seed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import WORKLOADS, Workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None
_LOCK = threading.Lock()

LAYER_TENSORS = ("input_norm", "q", "k", "v", "q_norm", "k_norm", "o", "post_norm", "gate", "up", "down")
MATRICES = ("q", "k", "v", "o", "gate", "up", "down")
NORMS = ("input_norm", "q_norm", "k_norm", "post_norm")
KV_STREAM_K = 1 << 20
KV_STREAM_V = (1 << 20) + 1
PROMPT_STREAM = 1 << 21


def build(force: bool = False) -> str:
    """Compile qwgen.c into qw_inputs/_build/libqwgen.so (plain C, -O2)."""
    out_dir = os.path.join(_HERE, "_build")
    so = os.path.join(out_dir, "libqwgen.so")
    src = os.path.join(_HERE, "qwgen.c")
    if not force and os.path.exists(so) and os.path.getmtime(so) >= os.path.getmtime(src):
        return so
    os.makedirs(out_dir, exist_ok=True)
    tmp = so + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, so)
    return so


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            lib.qwgen_normal_bf16.argtypes = [u16p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                              ctypes.c_double, ctypes.c_double, ctypes.c_int]
            lib.qwgen_pcg32_words.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int64, ctypes.c_uint64,
                                              ctypes.c_uint64, ctypes.c_uint64]
            lib.qwgen_tokens.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int64, ctypes.c_uint64,
                                         ctypes.c_uint64, ctypes.c_int32]
            lib.qwgen_quantize_q8_g32.argtypes = [u16p, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.POINTER(ctypes.c_int8), u16p]
            lib.qwgen_f32_to_f16.argtypes = [ctypes.c_float]
            lib.qwgen_f32_to_f16.restype = ctypes.c_uint16
            lib.qwgen_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.qwgen_f32_to_bf16.restype = ctypes.c_uint16
            _LIB = lib
    return _LIB


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def pcg32_words(n: int, seed: int, stream: int, skip: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    _lib().qwgen_pcg32_words(_ptr(out, ctypes.c_uint32), n, seed, stream, skip)
    return out


def normal_bf16(shape, seed: int, stream: int, std: float, mean: float = 0.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, std^2) deviates, C-contiguous."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if n:
        _lib().qwgen_normal_bf16(_ptr(out, ctypes.c_uint16), n, seed, stream, mean, std, threads())
    return out.reshape(shape)


def tokens(n: int, seed: int, vocab: int, stream: int = PROMPT_STREAM) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _lib().qwgen_tokens(_ptr(out, ctypes.c_int32), n, seed, stream, vocab)
    return out


def quantize_q8_g32(w_bf16: np.ndarray):
    """Symmetric int8 codes [rows, cols] and fp16 scales [rows, cols/32] (as uint16 bits)."""
    rows, cols = w_bf16.shape
    if cols % 32:
        raise ValueError("cols must be a multiple of 32")
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    q = np.empty((rows, cols), dtype=np.int8)
    s = np.empty((rows, cols // 32), dtype=np.uint16)
    _lib().qwgen_quantize_q8_g32(_ptr(w, ctypes.c_uint16), rows, cols, _ptr(q, ctypes.c_int8),
                                 _ptr(s, ctypes.c_uint16))
    return q, s


def f32_to_f16_bits(x: float) -> int:
    return int(_lib().qwgen_f32_to_f16(ctypes.c_float(x)))


def f32_to_bf16_bits(x: float) -> int:
    return int(_lib().qwgen_f32_to_bf16(ctypes.c_float(x)))


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a data-format conversion)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def tensor_shapes(wl: Workload):
    """[out, in] shapes of one decoder block, in checkpoint order."""
    H, d, Hq, Hkv, I = wl.hidden, wl.head_dim, wl.n_heads, wl.n_kv_heads, wl.intermediate
    return {
        "input_norm": (H,), "q": (Hq * d, H), "k": (Hkv * d, H), "v": (Hkv * d, H),
        "q_norm": (d,), "k_norm": (d,), "o": (H, Hq * d), "post_norm": (H,),
        "gate": (I, H), "up": (I, H), "down": (H, I),
    }


def make_weights(wl: Workload, weight_std: float = 0.02, norm_std: float = 0.01):
    """Random-init weights of the workload's architecture.

    Returns {"embed": u16[V,H], "final_norm": u16[H], "layers": [dict]}; each layer dict
    holds bf16 arrays for every tensor and, for the int8 format, "<m>_q8" (int8 [out,in])
    and "<m>_s" (fp16 bits [out,in/32]) for the seven matrices.
    """
    seed = wl.seed
    shapes = tensor_shapes(wl)
    embed = normal_bf16((wl.vocab, wl.hidden), seed, 0, weight_std)
    layers = []
    for l in range(wl.n_layers):
        layer = {}
        for j, name in enumerate(LAYER_TENSORS):
            stream = 1 + 11 * l + j
            if name in NORMS:
                layer[name] = normal_bf16(shapes[name], seed, stream, norm_std, mean=1.0)
            else:
                layer[name] = normal_bf16(shapes[name], seed, stream, weight_std)
        if wl.weight_format == "int8_g32":
            for m in MATRICES:
                layer[m + "_q8"], layer[m + "_s"] = quantize_q8_g32(layer[m])
        layers.append(layer)
    final_norm = normal_bf16((wl.hidden,), seed, 1 + 11 * wl.n_layers, norm_std, mean=1.0)
    return {"embed": embed, "final_norm": final_norm, "layers": layers}


def prompt(wl: Workload) -> np.ndarray:
    return tokens(wl.prompt_len, wl.seed, wl.vocab)


def first_decode_token(wl: Workload) -> int:
    """Input token for workloads that start from an imported K/V cache instead of a prompt."""
    return int(tokens(1, wl.seed, wl.vocab, stream=PROMPT_STREAM + 1)[0])


def kv_fill(wl: Workload, n_pos: int, std: float = 1.0):
    """bf16 K and V planes [L][Hkv][n_pos][d] ~ N(0, std^2)."""
    shape = (wl.n_layers, wl.n_kv_heads, n_pos, wl.head_dim)
    return (normal_bf16(shape, wl.seed, KV_STREAM_K, std), normal_bf16(shape, wl.seed, KV_STREAM_V, std))
