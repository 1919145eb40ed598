"""CPU oracle for the batch-one Qwen3 decoder forward (plain fp32, no FMA).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the bench's
``cpu_baseline`` leg (and its ``--impl reference`` arm) may import this package.
The product path never loads it; it shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (see its header for the equations and the
readings of the pages where their display equations were lost).  This module is
argument marshalling plus the shape-set check of ``shapes.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None
_LOCK = threading.Lock()

OK = 0
INVALID_ARGUMENT = 1
UNSUPPORTED_QUANTIZATION = 12
UNSUPPORTED_SHAPE = 13
CONTEXT_EXCEEDED = 14
NUMERICAL_FAILURE = 18

W_BF16 = 0
W_INT8_G32 = 1
W_Q8Q8 = 2
MATRICES = ("q", "k", "v", "o", "gate", "up", "down")


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


class _Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("max_ctx", ctypes.c_int32), ("weight_format", ctypes.c_int32), ("nthreads", ctypes.c_int32)]


class _Layer(ctypes.Structure):
    _fields_ = [("input_norm", ctypes.c_void_p), ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("post_norm", ctypes.c_void_p), ("w", ctypes.c_void_p * 7), ("s", ctypes.c_void_p * 7)]


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc: -O2, no fast-math, no FMA contraction."""
    out_dir = os.path.join(_HERE, "_build")
    so = os.path.join(out_dir, "liboracle.so")
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(so) and os.path.getmtime(so) >= os.path.getmtime(src):
        return so
    os.makedirs(out_dir, exist_ok=True)
    tmp = so + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                           "-fno-fast-math", "-o", tmp, src, "-lm"])
    os.replace(tmp, so)
    return so


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            f32p = ctypes.POINTER(ctypes.c_float)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            vp = ctypes.c_void_p
            L.ora_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.ora_bf16_to_f32.restype = ctypes.c_float
            L.ora_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.ora_f16_to_f32.restype = ctypes.c_float
            L.ora_silu.argtypes = [ctypes.c_float]
            L.ora_silu.restype = ctypes.c_float
            L.ora_matvec.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, f32p, f32p, ctypes.c_int]
            L.ora_f32_to_f16.argtypes = [ctypes.c_float]
            L.ora_f32_to_f16.restype = ctypes.c_uint16
            L.ora_quantize_q8_block.argtypes = [f32p, vp, vp]
            L.ora_q8_block_dot.argtypes = [vp, vp]
            L.ora_q8_block_dot.restype = ctypes.c_int32
            L.ora_rmsnorm.argtypes = [f32p, vp, ctypes.c_int, ctypes.c_float, f32p]
            L.ora_rope_angles.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, f32p, f32p]
            L.ora_rope_apply.argtypes = [f32p, ctypes.c_int, f32p, f32p]
            L.ora_attention_head.argtypes = [f32p, f32p, f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, f32p, f32p]
            L.ora_argmax.argtypes = [f32p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int32)]
            u64p = ctypes.POINTER(ctypes.c_uint64)
            i32p = ctypes.POINTER(ctypes.c_int32)
            L.ora_pcg32_seed.argtypes = [ctypes.c_uint64, ctypes.c_uint64, u64p]
            L.ora_pcg32_seed.restype = None
            L.ora_sample.argtypes = [f32p, ctypes.c_int32, i32p, ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                     ctypes.c_float, ctypes.c_float, u64p, i32p, i32p, f32p, i32p, f32p]
            L.ora_create.argtypes = [ctypes.POINTER(_Config), vp, vp, ctypes.POINTER(_Layer), ctypes.POINTER(vp)]
            L.ora_destroy.argtypes = [vp]
            L.ora_destroy.restype = None
            L.ora_length.argtypes = [vp]
            L.ora_length.restype = ctypes.c_int32
            L.ora_kv_reset.argtypes = [vp]
            L.ora_kv_reset.restype = None
            L.ora_kv_import.argtypes = [vp, u16p, u16p, ctypes.c_int32]
            L.ora_step.argtypes = [vp, ctypes.c_int32, f32p, vp]
            L.ora_full.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, f32p]
            L.ora_set_kv_round_bf16.argtypes = [vp, ctypes.c_int]
            L.ora_set_kv_round_bf16.restype = None
            L.ora_kv_row.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, f32p, f32p]
            _LIB = L
    return _LIB


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _fp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


# ---------------------------------------------------------------- operators

def bf16_to_f32(b: int) -> float:
    return float(lib().ora_bf16_to_f32(b))


def f16_to_f32(h: int) -> float:
    return float(lib().ora_f16_to_f32(h))


def silu(g: float) -> float:
    return float(lib().ora_silu(ctypes.c_float(g)))


def rmsnorm(x, w_bf16=None, eps: float = 1e-6) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    w = None if w_bf16 is None else np.ascontiguousarray(w_bf16, dtype=np.uint16)
    lib().ora_rmsnorm(_fp(x), None if w is None else w.ctypes.data, x.size, eps, _fp(y))
    return y


def rope_angles(pos: int, d: int, theta: float):
    c = np.empty(d // 2, np.float32)
    s = np.empty(d // 2, np.float32)
    lib().ora_rope_angles(pos, d, theta, _fp(c), _fp(s))
    return c, s


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = _f32(v).copy()
    c, s = rope_angles(pos, v.size, theta)
    lib().ora_rope_apply(_fp(v), v.size, _fp(c), _fp(s))
    return v


def attention_head(q, K, V) -> np.ndarray:
    q, K, V = _f32(q), _f32(K), _f32(V)
    n, d = K.shape
    o = np.empty(d, np.float32)
    scr = np.empty(max(n, 1), np.float32)
    rc = lib().ora_attention_head(_fp(q), _fp(K), _fp(V), n, d, d, _fp(o), _fp(scr))
    if rc:
        raise OracleError(rc, "attention_head")
    return o


def matvec(w, x, scales=None, q8_act: bool = False) -> np.ndarray:
    """y = W x with W bf16 bits [rows, cols] (uint16) or int8 codes [rows, cols] + fp16 scales;
    q8_act: the input quantized per 32-element block first (the Q8 x Q8 format)."""
    x = _f32(x)
    rows, cols = w.shape
    y = np.empty(rows, np.float32)
    if scales is None:
        w = np.ascontiguousarray(w, dtype=np.uint16)
        rc = lib().ora_matvec(W_BF16, w.ctypes.data, None, rows, cols, _fp(x), _fp(y), 1)
    else:
        w = np.ascontiguousarray(w, dtype=np.int8)
        s = np.ascontiguousarray(scales, dtype=np.uint16)
        rc = lib().ora_matvec(W_Q8Q8 if q8_act else W_INT8_G32, w.ctypes.data, s.ctypes.data, rows, cols, _fp(x),
                              _fp(y), 1)
    if rc:
        raise OracleError(rc, "matvec")
    return y


def f32_to_f16(v: float) -> int:
    """binary32 -> binary16 bits, round to nearest even."""
    return int(lib().ora_f32_to_f16(ctypes.c_float(v)))


def quantize_q8_block(a):
    """(int8 codes [32], fp16 scale bits) of one 32-element activation block (Q8 x Q8 format)."""
    a = _f32(a)
    if a.size != 32:
        raise ValueError("a block has 32 elements")
    q = np.empty(32, np.int8)
    s = np.zeros(1, np.uint16)
    lib().ora_quantize_q8_block(_fp(a), q.ctypes.data, s.ctypes.data)
    return q, int(s[0])


def q8_block_dot(w, a) -> int:
    """i32 sum of the 32 products of two int8 blocks."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    a = np.ascontiguousarray(a, dtype=np.int8)
    return int(lib().ora_q8_block_dot(w.ctypes.data, a.ctypes.data))


def argmax(logits) -> int:
    x = _f32(logits)
    out = ctypes.c_int32(-1)
    rc = lib().ora_argmax(_fp(x), x.size, ctypes.byref(out))
    if rc:
        raise OracleError(rc, "argmax")
    return int(out.value)


# -------------------------------------------------------------------- model

def pcg32_seed(seed: int, stream: int) -> np.ndarray:
    """PCG32 state (state, increment) after the pages' seeding procedure."""
    out = np.zeros(2, np.uint64)
    lib().ora_pcg32_seed(ctypes.c_uint64(seed), ctypes.c_uint64(stream), out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
    return out


def sample(logits, rng: np.ndarray, temperature: float, top_k: int = 0, top_p: float = 1.0, penalty: float = 1.0,
           history=()):
    """One sampling step over f32 logits; rng ([state, increment], uint64) advances in place.

    Returns (token, retained candidate ids in draw order, their cumulative probabilities, u)."""
    x = _f32(logits)
    V = x.size
    h = np.ascontiguousarray(history, dtype=np.int32)
    ids = np.empty(V, np.int32)
    cum = np.empty(V, np.float32)
    n = ctypes.c_int32(0)
    tok = ctypes.c_int32(-1)
    u = ctypes.c_float(0.0)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = lib().ora_sample(_fp(x), V, h.ctypes.data_as(i32p), h.size, float(temperature), int(top_k), float(top_p),
                          float(penalty), rng.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), ctypes.byref(tok),
                          ids.ctypes.data_as(i32p), _fp(cum), ctypes.byref(n), ctypes.byref(u))
    if rc:
        raise OracleError(rc, "sample")
    return int(tok.value), ids[:n.value].copy(), cum[:n.value].copy(), float(u.value)


class OracleModel:
    """The decoder over borrowed numpy weights (from ``qw_inputs.make_weights``)."""

    def __init__(self, wl, weights, max_ctx: int | None = None, nthreads: int | None = None):
        self.wl = wl
        self._w = weights  # keep the arrays alive
        fmt = W_INT8_G32 if wl.weight_format == "int8_g32" else W_BF16
        if getattr(wl, "act_format", "f32") == "q8":
            if fmt != W_INT8_G32:
                raise ValueError("int8 activations need int8 g32 weights")
            fmt = W_Q8Q8
        cfg = _Config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate, wl.vocab,
                      wl.rms_eps, wl.rope_theta, max_ctx or wl.max_ctx, fmt,
                      nthreads or max(1, os.cpu_count() or 1))
        self.cfg = cfg
        layers = (_Layer * wl.n_layers)()
        for l, lw in enumerate(weights["layers"]):
            L = layers[l]
            L.input_norm = lw["input_norm"].ctypes.data
            L.q_norm = lw["q_norm"].ctypes.data
            L.k_norm = lw["k_norm"].ctypes.data
            L.post_norm = lw["post_norm"].ctypes.data
            for j, m in enumerate(MATRICES):
                if fmt != W_BF16:
                    L.w[j] = lw[m + "_q8"].ctypes.data
                    L.s[j] = lw[m + "_s"].ctypes.data
                else:
                    L.w[j] = lw[m].ctypes.data
                    L.s[j] = None
        self._layers = layers
        h = ctypes.c_void_p()
        rc = lib().ora_create(ctypes.byref(cfg), weights["embed"].ctypes.data, weights["final_norm"].ctypes.data,
                              layers, ctypes.byref(h))
        if rc:
            raise OracleError(rc, "create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().ora_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @property
    def length(self) -> int:
        return int(lib().ora_length(self._h))

    def reset(self):
        lib().ora_kv_reset(self._h)

    def kv_import(self, k_bf16: np.ndarray, v_bf16: np.ndarray, n_pos: int):
        k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
        v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
        rc = lib().ora_kv_import(self._h, k.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                 v.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), n_pos)
        if rc:
            raise OracleError(rc, "kv_import")

    def set_kv_round_bf16(self, on: bool):
        """Error attribution only: store K/V rounded to bf16 (not the reference computation)."""
        lib().ora_set_kv_round_bf16(self._h, 1 if on else 0)

    def kv_row(self, l: int, kvh: int, pos: int):
        """The cached f32 (key, value) rows of one layer, KV head and position."""
        k = np.empty(self.cfg.head_dim, np.float32)
        v = np.empty(self.cfg.head_dim, np.float32)
        rc = lib().ora_kv_row(self._h, l, kvh, pos, _fp(k), _fp(v))
        if rc:
            raise OracleError(rc, "kv_row")
        return k, v

    def step(self, token: int, want_hidden: bool = False, want_logits: bool = True):
        """One decode step: (logits [V] or None, hidden [L+1, H] or None).

        want_logits=False skips the final norm and head (a prompt row before the last)."""
        logits = np.empty(self.cfg.vocab, np.float32) if want_logits else None
        hidden = np.empty((self.cfg.n_layers + 1, self.cfg.hidden), np.float32) if want_hidden else None
        rc = lib().ora_step(self._h, int(token), None if logits is None else _fp(logits),
                            None if hidden is None else hidden.ctypes.data)
        if rc:
            raise OracleError(rc, "step")
        return logits, hidden

    def full(self, tokens) -> np.ndarray:
        """No-cache, causal-mask recomputation of every position's logits [T, V]."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty((t.size, self.cfg.vocab), np.float32)
        rc = lib().ora_full(self._h, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), t.size, _fp(logits))
        if rc:
            raise OracleError(rc, "full")
        return logits


def top2_margin(logits: np.ndarray) -> float:
    """Difference between the largest and second-largest logit."""
    part = np.partition(np.asarray(logits, np.float64), -2)[-2:]
    return float(part[1] - part[0])


def run_sequence(model: OracleModel, prompt, n_decode: int, want_hidden: bool = False, forced=None):
    """Prefill token by token, then greedy decode (or teacher-force `forced`).

    Returns dict with per-step logits (only for the last prompt position and
    each decode step), tokens fed, greedy picks, and hidden states if asked.
    """
    out = {"logits": [], "hidden": [], "inputs": [], "picks": []}
    last = None
    for i, tok in enumerate(prompt):
        is_last = i == len(prompt) - 1
        logits, hid = model.step(int(tok), want_hidden and is_last, want_logits=is_last)
        last = logits
    if len(prompt):
        out["logits"].append(last)
        out["hidden"].append(hid)
        out["picks"].append(argmax(last))
    nxt = out["picks"][-1] if out["picks"] else None
    for s in range(n_decode):
        tok = int(forced[s]) if forced is not None else nxt
        out["inputs"].append(tok)
        logits, hid = model.step(tok, want_hidden)
        out["logits"].append(logits)
        out["hidden"].append(hid)
        nxt = argmax(logits)
        out["picks"].append(nxt)
    return out
