"""ctypes binding of libqw.so (include/qw.h): argument marshalling only.

Every step of the decoder runs in the library's CUDA kernels; PyTorch provides the
device memory (weights, workspace) and the stream.  Importing this module does not
need a GPU; creating a model does, and there is no fallback: if the library is not
built or the device cannot run it, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqw.so")

OK = 0
INVALID_ARGUMENT = 1
INVALID_HANDLE = 4
ALIGNMENT = 7
INTEGER_OVERFLOW = 8
OUT_OF_MEMORY = 9
UNSUPPORTED_QUANTIZATION = 12
UNSUPPORTED_SHAPE = 13
CONTEXT_EXCEEDED = 14
NUMERICAL_FAILURE = 18
INTERNAL_INVARIANT = 20
CUDA_ERROR = 21

W_BF16 = 0
W_INT8_G32 = 1
W_Q8Q8 = 2
KV_F32 = 0
KV_BF16 = 1
DEBUG_HIDDEN = 1
DEBUG_PREFILL_BY_TOKEN = 2
DEBUG_TRACE = 4
DEBUG_ONE_GROUP = 8
DEBUG_WITHHOLD = 16
QUERY_DECODE_CTAS = 1
QUERY_TRACE_LEN = 2
QUERY_WORKSPACE_BYTES = 3
QUERY_DECODE_GROUPS = 4
QUERY_GROUP0_CTAS = 5
QUERY_RT_NEAR_NS = 6
QUERY_RT_FAR_NS = 7
QUERY_XREGION_OFFSET = 8
MATRICES = ("q", "k", "v", "o", "gate", "up", "down")

# every symbol include/qw.h declares
EXPORTS = ("qw_workspace_bytes", "qw_model_create", "qw_prefill", "qw_decode_step", "qw_generate", "qw_logits",
           "qw_kv_reset", "qw_kv_length", "qw_sync", "qw_model_destroy", "qw_kv_import", "qw_kv_export",
           "qw_set_debug", "qw_debug_hidden", "qw_status_string", "qw_abi_version", "qw_debug_trace", "qw_query",
           "qw_decode_step_noalloc", "qw_debug_gemm_f16", "qw_sample_scratch_bytes", "qw_sample_logits",
           "qw_sampler_seed", "qw_sampler_state", "qw_sample", "qw_batch_workspace_bytes", "qw_batch_create",
           "qw_batch_destroy", "qw_batch_reset", "qw_batch_length", "qw_batch_prefill", "qw_batch_step",
           "qw_batch_logits", "qw_batch_debug_hidden", "qw_batch_sync", "qw_checkpoint_open",
           "qw_checkpoint_close", "qw_checkpoint_last_error", "qw_checkpoint_count", "qw_checkpoint_tensor",
           "qw_checkpoint_check", "qw_checkpoint_upload_bytes", "qw_checkpoint_upload")
DT_BF16, DT_F16, DT_F32, DT_I8, DT_Q8_0 = 0, 1, 2, 3, 4
BATCH_MAX = 8


class CheckpointReport(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_int32), ("n_expected", ctypes.c_int32), ("n_found", ctypes.c_int32),
                ("n_missing", ctypes.c_int32), ("n_misshaped", ctypes.c_int32), ("n_unexpected", ctypes.c_int32),
                ("n_bad_dtype", ctypes.c_int32), ("lm_head_copy", ctypes.c_int32), ("stored_params", ctypes.c_int64),
                ("logical_params", ctypes.c_int64), ("embedding_params", ctypes.c_int64),
                ("first_problem", ctypes.c_char * 256)]


class QwError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = _lib().qw_status_string(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{what}: {msg} (status {code})")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("max_ctx", ctypes.c_int32), ("weight_format", ctypes.c_int32), ("kv_format", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("input_norm", ctypes.c_void_p), ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("post_norm", ctypes.c_void_p), ("w", ctypes.c_void_p * 7), ("s", ctypes.c_void_p * 7)]


class Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("repetition_penalty", ctypes.c_float)]


SAMPLE_MAX_TOP_K = 64


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


_LIB = None
_LOCK = threading.Lock()


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libqw.so is not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            i32p = ctypes.POINTER(ctypes.c_int32)
            L.qw_workspace_bytes.argtypes = [ctypes.POINTER(Config)]
            L.qw_workspace_bytes.restype = ctypes.c_size_t
            L.qw_model_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, ctypes.c_size_t, vp,
                                          ctypes.POINTER(vp)]
            L.qw_prefill.argtypes = [vp, i32p, i32, i32p]
            L.qw_decode_step.argtypes = [vp, i32, i32p]
            L.qw_generate.argtypes = [vp, i32, i32, vp]
            L.qw_logits.argtypes = [vp, vp, i64]
            L.qw_kv_reset.argtypes = [vp]
            L.qw_kv_length.argtypes = [vp, i32p]
            L.qw_sync.argtypes = [vp]
            L.qw_model_destroy.argtypes = [vp]
            L.qw_model_destroy.restype = None
            L.qw_kv_import.argtypes = [vp, vp, vp, i32]
            L.qw_kv_export.argtypes = [vp, vp, vp, i32]
            L.qw_set_debug.argtypes = [vp, i32]
            L.qw_debug_hidden.argtypes = [vp, vp, i64]
            L.qw_debug_trace.argtypes = [vp, vp, i64]
            L.qw_query.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64)]
            L.qw_decode_step_noalloc.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, vp, i32, i32, vp,
                                                 vp, vp, i32]
            L.qw_debug_gemm_f16.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
            L.qw_sample_scratch_bytes.argtypes = [i32]
            L.qw_sample_scratch_bytes.restype = ctypes.c_size_t
            L.qw_sample_logits.argtypes = [vp, i32, vp, i32, ctypes.POINTER(Sampling), vp, vp, vp, ctypes.c_size_t, vp]
            L.qw_sampler_seed.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64]
            L.qw_sampler_state.argtypes = [vp, vp]
            L.qw_sample.argtypes = [vp, ctypes.POINTER(Sampling), vp, i32, vp]
            L.qw_batch_workspace_bytes.argtypes = [vp, i32, i32]
            L.qw_batch_workspace_bytes.restype = ctypes.c_size_t
            L.qw_batch_create.argtypes = [vp, i32, i32, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)]
            L.qw_batch_destroy.argtypes = [vp]
            L.qw_batch_destroy.restype = None
            L.qw_batch_reset.argtypes = [vp, i32]
            L.qw_batch_length.argtypes = [vp, i32, i32p]
            L.qw_batch_prefill.argtypes = [vp, i32, i32p, i32, i32p]
            L.qw_batch_step.argtypes = [vp, i32, i32p, i32p]
            L.qw_batch_logits.argtypes = [vp, vp, i64]
            L.qw_batch_debug_hidden.argtypes = [vp, vp, i64]
            L.qw_batch_sync.argtypes = [vp]
            u64 = ctypes.c_uint64
            L.qw_checkpoint_open.argtypes = [vp, u64, u64, ctypes.POINTER(ctypes.c_void_p)]
            L.qw_checkpoint_close.argtypes = [vp]
            L.qw_checkpoint_close.restype = None
            L.qw_checkpoint_last_error.argtypes = []
            L.qw_checkpoint_last_error.restype = ctypes.c_char_p
            L.qw_checkpoint_count.argtypes = [vp]
            L.qw_checkpoint_count.restype = i32
            L.qw_checkpoint_tensor.argtypes = [vp, i32, ctypes.c_char_p, i32, i32p, i32p,
                                               ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(u64),
                                               ctypes.POINTER(u64)]
            L.qw_checkpoint_check.argtypes = [vp, ctypes.POINTER(Config), ctypes.POINTER(CheckpointReport)]
            L.qw_checkpoint_upload_bytes.argtypes = [vp, ctypes.POINTER(Config)]
            L.qw_checkpoint_upload_bytes.restype = ctypes.c_size_t
            L.qw_checkpoint_upload.argtypes = [vp, ctypes.POINTER(Config), vp, ctypes.c_size_t,
                                               ctypes.POINTER(LayerWeights), ctypes.POINTER(Weights), vp]
            L.qw_status_string.argtypes = [ctypes.c_int]
            L.qw_status_string.restype = ctypes.c_char_p
            L.qw_abi_version.argtypes = []
            L.qw_abi_version.restype = i32
            _LIB = L
    return _LIB


def lib():
    return _lib()


def _check(rc: int, what: str):
    if rc != OK:
        raise QwError(rc, what)


def make_config(dims, max_ctx: int | None = None) -> Config:
    """dims: any object with the Qwen3 dimension attributes (n_layers, hidden, ...)."""
    fmt = {"bf16": W_BF16, "int8_g32": W_INT8_G32}.get(getattr(dims, "weight_format", "bf16"), -1)
    if getattr(dims, "act_format", "f32") == "q8":
        fmt = W_Q8Q8 if fmt == W_INT8_G32 else -1
    kvf = {"f32": KV_F32, "bf16": KV_BF16}.get(getattr(dims, "kv_format", "f32"), -1)
    return Config(dims.n_layers, dims.hidden, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.intermediate,
                  dims.vocab, dims.rms_eps, dims.rope_theta, int(max_ctx or dims.max_ctx), fmt, kvf)


def workspace_bytes(cfg: Config) -> int:
    return int(_lib().qw_workspace_bytes(ctypes.byref(cfg)))


def weights_to_device(host_weights: dict, int8: bool, device="cuda"):
    """Copy a {embed, final_norm, layers[...]} dict of numpy arrays to device tensors.

    bf16 tensors travel as int16 bit patterns (the library reads raw bytes).  For the
    int8 format, each matrix m comes as "<m>_q8" (int8) and "<m>_s" (fp16 bits).
    """
    import torch

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(device)

    out = {"embed": dev(host_weights["embed"]), "final_norm": dev(host_weights["final_norm"]), "layers": []}
    for lw in host_weights["layers"]:
        d = {k: dev(lw[k]) for k in ("input_norm", "q_norm", "k_norm", "post_norm")}
        for m in MATRICES:
            if int8:
                d[m + "_q8"] = dev(lw[m + "_q8"])
                d[m + "_s"] = dev(lw[m + "_s"])
            else:
                d[m] = dev(lw[m])
        out["layers"].append(d)
    return out


def weight_table(dev_weights: dict, int8: bool):
    """(Weights struct, layer array) for device weights from ``weights_to_device``; keep both alive."""
    n = len(dev_weights["layers"])
    layers = (LayerWeights * n)()
    for l, lw in enumerate(dev_weights["layers"]):
        L = layers[l]
        L.input_norm = lw["input_norm"].data_ptr()
        L.q_norm = lw["q_norm"].data_ptr()
        L.k_norm = lw["k_norm"].data_ptr()
        L.post_norm = lw["post_norm"].data_ptr()
        for j, m in enumerate(MATRICES):
            if int8:
                L.w[j] = lw[m + "_q8"].data_ptr()
                L.s[j] = lw[m + "_s"].data_ptr()
            else:
                L.w[j] = lw[m].data_ptr()
    w = Weights(dev_weights["embed"].data_ptr(), dev_weights["final_norm"].data_ptr(), None, layers)
    return w, layers


def decode_step_noalloc(cfg: Config, dev_weights: dict, k_cache, v_cache, pos: int, token: int, logits_out,
                        next_token_out, stream=None, wait: bool = True):
    """qw_decode_step_noalloc: one step over caller-owned K/V planes; no device allocation.

    The library cannot see the sizes of the caller's buffers, so they are checked here:
    CUDA, contiguous, K/V planes of the cache element type cfg.kv_format names holding
    n_layers * n_kv_heads * max_ctx * head_dim elements each, f32 logits of at least
    vocab elements, an int32 slot for the pick.
    """
    import torch
    kv_dtype = torch.float32 if cfg.kv_format == KV_F32 else torch.bfloat16
    plane = cfg.n_layers * cfg.n_kv_heads * cfg.max_ctx * cfg.head_dim
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype != kv_dtype:
            raise ValueError(f"{name} must be {kv_dtype} for this kv_format")
        if t.numel() < plane:
            raise ValueError(f"{name} holds {t.numel()} elements, the config needs {plane}")
    if not (logits_out.is_cuda and logits_out.is_contiguous()) or logits_out.dtype != torch.float32 \
            or logits_out.numel() < cfg.vocab:
        raise ValueError("logits_out must be a contiguous CUDA float32 tensor of at least vocab elements")
    if not next_token_out.is_cuda or next_token_out.dtype != torch.int32 or next_token_out.numel() < 1:
        raise ValueError("next_token_out must be a CUDA int32 tensor")
    w, layers = weight_table(dev_weights, cfg.weight_format != W_BF16)
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(_lib().qw_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(w), k_cache.data_ptr(), v_cache.data_ptr(),
                                         int(pos), int(token), logits_out.data_ptr(), next_token_out.data_ptr(),
                                         st.cuda_stream, 1 if wait else 0), "qw_decode_step_noalloc")


def debug_gemm_f16(a, b, c, bn: int = 256, stream=None):
    """qw_debug_gemm_f16: c[M,N] = a[M,K] @ b[N,K]^T on the prefill's tensor-core GEMM (fp16 in, f32 out)."""
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    M, K = a.shape
    N = b.shape[0]
    _check(_lib().qw_debug_gemm_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), int(M), int(N), int(K), int(bn),
                                    st.cuda_stream), "qw_debug_gemm_f16")


def sample_logits(logits, params: Sampling, rng, token_out, history=None, scratch=None, stream=None):
    """qw_sample_logits on device tensors: logits f32 [V], rng uint64 [2] (int64 tensor),
    token_out int32 [1], history int32 [n] or None."""
    import torch
    V = logits.numel()
    need = _lib().qw_sample_scratch_bytes(V)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = stream if stream is not None else torch.cuda.current_stream()
    n = 0 if history is None else history.numel()
    _check(_lib().qw_sample_logits(logits.data_ptr(), V, history.data_ptr() if n else None, n, ctypes.byref(params),
                                   rng.data_ptr(), token_out.data_ptr(), scratch.data_ptr(), scratch.numel(),
                                   st.cuda_stream), "qw_sample_logits")


class Model:
    """One decoder instance on the current CUDA device and stream."""

    def __init__(self, dims, dev_weights: dict | None, max_ctx: int | None = None, stream=None, table=None):
        """dev_weights: device tensors from weights_to_device; or table = (keep-alive object,
        Weights, layer array) as Checkpoint.upload returns it."""
        import torch

        self.dims = dims
        self.cfg = make_config(dims, max_ctx)
        self.int8 = self.cfg.weight_format in (W_INT8_G32, W_Q8Q8)
        nbytes = workspace_bytes(self.cfg)
        if nbytes == 0:
            raise QwError(UNSUPPORTED_SHAPE, "workspace_bytes")
        self._w = dev_weights if table is None else table
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        if table is not None:
            self._layers = table[2]
            h = ctypes.c_void_p()
            _check(_lib().qw_model_create(ctypes.byref(self.cfg), ctypes.byref(table[1]), self.workspace.data_ptr(),
                                          nbytes, self.stream.cuda_stream, ctypes.byref(h)), "qw_model_create")
            self._h = h
            return
        layers = (LayerWeights * self.cfg.n_layers)()
        for l, lw in enumerate(dev_weights["layers"]):
            L = layers[l]
            L.input_norm = lw["input_norm"].data_ptr()
            L.q_norm = lw["q_norm"].data_ptr()
            L.k_norm = lw["k_norm"].data_ptr()
            L.post_norm = lw["post_norm"].data_ptr()
            for j, m in enumerate(MATRICES):
                if self.int8:
                    L.w[j] = lw[m + "_q8"].data_ptr()
                    L.s[j] = lw[m + "_s"].data_ptr()
                else:
                    L.w[j] = lw[m].data_ptr()
        self._layers = layers
        w = Weights(dev_weights["embed"].data_ptr(), dev_weights["final_norm"].data_ptr(), None, layers)
        h = ctypes.c_void_p()
        _check(_lib().qw_model_create(ctypes.byref(self.cfg), ctypes.byref(w), self.workspace.data_ptr(), nbytes,
                                      self.stream.cuda_stream, ctypes.byref(h)), "qw_model_create")
        self._h = h

    # ---------------------------------------------------------------- lifecycle
    def close(self):
        if getattr(self, "_h", None):
            _lib().qw_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # ------------------------------------------------------------------- calls
    def prefill(self, tokens, want_token: bool = True):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = ctypes.c_int32(-1)
        _check(_lib().qw_prefill(self._h, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), t.size,
                                 ctypes.byref(out) if want_token else None), "qw_prefill")
        return int(out.value) if want_token else None

    def decode_step(self, token: int = -1, want_token: bool = True):
        out = ctypes.c_int32(-1)
        _check(_lib().qw_decode_step(self._h, int(token), ctypes.byref(out) if want_token else None),
               "qw_decode_step")
        return int(out.value) if want_token else None

    def generate(self, n: int, token: int = -1, tokens_out=None):
        """Greedy n steps with no host sync; tokens_out: device int32 tensor [n] or None."""
        _check(_lib().qw_generate(self._h, int(token), int(n),
                                  tokens_out.data_ptr() if tokens_out is not None else None), "qw_generate")

    def logits(self, out=None):
        import torch
        if out is None:
            out = torch.empty(self.cfg.vocab, dtype=torch.float32, device="cuda")
        _check(_lib().qw_logits(self._h, out.data_ptr(), out.numel()), "qw_logits")
        return out

    def sync(self):
        _check(_lib().qw_sync(self._h), "qw_sync")

    def kv_reset(self):
        _check(_lib().qw_kv_reset(self._h), "qw_kv_reset")

    @property
    def kv_length(self) -> int:
        n = ctypes.c_int32(-1)
        _check(_lib().qw_kv_length(self._h, ctypes.byref(n)), "qw_kv_length")
        return int(n.value)

    def kv_import(self, k, v, n_pos: int):
        _check(_lib().qw_kv_import(self._h, k.data_ptr(), v.data_ptr(), int(n_pos)), "qw_kv_import")

    def kv_export(self, n_pos: int):
        import torch
        c = self.cfg
        shape = (c.n_layers, c.n_kv_heads, n_pos, c.head_dim)
        dt = torch.float32 if c.kv_format == KV_F32 else torch.bfloat16
        k = torch.empty(shape, dtype=dt, device="cuda")
        v = torch.empty(shape, dtype=dt, device="cuda")
        _check(_lib().qw_kv_export(self._h, k.data_ptr(), v.data_ptr(), int(n_pos)), "qw_kv_export")
        return k, v

    def sampler_seed(self, seed: int, stream: int):
        _check(_lib().qw_sampler_seed(self._h, ctypes.c_uint64(seed), ctypes.c_uint64(stream)), "qw_sampler_seed")

    def sampler_state(self):
        out = (ctypes.c_uint64 * 2)()
        _check(_lib().qw_sampler_state(self._h, out), "qw_sampler_state")
        return int(out[0]), int(out[1])

    def sample(self, params: Sampling, history=None, want_token: bool = True):
        """qw_sample: next token from the last position's logits; history: device int32 tensor or None."""
        out = ctypes.c_int32(-1)
        n = 0 if history is None else history.numel()
        _check(_lib().qw_sample(self._h, ctypes.byref(params), history.data_ptr() if n else None, n,
                                ctypes.byref(out) if want_token else None), "qw_sample")
        return int(out.value) if want_token else None

    def set_debug(self, flags: int):
        _check(_lib().qw_set_debug(self._h, int(flags)), "qw_set_debug")

    def query(self, what: int) -> int:
        v = ctypes.c_int64(-1)
        _check(_lib().qw_query(self._h, int(what), ctypes.byref(v)), "qw_query")
        return int(v.value)

    def debug_trace(self):
        """[phase, cta, 16] uint64 ns timeline of the last decode step (needs DEBUG_TRACE)."""
        import torch
        n = self.query(QUERY_TRACE_LEN)
        ncta = self.query(QUERY_DECODE_CTAS)
        out = torch.zeros(n, dtype=torch.int64, device="cuda")
        _check(_lib().qw_debug_trace(self._h, out.data_ptr(), n), "qw_debug_trace")
        return out.view(-1, ncta, 16)

    def debug_hidden(self):
        import torch
        c = self.cfg
        out = torch.empty((c.n_layers + 1, c.hidden), dtype=torch.float32, device="cuda")
        _check(_lib().qw_debug_hidden(self._h, out.data_ptr(), out.numel()), "qw_debug_hidden")
        return out


class Batch:
    """Up to BATCH_MAX sequences of one Model decoded together (qw_batch_*), each with its own
    K/V cache and length; workspace from torch on the model's device."""

    def __init__(self, model: "Model", max_batch: int, max_ctx: int):
        import torch

        self.model = model
        self.max_batch = max_batch
        self.max_ctx = max_ctx
        n = _lib().qw_batch_workspace_bytes(model._h, max_batch, max_ctx)
        if n == 0:
            raise QwError(INVALID_ARGUMENT, "qw_batch_workspace_bytes")
        self.workspace = torch.empty(n, dtype=torch.uint8, device="cuda")
        h = ctypes.c_void_p()
        _check(_lib().qw_batch_create(model._h, max_batch, max_ctx, self.workspace.data_ptr(), n, ctypes.byref(h)),
               "qw_batch_create")
        self._h = h
        self.last_n = 0

    def close(self):
        if getattr(self, "_h", None):
            _lib().qw_batch_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, seq: int = -1):
        _check(_lib().qw_batch_reset(self._h, seq), "qw_batch_reset")

    def length(self, seq: int) -> int:
        out = ctypes.c_int32()
        _check(_lib().qw_batch_length(self._h, seq, ctypes.byref(out)), "qw_batch_length")
        return out.value

    def prefill(self, seq: int, tokens, want_token: bool = True):
        t = (ctypes.c_int32 * len(tokens))(*[int(x) for x in tokens])
        out = ctypes.c_int32(-1)
        _check(_lib().qw_batch_prefill(self._h, seq, t, len(tokens), ctypes.byref(out) if want_token else None),
               "qw_batch_prefill")
        return out.value if want_token else None

    def step(self, n_seq: int, tokens=None, want_tokens: bool = True):
        """One step of sequences 0..n_seq-1; tokens None (or -1 entries) = each one's last pick."""
        t = None if tokens is None else (ctypes.c_int32 * n_seq)(*[int(x) for x in tokens])
        out = (ctypes.c_int32 * n_seq)()
        _check(_lib().qw_batch_step(self._h, n_seq, t, out if want_tokens else None), "qw_batch_step")
        self.last_n = n_seq
        return list(out) if want_tokens else None

    def logits(self):
        import torch

        V = self.model.cfg.vocab
        out = torch.empty((self.last_n, V), dtype=torch.float32, device="cuda")
        _check(_lib().qw_batch_logits(self._h, out.data_ptr(), out.numel()), "qw_batch_logits")
        return out

    def debug_hidden(self):
        import torch

        c = self.model.cfg
        out = torch.empty((c.n_layers + 1, self.last_n, c.hidden), dtype=torch.float32, device="cuda")
        _check(_lib().qw_batch_debug_hidden(self._h, out.data_ptr(), out.numel()), "qw_batch_debug_hidden")
        return out

    def sync(self):
        _check(_lib().qw_batch_sync(self._h), "qw_batch_sync")


class Checkpoint:
    """A safetensors / SLM2 checkpoint held in host memory (qw_checkpoint_*): `data` is the file's
    bytes (or only its prefix and header, with file_size the whole file's size)."""

    def __init__(self, data, file_size: int | None = None):
        self._buf = bytes(data) if not isinstance(data, (bytes, bytearray)) else data
        self._c = ctypes.create_string_buffer(bytes(self._buf), len(self._buf))
        size = len(self._buf) if file_size is None else file_size
        h = ctypes.c_void_p()
        rc = _lib().qw_checkpoint_open(ctypes.cast(self._c, ctypes.c_void_p), len(self._buf), size, ctypes.byref(h))
        if rc != OK:
            raise QwError(rc, "qw_checkpoint_open: " + _lib().qw_checkpoint_last_error().decode())
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            _lib().qw_checkpoint_close(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def tensors(self):
        """[(name, dtype, shape, begin, end)] sorted by begin."""
        out = []
        for i in range(_lib().qw_checkpoint_count(self._h)):
            name = ctypes.create_string_buffer(512)
            dt, rk = ctypes.c_int32(), ctypes.c_int32()
            dims = (ctypes.c_int64 * 4)()
            b, e = ctypes.c_uint64(), ctypes.c_uint64()
            _check(_lib().qw_checkpoint_tensor(self._h, i, name, 512, ctypes.byref(dt), ctypes.byref(rk), dims,
                                               ctypes.byref(b), ctypes.byref(e)), "qw_checkpoint_tensor")
            out.append((name.value.decode(), dt.value, tuple(dims[:rk.value]), b.value, e.value))
        return out

    def check(self, cfg: Config):
        """(status, CheckpointReport): status OK when the file matches cfg's tensor set."""
        rep = CheckpointReport()
        rc = _lib().qw_checkpoint_check(self._h, ctypes.byref(cfg), ctypes.byref(rep))
        return rc, rep

    def upload(self, cfg: Config):
        """Device copy of the weights in the layout qw_model_create takes: (workspace tensor, Weights, layers)."""
        import torch

        n = _lib().qw_checkpoint_upload_bytes(self._h, ctypes.byref(cfg))
        if n == 0:
            raise QwError(INVALID_ARGUMENT, "qw_checkpoint_upload_bytes")
        buf = torch.empty(n, dtype=torch.uint8, device="cuda")
        layers = (LayerWeights * cfg.n_layers)()
        table = Weights()
        rc = _lib().qw_checkpoint_upload(self._h, ctypes.byref(cfg), buf.data_ptr(), n, layers, ctypes.byref(table),
                                         torch.cuda.current_stream().cuda_stream)
        if rc != OK:
            raise QwError(rc, "qw_checkpoint_upload: " + _lib().qw_checkpoint_last_error().decode())
        return buf, table, layers
