"""Host-only checks of the C ABI: the library loads, exports every declared symbol, and
rejects bad arguments before it touches a device (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import qw_inputs as qi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qw():
    from runtime_qwen3_decode_gb300 import build, qw as binding
    build.build()
    return binding


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qw.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qw_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(qw):
    decl = declared_functions()
    assert len(decl) >= 16
    L = qw.lib()
    for name in decl:
        assert hasattr(L, name), f"{name} declared in qw.h but not exported"
    assert sorted(qw.EXPORTS) == decl
    assert L.qw_abi_version() == 1
    assert L.qw_status_string(14) == b"context exceeded"


def cfg_of(qw, **kw):
    wl = qi.WORKLOADS["qwen3_0p6b_decode"].with_(**kw)
    return qw.make_config(wl, wl.max_ctx)


def test_workspace_bytes(qw):
    c = cfg_of(qw)
    n = qw.workspace_bytes(c)
    kv = 2 * 28 * 8 * c.max_ctx * 128 * 4  # f32 cache
    # fp16 copies of the seven projection matrices for the tensor-core prefill
    H, QD, KD, I = 1024, 2048, 1024, 3072
    w16 = 28 * 2 * ((QD + 2 * KD) * H + H * QD + 2 * I * H + H * I)
    assert n > kv + w16
    assert qw.workspace_bytes(cfg_of(qw, kv_format="bf16")) < n - kv // 2 + 2 ** 20
    assert n < kv + w16 + 200 * 2 ** 20  # activations, RoPE table, prefill buffers
    # unsupported or invalid configs report 0
    assert qw.workspace_bytes(cfg_of(qw, head_dim=64)) == 0
    assert qw.workspace_bytes(cfg_of(qw, hidden=1000)) == 0
    assert qw.workspace_bytes(cfg_of(qw, n_kv_heads=3)) == 0
    assert qw.workspace_bytes(cfg_of(qw, n_kv_heads=4)) == 0   # group of 4: not built
    assert qw.workspace_bytes(cfg_of(qw, intermediate=4096)) == 0


def _create(qw, cfg, weights=None, ws=0x100000, ws_bytes=None):
    if weights is None:
        layers = (qw.LayerWeights * cfg.n_layers)()
        fake = 0x7F0000000000
        for L in layers:
            L.input_norm = L.q_norm = L.k_norm = L.post_norm = fake
            for i in range(7):
                L.w[i] = fake
                L.s[i] = fake
        weights = qw.Weights(fake, fake, None, layers)
    h = ctypes.c_void_p()
    nbytes = ws_bytes if ws_bytes is not None else qw.workspace_bytes(cfg)
    rc = qw.lib().qw_model_create(ctypes.byref(cfg), ctypes.byref(weights), ws, nbytes, None, ctypes.byref(h))
    return rc, h


def test_create_validates_before_device(qw):
    c = cfg_of(qw)
    bad = cfg_of(qw)
    bad.weight_format = 7
    assert _create(qw, bad)[0] == qw.UNSUPPORTED_QUANTIZATION
    assert _create(qw, cfg_of(qw, hidden=1000))[0] == qw.UNSUPPORTED_QUANTIZATION   # not a multiple of 32
    assert _create(qw, cfg_of(qw, hidden=1056))[0] == qw.UNSUPPORTED_SHAPE          # /32 but not /1024
    assert _create(qw, cfg_of(qw, head_dim=64))[0] == qw.UNSUPPORTED_SHAPE
    assert _create(qw, cfg_of(qw, n_kv_heads=5))[0] == qw.UNSUPPORTED_SHAPE
    assert _create(qw, cfg_of(qw, decode_steps=-200))[0] == qw.INVALID_ARGUMENT    # max_ctx < 1
    bad = cfg_of(qw)
    bad.kv_format = 3
    assert _create(qw, bad)[0] == qw.INVALID_ARGUMENT
    assert _create(qw, c, ws=0x100010)[0] == qw.ALIGNMENT
    assert _create(qw, c, ws_bytes=1000)[0] == qw.OUT_OF_MEMORY
    w = qw.Weights(None, None, None, None)
    assert _create(qw, c, weights=w)[0] == qw.INVALID_ARGUMENT
    # misaligned weight pointer
    layers = (qw.LayerWeights * c.n_layers)()
    for L in layers:
        L.input_norm = L.q_norm = L.k_norm = L.post_norm = 0x7F0000000000
        for i in range(7):
            L.w[i] = 0x7F0000000000
    layers[3].w[2] = 0x7F0000000002
    assert _create(qw, c, weights=qw.Weights(0x7F0000000000, 0x7F0000000000, None, layers))[0] == qw.ALIGNMENT
    # int8 format needs scale pointers
    c8 = cfg_of(qw, weight_format="int8_g32")
    layers[3].w[2] = 0x7F0000000000
    assert _create(qw, c8, weights=qw.Weights(0x7F0000000000, 0x7F0000000000, None, layers))[0] == \
        qw.INVALID_ARGUMENT


def test_create_without_device_fails_loudly(qw):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    rc, h = _create(qw, cfg_of(qw))
    assert rc == qw.CUDA_ERROR and not h.value


def test_handles_are_checked(qw):
    L = qw.lib()
    n = ctypes.c_int32()
    assert L.qw_kv_length(None, ctypes.byref(n)) == qw.INVALID_HANDLE
    assert L.qw_kv_length(0x1234560, ctypes.byref(n)) == qw.INVALID_HANDLE
    assert L.qw_decode_step(0x1234560, 0, None) == qw.INVALID_HANDLE
    assert L.qw_prefill(None, None, 0, None) == qw.INVALID_HANDLE
    L.qw_model_destroy(None)
    L.qw_model_destroy(0x1234560)  # unknown handles are ignored


def test_binding_refuses_without_library(tmp_path, monkeypatch):
    import runtime_qwen3_decode_gb300.qw as b
    monkeypatch.setattr(b, "_LIB", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        b.lib()
