"""Checkpoint upload (qw_checkpoint_upload): a model created from an uploaded synthetic checkpoint
decodes bit for bit like the same model created from the weights directly, for bf16 matrices with
bf16 norms and for SLM2-style Q8_0 matrices with f32 norms (the int8 g32 path)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import qw_inputs as qi  # noqa: E402
from _ckpt import build, model_entries  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build as b, qw as binding
    b.build()
    return binding


def _decode(m, prompt, n):
    picks = [m.prefill(prompt)]
    logits = [m.logits().cpu().numpy()]
    for _ in range(n):
        picks.append(m.decode_step(-1))
        logits.append(m.logits().cpu().numpy())
    return picks, logits


@pytest.mark.parametrize("q8", [False, True])
def test_uploaded_checkpoint_decodes_identically(qw, q8):
    wl = qi.WORKLOADS["tiny"].with_(weight_format="int8_g32") if q8 else qi.WORKLOADS["tiny"]
    w = qi.make_weights(wl)
    ck = qw.Checkpoint(build(model_entries(wl, w, q8=q8, f32_norms=q8)))
    cfg = qw.make_config(wl, 64)
    assert ck.check(cfg)[0] == qw.OK
    a = qw.Model(wl, None, max_ctx=64, table=ck.upload(cfg))
    b = qw.Model(wl, qw.weights_to_device(w, int8=q8), max_ctx=64)
    prompt = qi.prompt(wl)
    pa, la = _decode(a, prompt, 6)
    pb, lb = _decode(b, prompt, 6)
    assert pa == pb
    for x, y in zip(la, lb):
        np.testing.assert_array_equal(x, y)
    a.close()
    b.close()


def test_f32_norm_off_the_bf16_grid_is_refused(qw):
    wl = qi.WORKLOADS["tiny"]
    w = qi.make_weights(wl)
    ents = model_entries(wl, w, f32_norms=True)
    name, dt, shape, payload = ents[1]  # layer 0 input_layernorm, f32
    v = np.frombuffer(payload, np.uint32).copy()
    v[3] |= 1  # one low mantissa bit: not a bf16 value
    ents[1] = (name, dt, shape, v.tobytes())
    ck = qw.Checkpoint(build(ents))
    with pytest.raises(qw.QwError) as e:
        ck.upload(qw.make_config(wl, 64))
    assert e.value.code == qw.UNSUPPORTED_QUANTIZATION
