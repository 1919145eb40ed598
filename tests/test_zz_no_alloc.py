"""qw_decode_step_noalloc: the decode step for callers that cannot allocate device memory.

Code that runs inside another framework's memory pool, or under a hard device-memory
budget, may not be able to call cudaMalloc when it decodes.  The entry point keeps all of
its intermediate buffers in one fixed array inside the library instead, and runs the same
decode kernel with the same SM groups as a model created on the same device.  These tests
check, through the C ABI, that two consecutive steps give exactly the same logits, greedy
picks and appended K/V rows as the regular handle-based step (qw_decode_step) on the same
inputs, for both cache formats and both weight formats, and that a call after the first
one leaves the device's free memory unchanged.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import qw_inputs as qi  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("weight_format,kv_format", [("bf16", "f32"), ("bf16", "bf16"), ("int8_g32", "f32")])
def test_noalloc_step_matches_regular_step_twice(weight_format, kv_format):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw
    build.build()

    wl = qi.WORKLOADS["tiny"].with_(weight_format=weight_format, kv_format=kv_format)
    int8 = weight_format == "int8_g32"
    max_ctx = 64
    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=int8)
    model = qw.Model(wl, dev, max_ctx=max_ctx)
    prompt = qi.prompt(wl)
    tok = model.prefill(prompt)
    n = len(prompt)

    # the caller's own cache planes, holding the rows the regular model has so far
    kv_dtype = torch.float32 if kv_format == "f32" else torch.bfloat16
    shape = (wl.n_layers, wl.n_kv_heads, max_ctx, wl.head_dim)
    kc = torch.zeros(shape, dtype=kv_dtype, device="cuda")
    vc = torch.zeros(shape, dtype=kv_dtype, device="cuda")
    k0, v0 = model.kv_export(n)
    kc[:, :, :n] = k0
    vc[:, :, :n] = v0
    cfg = qw.make_config(wl, max_ctx)
    logits = torch.empty(wl.vocab, dtype=torch.float32, device="cuda")
    pick = torch.full((1,), -1, dtype=torch.int32, device="cuda")

    for step in range(2):
        pos = n + step
        ref_pick = model.decode_step(tok)
        ref_logits = model.logits().cpu().numpy()
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        qw.decode_step_noalloc(cfg, dev, kc, vc, pos, tok, logits, pick, wait=True)
        free_after = torch.cuda.mem_get_info()[0]
        if step == 1:  # the first call sets the fixed array up; later calls allocate nothing
            assert free_after == free_before
        got = logits.cpu().numpy()
        assert np.all(np.isfinite(got))
        np.testing.assert_array_equal(got, ref_logits)
        assert int(pick.item()) == ref_pick
        # the step appended this position's K/V to the caller's planes, bit for bit
        k_ref, v_ref = model.kv_export(pos + 1)
        assert torch.equal(kc[:, :, pos].contiguous().view(torch.int16), k_ref[:, :, pos].contiguous().view(torch.int16))
        assert torch.equal(vc[:, :, pos].contiguous().view(torch.int16), v_ref[:, :, pos].contiguous().view(torch.int16))
        tok = ref_pick
    model.close()


def test_noalloc_rejects_bad_arguments():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw
    build.build()
    wl = qi.WORKLOADS["tiny"]
    dev = qw.weights_to_device(qi.make_weights(wl), int8=False)
    cfg = qw.make_config(wl, 16)
    shape = (wl.n_layers, wl.n_kv_heads, 16, wl.head_dim)
    kc = torch.zeros(shape, dtype=torch.float32, device="cuda")
    vc = torch.zeros(shape, dtype=torch.float32, device="cuda")
    logits = torch.empty(wl.vocab, dtype=torch.float32, device="cuda")
    pick = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(qw.QwError) as e:
        qw.decode_step_noalloc(cfg, dev, kc, vc, 16, 1, logits, pick)
    assert e.value.code == qw.CONTEXT_EXCEEDED
    with pytest.raises(qw.QwError) as e:
        qw.decode_step_noalloc(cfg, dev, kc, vc, 0, wl.vocab, logits, pick)
    assert e.value.code == qw.INVALID_ARGUMENT
    # buffers the library cannot size are checked by the binding before the call
    with pytest.raises(ValueError):
        qw.decode_step_noalloc(cfg, dev, kc[:, :, :8].contiguous(), vc, 0, 1, logits, pick)
    with pytest.raises(ValueError):
        qw.decode_step_noalloc(cfg, dev, kc.to(torch.bfloat16), vc, 0, 1, logits, pick)
    with pytest.raises(ValueError):
        qw.decode_step_noalloc(cfg, dev, kc, vc, 0, 1, logits[:100], pick)
