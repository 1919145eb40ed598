"""qw_decode_step_noalloc: the decode step for callers that cannot allocate device memory.

The entry point keeps all of its intermediate buffers in one fixed array inside the
library, so a caller running under someone else's memory pool or a hard memory budget
can decode without any cudaMalloc.  This test checks, through the C ABI, that two
consecutive steps give the same logits, greedy picks and appended K/V rows as the
regular handle-based decode step (qw_decode_step) on the same inputs.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import qw_inputs as qi  # noqa: E402
from _helpers import LOGITS_MAX_ABS  # noqa: E402

pytestmark = pytest.mark.gpu


def test_noalloc_step_matches_regular_step_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw
    build.build()

    wl = qi.WORKLOADS["tiny"]
    max_ctx = 64
    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=False)
    model = qw.Model(wl, dev, max_ctx=max_ctx)
    prompt = qi.prompt(wl)
    tok = model.prefill(prompt)
    n = len(prompt)

    # the caller's own cache planes, holding the rows the regular model has so far
    shape = (wl.n_layers, wl.n_kv_heads, max_ctx, wl.head_dim)
    kc = torch.zeros(shape, dtype=torch.float32, device="cuda")
    vc = torch.zeros(shape, dtype=torch.float32, device="cuda")
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
        qw.decode_step_noalloc(cfg, dev, kc, vc, pos, tok, logits, pick, wait=True)
        got = logits.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.abs(got - ref_logits).max()) <= LOGITS_MAX_ABS
        assert int(pick.item()) == ref_pick
        # the step appended this position's K/V to the caller's planes
        k_ref, v_ref = model.kv_export(pos + 1)
        np.testing.assert_allclose(kc[:, :, pos].cpu().numpy(), k_ref[:, :, pos].cpu().numpy(), rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(vc[:, :, pos].cpu().numpy(), v_ref[:, :, pos].cpu().numpy(), rtol=1e-5, atol=1e-5)
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
