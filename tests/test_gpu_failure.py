"""The decode kernel's bounded-wait failure path, exercised without a fault or a hang.

Under QW_DEBUG_WITHHOLD one SM leaves out its outputs of the step's first phase and every
device-side wait gives up after 1 ms: the waiting CTAs record QW_INTERNAL_INVARIANT, raise the
abort flag the others watch, drain their copies in flight and return.  The model then refuses
further work until qw_kv_reset, after which decoding matches the oracle again.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import qw_inputs as qi  # noqa: E402
from _helpers import check_position  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw as binding
    build.build()
    return binding


def _expect_status(qw, fn, code):
    with pytest.raises(qw.QwError) as ei:
        fn()
    assert ei.value.code == code, (ei.value.code, str(ei.value))


@pytest.mark.parametrize("one_group", [False, True])
def test_withheld_output_fails_the_step_then_reset_recovers(qw, one_group):
    wl = qi.WORKLOADS["tiny"]
    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=False)
    m = qw.Model(wl, dev)
    base = qw.DEBUG_ONE_GROUP if one_group else 0
    m.set_debug(base)
    prompt = qi.prompt(wl)
    m.prefill(prompt[:3])

    m.set_debug(base | qw.DEBUG_WITHHOLD)
    t = time.perf_counter()
    _expect_status(qw, lambda: m.decode_step(int(prompt[3])), qw.INTERNAL_INVARIANT)
    assert time.perf_counter() - t < 5.0  # the 1 ms limit, not the normal 1 s one, ended the waits
    # refused without launching: same status for every call until the reset
    m.set_debug(base)
    _expect_status(qw, lambda: m.decode_step(int(prompt[3])), qw.INTERNAL_INVARIANT)
    _expect_status(qw, lambda: m.prefill(prompt[3:5]), qw.INTERNAL_INVARIANT)
    _expect_status(qw, lambda: m.generate(2, int(prompt[3])), qw.INTERNAL_INVARIANT)

    # the reset clears the failure; a fresh sequence matches the oracle position by position
    m.kv_reset()
    assert m.kv_length == 0
    ref = oracle.OracleModel(wl, host)
    nxt = int(prompt[0])
    for s in range(6):
        ologits, _ = ref.step(nxt)
        gpick = m.decode_step(nxt)
        check_position(m.logits().cpu().numpy(), ologits, gpu_pick=gpick, ora_pick=oracle.argmax(ologits),
                       what=f"step {s} after recovery")
        nxt = int(prompt[s + 1]) if s + 1 < len(prompt) else oracle.argmax(ologits)
    ref.close()
    m.close()
