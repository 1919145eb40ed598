"""Batched decode (qw_batch_*): B sequences with their own prompts, caches and lengths, one
token each per step, against B independent oracle runs (teacher-forced with each oracle's
greedy picks).  Every position is held to the parity bar: the residual stream after each
layer, the logits and the greedy pick where the margin allows it.
"""
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


def _prompts(wl, B, base_len, seed):
    g = np.random.default_rng(seed)
    return [g.integers(0, wl.vocab, size=base_len + 3 * s).astype(np.int32) for s in range(B)]


def run_batch(qw, wl, B, base_len, n_steps, seed=7, max_ctx=None):
    host = qi.make_weights(wl)
    prompts = _prompts(wl, B, base_len, seed)
    n_ctx = max(len(p) for p in prompts) + n_steps + 1
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    m = qw.Model(wl, dev, max_ctx=max_ctx or n_ctx)
    m.set_debug(qw.DEBUG_HIDDEN)
    b = qw.Batch(m, B, n_ctx)
    refs = [oracle.OracleModel(wl, host, max_ctx=n_ctx) for _ in range(B)]
    nxt = []
    worst = {"logits_max_abs": 0.0, "hidden_rel_l2_max": 0.0}
    for s in range(B):
        ora = oracle.run_sequence(refs[s], prompts[s], 0)
        pick = b.prefill(s, prompts[s])
        if oracle.top2_margin(ora["logits"][0]) > 0.1:
            assert pick == ora["picks"][0], (s, pick, ora["picks"][0])
        nxt.append(ora["picks"][0])
    for step in range(n_steps):
        outs = [refs[s].step(nxt[s], want_hidden=True) for s in range(B)]
        picks = b.step(B, nxt)
        lg = b.logits().cpu().numpy()
        hid = b.debug_hidden().cpu().numpy()  # [L+1][B][H]
        for s in range(B):
            ologits, ohid = outs[s]
            st = check_position(lg[s], ologits, hid[:, s], ohid, picks[s], oracle.argmax(ologits),
                                what=f"B={B} sequence {s} step {step}")
            worst["logits_max_abs"] = max(worst["logits_max_abs"], st["logits_max_abs"])
            worst["hidden_rel_l2_max"] = max(worst["hidden_rel_l2_max"], st["hidden_rel_l2_max"])
            nxt[s] = oracle.argmax(ologits)
    for s in range(B):
        assert b.length(s) == refs[s].length
        refs[s].close()
    b.close()
    m.close()
    return worst


@pytest.mark.parametrize("B", [1, 2, 8])
def test_tiny_batch_matches_independent_sequences(qw, B):
    print(B, run_batch(qw, qi.WORKLOADS["tiny"], B, 5, 6))


def test_tiny_batch_long_sequences_many_splits(qw):
    # prompts of 118..124 tokens + 12 steps: the attention runs 4 splits of at most 32
    # positions, then 8 once the longest sequence passes 128 (a second captured graph)
    print(run_batch(qw, qi.WORKLOADS["tiny"], 3, 118, 12))


def test_tiny_batch_int8_weights(qw):
    print(run_batch(qw, qi.WORKLOADS["tiny"].with_(weight_format="int8_g32"), 3, 4, 4))


def test_full_shape_batch_of_eight(qw):
    print(run_batch(qw, qi.WORKLOADS["qwen3_0p6b_decode"], 8, 12, 3))


def test_batch_refusals(qw):
    wl = qi.WORKLOADS["tiny"]
    dev = qw.weights_to_device(qi.make_weights(wl), int8=False)
    m = qw.Model(wl, dev, max_ctx=16)
    with pytest.raises(qw.QwError):
        qw.Batch(m, qw.BATCH_MAX + 1, 16)
    with pytest.raises(qw.QwError):
        qw.Batch(m, 2, 17)  # longer than the model's context
    b = qw.Batch(m, 2, 8)
    with pytest.raises(qw.QwError) as e:
        b.step(2)  # no last token yet
    assert e.value.code == qw.INVALID_ARGUMENT
    with pytest.raises(qw.QwError) as e:
        b.step(3, [1, 2, 3])
    assert e.value.code == qw.INVALID_ARGUMENT
    b.prefill(0, [1, 2, 3, 4, 5, 6, 7])
    b.prefill(1, [3])
    b.step(2)  # sequence 0 reaches 8 = max_ctx
    with pytest.raises(qw.QwError) as e:
        b.step(2)
    assert e.value.code == qw.CONTEXT_EXCEEDED
    assert b.length(0) == 8 and b.length(1) == 2  # nothing appended by the refused step
    b.reset(0)
    assert b.length(0) == 0
    b.step(2, [5, -1])
    assert b.length(0) == 1 and b.length(1) == 3
    b.close()
    m.close()
