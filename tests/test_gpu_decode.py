"""GPU parity of the decode path (C ABI) against the CPU oracle, teacher-forced.

Both sides consume the same seeded inputs; the GPU is fed the oracle's tokens so the
comparison stays position-aligned even where greedy picks would diverge at tiny margins.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import qw_inputs as qi  # noqa: E402
from _helpers import HIDDEN_REL_L2, LOGITS_MAX_ABS, MARGIN, check_position, rel_l2, top2_margin  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw as binding
    build.build()
    return binding


def _run_parity(qw, wl, n_prompt, n_decode, check_hidden=True, by_token=False, host=None, kv=None):
    host = host if host is not None else qi.make_weights(wl)
    ref = oracle.OracleModel(wl, host)
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    m = qw.Model(wl, dev)
    if kv is not None:
        k, v, n = kv
        ref.kv_import(k, v, n)
        m.kv_import(torch.from_numpy(k.view(np.int16)).cuda(), torch.from_numpy(v.view(np.int16)).cuda(), n)
    flags = qw.DEBUG_HIDDEN | (qw.DEBUG_PREFILL_BY_TOKEN if by_token else 0)
    m.set_debug(flags)
    prompt = qi.prompt(wl)[:n_prompt]
    stats = []
    if n_prompt:
        ora = oracle.run_sequence(ref, prompt, 0, want_hidden=True)
        pick = m.prefill(prompt)
        gh = m.debug_hidden().cpu().numpy() if (check_hidden and by_token) else None
        stats.append(check_position(m.logits().cpu().numpy(), ora["logits"][0], gh,
                                    ora["hidden"][0] if gh is not None else None, pick, ora["picks"][0],
                                    what="prefill last row"))
        nxt = ora["picks"][0]
    else:
        nxt = qi.first_decode_token(wl)
    for s in range(n_decode):
        ologits, ohid = ref.step(nxt, want_hidden=True)
        opick = oracle.argmax(ologits)
        gpick = m.decode_step(nxt)
        gh = m.debug_hidden().cpu().numpy() if check_hidden else None
        stats.append(check_position(m.logits().cpu().numpy(), ologits, gh, ohid if check_hidden else None, gpick,
                                    opick, what=f"decode step {s}"))
        nxt = opick
    assert m.kv_length == ref.length
    m.close()
    return stats


def test_tiny_prefill_and_decode(qw):
    wl = qi.WORKLOADS["tiny"]
    stats = _run_parity(qw, wl, wl.prompt_len, wl.decode_steps, by_token=True)
    print(stats)


def test_tiny_ragged_positions_cross_split_boundaries(qw):
    # positions 0..300 exercise 1, 2 and 3 attention splits and ragged 32-row chunks
    wl = qi.WORKLOADS["tiny"].with_(prompt_len=300, decode_steps=4)
    _run_parity(qw, wl, 300, 4, by_token=True)


def test_tiny_bf16_cache_long_import(qw):
    # bf16 cache over 3000 imported rows plus 8 new ones
    wl = qi.WORKLOADS["tiny"].with_(prompt_len=0, kv_prefill=3000, decode_steps=8, kv_format="bf16")
    k, v = qi.kv_fill(wl, 3000)
    _run_parity(qw, wl, 0, 8, kv=(k, v, 3000))


def test_full_shape_decode_config(qw):
    wl = qi.WORKLOADS["qwen3_0p6b_decode"]
    stats = _run_parity(qw, wl, wl.prompt_len, 4, by_token=True)
    print(stats)


def test_full_shape_int8(qw):
    wl = qi.WORKLOADS["qwen3_0p6b_int8"]
    stats = _run_parity(qw, wl, 32, 4, by_token=True)
    print(stats)


def test_long_context_32k_decode(qw):
    # bf16 cache (the workload's format): imported rows are exact, only new rows round
    wl = qi.WORKLOADS["qwen3_0p6b_ctx32k"]
    k, v = qi.kv_fill(wl, wl.kv_prefill)
    stats = _run_parity(qw, wl, 0, 3, kv=(k, v, wl.kv_prefill))
    print(stats)


def test_greedy_device_loop_matches_stepwise(qw):
    wl = qi.WORKLOADS["tiny"].with_(decode_steps=12)
    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=False)
    prompt = qi.prompt(wl)
    a = qw.Model(wl, dev)
    first = a.prefill(prompt)
    picks = [first]
    for _ in range(8):
        picks.append(a.decode_step(-1))
    b = qw.Model(wl, dev)
    b.prefill(prompt, want_token=False)
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    b.generate(8, -1, out)
    b.sync()
    assert out.cpu().tolist() == picks[1:]
    # same inputs, same bits
    np.testing.assert_array_equal(a.logits().cpu().numpy(), b.logits().cpu().numpy())


@pytest.mark.parametrize("kv_format", ["f32", "bf16"])
def test_kv_cache_indexing_bit_exact(qw, kv_format):
    wl = qi.WORKLOADS["tiny"].with_(decode_steps=0, prompt_len=0, kv_prefill=37, kv_format=kv_format)
    host = qi.make_weights(wl)
    k, v = qi.kv_fill(wl, 37)
    dev = qw.weights_to_device(host, int8=False)
    m = qw.Model(wl, dev, max_ctx=64)
    m.kv_import(torch.from_numpy(k.view(np.int16)).cuda(), torch.from_numpy(v.view(np.int16)).cuda(), 37)
    m.decode_step(5)
    ke, ve = m.kv_export(38)
    ke, ve = ke.float().cpu().numpy(), ve.float().cpu().numpy()
    # imported rows come back bit for bit (an f32 cache holds their exact widening)
    np.testing.assert_array_equal(ke[:, :, :37], qi.bf16_to_f32(k))
    np.testing.assert_array_equal(ve[:, :, :37], qi.bf16_to_f32(v))
    # the appended position holds this step's key/value at [l][kvh][37]: compare with the oracle's
    ref = oracle.OracleModel(wl, host, max_ctx=64)
    ref.kv_import(k, v, 37)
    ref.step(5)
    ko, vo = oracle_kv(ref, wl, 37)
    tol = 1e-4 if kv_format == "f32" else 1e-2
    np.testing.assert_allclose(ke[:, :, 37], ko, rtol=tol, atol=tol)
    np.testing.assert_allclose(ve[:, :, 37], vo, rtol=tol, atol=tol)


def oracle_kv(ref, wl, pos):
    k = np.stack([np.stack([ref.kv_row(l, h, pos)[0] for h in range(wl.n_kv_heads)]) for l in range(wl.n_layers)])
    v = np.stack([np.stack([ref.kv_row(l, h, pos)[1] for h in range(wl.n_kv_heads)]) for l in range(wl.n_layers)])
    return k, v


def test_argmax_ties_break_to_lowest_id(qw):
    # identity layers: logits[v] = E[v] . RMSNorm(E[t]) peaks at v = t; copies of row t
    # at a lower and a higher id tie bit for bit, and the lowest id must win
    wl = qi.WORKLOADS["tiny"].with_(vocab=4096)
    host = qi.make_weights(wl)
    for lw in host["layers"]:
        lw["o"][:] = 0
        lw["down"][:] = 0
    t = 1000
    host["embed"][700] = host["embed"][t]
    host["embed"][3000] = host["embed"][t]
    dev = qw.weights_to_device(host, int8=False)
    m = qw.Model(wl, dev, max_ctx=8)
    assert m.decode_step(t) == 700
    lg = m.logits().cpu().numpy()
    assert lg[700] == lg[t] == lg[3000]


def test_context_exceeded_leaves_state(qw):
    wl = qi.WORKLOADS["tiny"]
    dev = qw.weights_to_device(qi.make_weights(wl), int8=False)
    m = qw.Model(wl, dev, max_ctx=4)
    m.prefill([1, 2, 3])
    m.decode_step(-1)
    assert m.kv_length == 4
    with pytest.raises(qw.QwError) as e:
        m.decode_step(-1)
    assert e.value.code == qw.CONTEXT_EXCEEDED
    with pytest.raises(qw.QwError) as e:
        m.prefill([1])
    assert e.value.code == qw.CONTEXT_EXCEEDED
    assert m.kv_length == 4
    with pytest.raises(qw.QwError) as e:
        m.decode_step(wl.vocab)
    assert e.value.code == qw.INVALID_ARGUMENT
    m.kv_reset()
    assert m.kv_length == 0
    with pytest.raises(qw.QwError) as e:
        m.decode_step(-1)  # no previous pick after a reset
    assert e.value.code == qw.INVALID_ARGUMENT


def test_nonfinite_logits_reported(qw):
    wl = qi.WORKLOADS["tiny"]
    host = qi.make_weights(wl)
    host["embed"][17, 5] = 0x7F80  # +inf in the tied head row 17
    dev = qw.weights_to_device(host, int8=False)
    m = qw.Model(wl, dev, max_ctx=8)
    with pytest.raises(qw.QwError) as e:
        m.decode_step(3)
    assert e.value.code == qw.NUMERICAL_FAILURE
    with pytest.raises(qw.QwError):
        m.decode_step(3, want_token=False)
    m.kv_reset()


# Q8 x Q8 (int8 weights times per-block int8 activations).  Floating point decides every
# activation code, and the two sides accumulate in different orders, so a value within an ulp
# of a rounding boundary can take the neighbouring code on one side; such a flip moves its block
# by one quantization step and later layers amplify it.  So: where the quantizer's inputs are
# (nearly) identical, the first layer of position 0, the GPU must match the oracle's Q8 x Q8
# arithmetic to a few flips; over a whole sequence it must stay within the quantization noise
# itself, measured per position as the oracle's own distance between Q8 x Q8 and f32
# activations (and never looser than the f32-activation bar).


def test_q8q8_first_layer_matches_the_oracle(qw):
    wl = qi.WORKLOADS["tiny"].with_(weight_format="int8_g32", act_format="q8")
    host = qi.make_weights(wl)
    ref = oracle.OracleModel(wl, host)
    m = qw.Model(wl, qw.weights_to_device(host, int8=True))
    m.set_debug(qw.DEBUG_HIDDEN)
    errs = []
    for tok in range(0, 8192, 129):
        ref.reset()
        m.kv_reset()
        _, oh = ref.step(tok, want_hidden=True)
        m.decode_step(tok)
        gh = m.debug_hidden().cpu().numpy()
        errs.append(rel_l2(gh[1], oh[1]))
    errs = np.array(errs)
    # without a flip the two agree to float rounding; a flip (about one in ten tokens here) moves
    # the layer by one quantization step of one element, up to ~1e-2 for this model's layer 0
    assert np.median(errs) <= 1e-5, np.sort(errs)
    assert np.mean(errs > 1e-5) <= 0.3, np.sort(errs)
    assert errs.max() <= 2e-2, np.sort(errs)
    print(np.median(errs), np.mean(errs > 1e-5), errs.max())
    m.close()


def _q8q8_sequence(qw, wl, n_prompt, n_decode, one_group=False):
    host = qi.make_weights(wl)
    n_ctx = n_prompt + n_decode + 1
    q8 = oracle.OracleModel(wl, host, max_ctx=n_ctx)
    f32 = oracle.OracleModel(wl.with_(act_format="f32"), host, max_ctx=n_ctx)
    m = qw.Model(wl, qw.weights_to_device(host, int8=True), max_ctx=n_ctx)
    m.set_debug(qw.DEBUG_HIDDEN | (qw.DEBUG_ONE_GROUP if one_group else 0))
    toks = [int(t) for t in np.random.default_rng(11).integers(0, wl.vocab, n_prompt)]
    worst = {"hidden_ratio": 0.0, "logits_ratio": 0.0}
    nxt = toks[0]
    for pos in range(n_prompt + n_decode):
        tok = toks[pos] if pos < n_prompt else nxt
        lq, hq = q8.step(tok, want_hidden=True)
        lf, hf = f32.step(tok, want_hidden=True)
        gpick = m.decode_step(tok)
        gl, gh = m.logits().cpu().numpy(), m.debug_hidden().cpu().numpy()
        for layer in range(1, len(hq)):
            noise = rel_l2(hq[layer], hf[layer])
            err = rel_l2(gh[layer], hq[layer])
            assert err <= max(HIDDEN_REL_L2, 1.5 * noise), (pos, layer, err, noise)
            worst["hidden_ratio"] = max(worst["hidden_ratio"], err / max(noise, 1e-12))
        lnoise = float(np.abs(lq - lf).max())
        lerr = float(np.abs(gl - lq).max())
        assert lerr <= max(LOGITS_MAX_ABS, 1.5 * lnoise), (pos, lerr, lnoise)
        worst["logits_ratio"] = max(worst["logits_ratio"], lerr / max(lnoise, 1e-12))
        if top2_margin(lq) > 2 * lnoise + MARGIN:
            assert gpick == oracle.argmax(lq), (pos, gpick)
        nxt = oracle.argmax(lq)
    m.close()
    return worst


def test_tiny_q8q8_sequence_within_quantization_noise(qw):
    wl = qi.WORKLOADS["tiny"].with_(weight_format="int8_g32", act_format="q8")
    print(_q8q8_sequence(qw, wl, 24, 16))


def test_full_shape_q8q8_sequence_within_quantization_noise(qw):
    print(_q8q8_sequence(qw, qi.WORKLOADS["qwen3_0p6b_int8"].with_(act_format="q8"), 12, 4))


def test_q8q8_one_group_layout(qw):
    # the one-group layout runs o_proj and down through the k-split core
    wl = qi.WORKLOADS["tiny"].with_(weight_format="int8_g32", act_format="q8")
    print(_q8q8_sequence(qw, wl, 8, 4, one_group=True))
