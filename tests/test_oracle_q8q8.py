"""Pins of the oracle's Q8 x Q8 format (int8 g32 weights times activations quantized per 32-element
block at run time; "Real-Browser WASM Qwen3 Execution Under Honest Memory And Isolation Limits",
section 5 "Q8_0 Mixed-Precision Matrix Multiplication", and the "Integer-overflow rule" of
"Portable WebAssembly Runtime Architecture for TinyRustLM").  Each pin holds the oracle to
something other than its own formula: numpy's binary16 rounding, closed forms, exact integer
arithmetic, the quantization error bound."""
import numpy as np
import pytest

import oracle
import qw_inputs as qi


def test_f32_to_f16_matches_numpy_round_to_nearest_even():
    g = np.random.default_rng(3)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 6, 20000),
        np.float32([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                    2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, np.inf, -np.inf]),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, want)


def test_block_quantizer_rounds_halves_away_and_maps_amax_to_127():
    # amax 127 gives d = 1 exactly, so the codes are the values rounded: halves away from zero
    a = np.zeros(32, np.float32)
    a[:8] = [127, -2.5, 2.5, -0.5, 0.5, 1.5, -126.5, 3.49]
    q, s = oracle.quantize_q8_block(a)
    assert list(q[:8]) == [127, -3, 3, -1, 1, 2, -127, 3]
    assert s == 0x3C00  # fp16(1.0)
    # a negative extreme maps to -127; the scale is the fp16 rounding of amax / 127
    b = np.linspace(-3.0, 1.0, 32).astype(np.float32)
    q, s = oracle.quantize_q8_block(b)
    assert q.min() == -127 and q.max() <= 127 and q[0] == -127
    assert s == int(np.float16(np.float32(3.0) / np.float32(127.0)).view(np.uint16))
    # scaling the block by a power of two leaves the codes alone
    q2, _ = oracle.quantize_q8_block(b * np.float32(0.25))
    np.testing.assert_array_equal(q, q2)
    # an all-zero block: codes 0, scale 0, no division by zero
    q, s = oracle.quantize_q8_block(np.zeros(32, np.float32))
    assert not q.any() and s == 0


def test_block_dot_is_exact_i32_within_the_overflow_bound():
    # n * max|a| * max|w| = 32 * 127 * 127 = 516,128 <= 2^31 - 1: the i32 accumulator is safe
    assert 32 * 127 * 127 <= 2 ** 31 - 1
    assert oracle.q8_block_dot(np.full(32, 127), np.full(32, -127)) == -516128
    assert oracle.q8_block_dot(np.full(32, -127), np.full(32, -127)) == 516128
    g = np.random.default_rng(4)
    for _ in range(200):
        w = g.integers(-127, 128, 32)
        a = g.integers(-127, 128, 32)
        assert oracle.q8_block_dot(w, a) == int(np.dot(w.astype(np.int64), a.astype(np.int64)))


def test_q8q8_matvec_is_exact_for_integer_inputs():
    # activations already integers with a 127 in every block (d = 1) and unit weight scales:
    # the Q8 x Q8 product is the exact integer matrix-vector product
    g = np.random.default_rng(5)
    rows, cols = 24, 96
    w = g.integers(-127, 128, (rows, cols)).astype(np.int8)
    s = np.full((rows, cols // 32), 0x3C00, np.uint16)
    x = g.integers(-126, 127, cols).astype(np.float32)
    x[::32] = 127.0
    y = oracle.matvec(w, x, s, q8_act=True)
    np.testing.assert_array_equal(y, (w.astype(np.int64) @ x.astype(np.int64)).astype(np.float32))


def test_one_block_product_uses_the_fp16_activation_scale():
    # one row, one block: y = f32(isum) * (f32(s_w) * f32(fp16(amax / 127))); amax = 3 makes
    # amax / 127 inexact in fp16, so using the unrounded f32 scale would change y
    x = np.linspace(-3.0, 2.0, 32).astype(np.float32)
    q, sa = oracle.quantize_q8_block(x)
    assert float(np.float16(np.float32(3.0) / np.float32(127.0))) != float(np.float32(3.0) / np.float32(127.0))
    w = (np.arange(32) % 7 - 3).astype(np.int8).reshape(1, 32)
    sw = np.float16(0.0173).view(np.uint16).reshape(1, 1)
    y = oracle.matvec(w, x, sw, q8_act=True)
    isum = int(np.dot(w[0].astype(np.int64), q.astype(np.int64)))
    want = np.float32(isum) * (np.float32(sw.view(np.float16)[0, 0]) * np.float32(np.uint16(sa).view(np.float16)))
    assert y[0] == want


def test_q8q8_matvec_within_the_quantization_bound_of_the_f32_input_product():
    # each activation moves by at most d/2 of its block (fp16 scale rounding adds 2^-11 relative)
    g = np.random.default_rng(6)
    rows, cols = 32, 256
    w = g.integers(-127, 128, (rows, cols)).astype(np.int8)
    s = np.float16(g.uniform(0.001, 0.01, (rows, cols // 32))).view(np.uint16)
    x = (g.standard_normal(cols) * 2).astype(np.float32)
    y8 = oracle.matvec(w, x, s, q8_act=True).astype(np.float64)
    yf = oracle.matvec(w, x, s).astype(np.float64)
    wd = w.astype(np.float64) * np.repeat(s.view(np.float16).astype(np.float64), 32, axis=1)
    d = np.abs(x.reshape(-1, 32)).max(axis=1) / 127.0
    bound = (np.abs(wd) * np.repeat(d, 32) * (0.5 + 130 * 2.0 ** -11)).sum(axis=1) + 1e-5 * np.abs(wd @ x)
    assert np.all(np.abs(y8 - yf) <= bound)
    assert np.abs(y8 - yf).max() > 0  # the formats do differ


def test_q8q8_model_decode_equals_full_recomputation_and_stays_near_f32_activations():
    wl = qi.Workload(name="pin", seed=98, n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                     intermediate=96, vocab=48, prompt_len=0, decode_steps=8, weight_format="int8_g32",
                     act_format="q8")
    w = qi.make_weights(wl)
    m = oracle.OracleModel(wl, w)
    toks = [3, 17, 5, 40, 8, 8, 1]
    steps = np.stack([m.step(t)[0] for t in toks])
    m2 = oracle.OracleModel(wl, w)
    np.testing.assert_array_equal(m2.full(toks), steps)
    f = oracle.OracleModel(wl.with_(act_format="f32"), w)
    ref = np.stack([f.step(t)[0] for t in toks])
    assert not np.array_equal(ref, steps)
    assert np.abs(ref - steps).max() < 0.05 * np.abs(ref).max()
    for x in (m, m2, f):
        x.close()
