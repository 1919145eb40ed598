"""Pins for the seeded input generator (PCG32, Box-Muller, bf16/f16 rounding, the Q8 quantiser)."""
import json
import os

import numpy as np
import pytest
import torch

import qw_inputs as qi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pcg32_python(seed, stream, n):
    """Arbitrary-precision restatement of the frozen transition, for the jump-ahead check."""
    M = 2 ** 64
    state, inc = 0, ((stream << 1) | 1) % M
    out = []

    def nxt():
        nonlocal state
        old = state
        state = (old * 6364136223846793005 + inc) % M
        xs = (((old >> 18) ^ old) >> 27) & 0xFFFFFFFF
        rot = old >> 59
        return ((xs >> rot) | (xs << ((32 - rot) & 31))) & 0xFFFFFFFF

    nxt()
    state = (state + seed) % M
    nxt()
    for _ in range(n):
        out.append(nxt())
    return out


def test_pcg32_published_vector():
    g = json.load(open(os.path.join(GOLDEN, "pcg32_vectors.json")))
    words = qi.pcg32_words(len(g["words_hex"]), g["seed"], g["stream"])
    assert [hex(int(w)) for w in words] == g["words_hex"]


def test_pcg32_jump_ahead_equals_sequential():
    seq = qi.pcg32_words(1000, 7, 3)
    assert list(seq) == _pcg32_python(7, 3, 1000)
    for skip in (1, 2, 17, 999):
        assert list(qi.pcg32_words(1, 7, 3, skip=skip)) == [int(seq[skip])]


def test_normal_thread_invariance_and_moments():
    a = qi.normal_bf16((1 << 20,), 11, 5, 1.0)
    b = qi.normal_bf16((1 << 20,), 11, 5, 1.0)
    np.testing.assert_array_equal(a, b)
    # the first elements come out of the single-thread path (n < 65536 pairs)
    small = qi.normal_bf16((1000,), 11, 5, 1.0)
    np.testing.assert_array_equal(small, a[:1000])
    f = qi.bf16_to_f32(a).astype(np.float64)
    assert abs(f.mean()) < 5e-3 and abs(f.std() - 1.0) < 5e-3
    # different streams differ
    assert not np.array_equal(qi.normal_bf16((64,), 11, 6, 1.0), a[:64])


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(20000).astype(np.float32) * 3
    ours = np.array([qi.f32_to_bf16_bits(float(v)) for v in x[:2000]], np.uint16)
    ref = torch.from_numpy(x[:2000]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(3000) * 1e-3, rng.standard_normal(1000) * 1e-6,
                           rng.standard_normal(1000) * 1e-8, rng.standard_normal(1000) * 6e4,
                           [0.0, -0.0, 65504.0, 65519.0, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])
    vals = vals.astype(np.float32)
    ours = np.array([qi.f32_to_f16_bits(float(v)) for v in vals], np.uint16)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_tokens_in_range_and_spread():
    t = qi.tokens(100000, 3, 151936)
    assert t.min() >= 0 and t.max() < 151936
    # distinct ids of n uniform draws from V: V * (1 - exp(-n/V)) in expectation
    expect = 151936 * (1 - np.exp(-100000 / 151936))
    assert abs(len(np.unique(t)) - expect) < 0.01 * expect


def test_quantiser_properties():
    w = qi.normal_bf16((64, 256), 9, 1, 0.02)
    w[3, 32:64] = 0  # an all-zero group
    q, s = qi.quantize_q8_g32(w)
    wf = qi.bf16_to_f32(w).reshape(64, 8, 32)
    sf = s.view(np.float16).astype(np.float32)
    qf = q.astype(np.float32).reshape(64, 8, 32)
    assert np.abs(q).max() <= 127
    assert sf[3, 1] == 0 and np.all(q[3, 32:64] == 0)
    nz = sf > 0
    # the group's largest magnitude maps to +-127 (up to the fp16 rounding of the scale)
    top = np.abs(qf).max(axis=2)
    assert np.all(top[nz] >= 126)
    # reconstruction error of each element is at most half a step (plus the clamp region)
    err = np.abs(qf * sf[:, :, None] - wf)
    assert np.all(err <= 0.5 * sf[:, :, None] * 1.0001 + 1e-12)


def test_make_weights_layout_and_determinism():
    wl = qi.WORKLOADS["tiny"]
    w1 = qi.make_weights(wl)
    assert w1["embed"].shape == (8192, 1024)
    assert len(w1["layers"]) == 2
    shapes = qi.tensor_shapes(wl)
    for name, shp in shapes.items():
        assert w1["layers"][0][name].shape == shp
    n = qi.bf16_to_f32(w1["layers"][1]["q_norm"])
    assert abs(n.mean() - 1.0) < 5e-3
    w2 = qi.make_weights(wl)
    np.testing.assert_array_equal(w1["layers"][1]["down"], w2["layers"][1]["down"])
