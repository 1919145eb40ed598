"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the fact it checks.  None re-types the oracle's own formula: the
expected values come from printed numbers (tests/golden), closed forms, invariants,
special cases that reduce to a library routine, or brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import qw_inputs as qi
from oracle import shapes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32_EPS = float(np.finfo(np.float32).eps)


def bf16(x) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def small_wl(**kw):
    base = dict(name="pin", seed=99, n_layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16,
                intermediate=96, vocab=48, prompt_len=0, decode_steps=8)
    base.update(kw)
    return qi.Workload(**base)


# ------------------------------------------------------------------ shape set

def test_tensor_set_matches_printed_counts():
    g = json.load(open(os.path.join(GOLDEN, "qwen3_0p6b_tensor_set.json")))
    d = g["dims"]
    ts = shapes.expected_tensors(d["vocab"], d["hidden"], d["n_layers"], d["n_heads"], d["n_kv_heads"],
                                 d["head_dim"], d["intermediate"])
    assert len(ts) == g["tensor_count"]
    stored, logical, emb = shapes.param_counts(ts)
    assert stored == g["params_stored"]
    assert logical == g["params_logical"]
    assert emb == g["params_embedding"]
    assert round(100.0 * emb / logical, 1) == g["embedding_share_percent"]
    layer0 = {n[len("model.layers.0."):]: s for n, s in ts if n.startswith("model.layers.0.")}
    assert {k: list(v) for k, v in layer0.items()} == g["layer0_shapes"]
    assert {k: shapes.numel(v) for k, v in layer0.items()} == g["layer0_params"]


def test_generated_weights_follow_the_tensor_set():
    wl = qi.WORKLOADS["qwen3_0p6b_decode"]
    ts = dict(shapes.expected_tensors(wl.vocab, wl.hidden, wl.n_layers, wl.n_heads, wl.n_kv_heads,
                                      wl.head_dim, wl.intermediate))
    names = {"input_norm": "input_layernorm", "q": "self_attn.q_proj", "k": "self_attn.k_proj",
             "v": "self_attn.v_proj", "q_norm": "self_attn.q_norm", "k_norm": "self_attn.k_norm",
             "o": "self_attn.o_proj", "post_norm": "post_attention_layernorm", "gate": "mlp.gate_proj",
             "up": "mlp.up_proj", "down": "mlp.down_proj"}
    for ours, theirs in names.items():
        assert qi.tensor_shapes(wl)[ours] == ts[f"model.layers.0.{theirs}.weight"]


def test_kv_cache_bytes_printed_value():
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_bytes.json")))
    assert shapes.kv_cache_bytes(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["ctx"],
                                 g["bytes_per_elem"]) == g["bytes"]


# -------------------------------------------------------------- conversions

def test_bf16_widening_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    ours = np.array([oracle.bf16_to_f32(int(b)) for b in bits[::7]], np.float32)
    r = ref[::7]
    fin = np.isfinite(r)
    np.testing.assert_array_equal(ours[fin], r[fin])
    assert np.all(np.isnan(ours[np.isnan(r)]))


def test_f16_widening_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    ours = np.array([oracle.f16_to_f32(int(b)) for b in bits], np.float32)
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])
    np.testing.assert_array_equal(np.signbit(ours[fin]), np.signbit(ref[fin]))
    assert np.all(np.isnan(ours[~fin]))


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_unit_weight_closed_form():
    rng = np.random.default_rng(0)
    for scale in (1e-2, 1.0, 30.0):
        x = (rng.standard_normal(1024) * scale).astype(np.float32)
        y = oracle.rmsnorm(x, None, 1e-6).astype(np.float64)
        ms = np.mean(x.astype(np.float64) ** 2)
        assert abs(math.sqrt(np.mean(y ** 2)) - math.sqrt(ms / (ms + 1e-6))) < 1e-5


def test_rmsnorm_eps_inside_the_root():
    # x = c everywhere: y = c / sqrt(c^2 + eps); with c^2 == eps this is 1/sqrt(2)
    x = np.full(1024, 1e-3, np.float32)
    y = oracle.rmsnorm(x, None, 1e-6)
    np.testing.assert_allclose(y, 1e-3 / math.sqrt(1e-6 + float(np.float32(1e-3)) ** 2), rtol=2e-6)
    np.testing.assert_allclose(y, 1 / math.sqrt(2), rtol=2e-6)


def test_rmsnorm_weight_is_elementwise_and_no_mean_centering():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(256) + 5.0).astype(np.float32)  # large mean: centering would change it
    w = bf16(rng.uniform(0.5, 2.0, 256))
    y1 = oracle.rmsnorm(x, None, 1e-6)
    yw = oracle.rmsnorm(x, w, 1e-6)
    np.testing.assert_allclose(yw, y1 * qi.bf16_to_f32(w), rtol=2 * F32_EPS)
    assert np.all(y1 > 0)  # no mean subtraction: all-positive input stays positive


# ---------------------------------------------------------------------- RoPE

THETA = 1e6


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(2).standard_normal(128).astype(np.float32)
    np.testing.assert_array_equal(oracle.rope(x, 0, THETA), x)


def test_rope_pairs_are_half_split_and_norm_preserving():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(128).astype(np.float32)
    for pos in (1, 7, 1000, 32767):
        y = oracle.rope(x, pos, THETA)
        n0 = np.hypot(x[:64].astype(np.float64), x[64:].astype(np.float64))
        n1 = np.hypot(y[:64].astype(np.float64), y[64:].astype(np.float64))
        np.testing.assert_allclose(n1, n0, rtol=4 * F32_EPS, atol=1e-7)
    # a one-hot at i moves only into i + d/2
    for i in (0, 5, 63):
        e = np.zeros(128, np.float32)
        e[i] = 1
        y = oracle.rope(e, 11, THETA)
        nz = set(np.nonzero(y)[0].tolist())
        assert nz <= {i, i + 64}


def test_rope_rotates_by_position_times_frequency():
    # the angle recovered from a rotated one-hot grows linearly in the position,
    # frequency 1 at i = 0 and a constant ratio theta^(-2/d) between neighbours
    d = 128
    e = np.zeros(d, np.float32)
    e[0] = 1
    for pos in (1, 2, 3):
        y = oracle.rope(e, pos, THETA)
        ang = math.atan2(float(y[64]), float(y[0]))
        assert abs(ang - math.remainder(pos, 2 * math.pi)) < 2e-7  # counter-clockwise, rate 1
    freqs = []
    for i in range(64):
        e = np.zeros(d, np.float32)
        e[i] = 1
        y = oracle.rope(e, 1, THETA)
        freqs.append(math.atan2(float(y[i + 64]), float(y[i])))
    ratios = np.array(freqs[1:]) / np.array(freqs[:-1])
    np.testing.assert_allclose(ratios, THETA ** (-2 / d), rtol=3e-6)
    # large positions: the angle is pos * frequency modulo 2 pi (slow pairs, measurable)
    for i in (40, 50, 63):
        e = np.zeros(d, np.float32)
        e[i] = 1
        pos = 32767
        y = oracle.rope(e, pos, THETA)
        got = math.atan2(float(y[i + 64]), float(y[i]))
        want = math.remainder(pos * freqs[i], 2 * math.pi)
        assert abs(got - want) < 1e-5


def test_rope_alternating_vector_at_large_position():
    # "Scalar-Native ..." section 9: alternating ones and zeros at a large position;
    # the fast (low-index) pairs change a lot, the slow (high-index) pairs barely move
    x = np.array([1.0, 0.0] * 64, np.float32)
    y = oracle.rope(x, 8191, THETA)
    moved = np.abs(y - x)
    assert moved[:8].max() > 0.5
    # slowest pair: angle 8191 * theta^(-126/128) ~ 0.01 rad
    assert moved[56:64].max() < 0.05 and moved[120:].max() < 0.05
    assert moved[62] < 0.013 and moved[126] < 0.013


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(128).astype(np.float32)
    k = rng.standard_normal(128).astype(np.float32)
    a = float(np.dot(oracle.rope(q, 10, THETA).astype(np.float64), oracle.rope(k, 3, THETA)))
    b = float(np.dot(oracle.rope(q, 1010, THETA).astype(np.float64), oracle.rope(k, 1003, THETA)))
    assert abs(a - b) < 1e-4


def test_qk_norm_precedes_rope():
    # one-hot pre-norm q with non-uniform norm weights: norm first scales the one-hot
    # by w_0 * sqrt(d); the rotation then splits it as (cos, sin).  Rotating first
    # would give (w_0 cos, w_64 sin) * sqrt(d) instead.
    d, pos = 128, 1
    w = np.ones(d, np.float32)
    w[:64] = 2.0
    wb = bf16(w)
    v = np.zeros(d, np.float32)
    v[0] = 3.0
    c, s = oracle.rope_angles(pos, d, THETA)
    tmp = np.empty(d, np.float32)
    import ctypes
    fp = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    oracle.lib().ora_qk_norm_rope.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_float, ctypes.POINTER(ctypes.c_float),
                                              ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    oracle.lib().ora_qk_norm_rope(fp(v), wb.ctypes.data, d, 1e-6, fp(c), fp(s), fp(tmp))
    mag = 2.0 * math.sqrt(d)
    # eps = 1e-6 against a mean square of 9/128 moves the magnitude by ~7e-6 relative
    assert abs(v[0] - mag * math.cos(1.0)) < 2e-5 * mag
    assert abs(v[64] - mag * math.sin(1.0)) < 2e-5 * mag
    assert np.count_nonzero(v) == 2


# ----------------------------------------------------------------- attention

def test_attention_single_position_returns_v0_exactly():
    rng = np.random.default_rng(5)
    q = rng.standard_normal(128).astype(np.float32) * 10
    K = rng.standard_normal((1, 128)).astype(np.float32)
    V = rng.standard_normal((1, 128)).astype(np.float32)
    np.testing.assert_array_equal(oracle.attention_head(q, K, V), V[0])


def test_attention_matches_softmax_brute_force():
    rng = np.random.default_rng(6)
    for n in (2, 5, 33):
        q = rng.standard_normal(16).astype(np.float32)
        K = rng.standard_normal((n, 16)).astype(np.float32)
        V = rng.standard_normal((n, 16)).astype(np.float32)
        s = (K.astype(np.float64) @ q.astype(np.float64)) / 4.0  # 1/sqrt(16)
        want = scipy.special.softmax(s) @ V.astype(np.float64)
        np.testing.assert_allclose(oracle.attention_head(q, K, V), want, rtol=1e-5, atol=1e-6)


def test_attention_shift_invariance_and_dominance():
    rng = np.random.default_rng(7)
    n, d = 9, 128
    q = rng.standard_normal(d).astype(np.float32)
    K = rng.standard_normal((n, d)).astype(np.float32)
    V = rng.standard_normal((n, d)).astype(np.float32)
    # adding u to every key with q.u = c adds the same constant to every score
    u = q / np.dot(q, q) * 3.0
    o1 = oracle.attention_head(q, K, V)
    o2 = oracle.attention_head(q, (K + u).astype(np.float32), V)
    np.testing.assert_allclose(o2, o1, rtol=1e-4, atol=1e-5)
    # one key aligned with a huge q dominates
    K2 = K.copy()
    K2[4] = q * 50
    np.testing.assert_allclose(oracle.attention_head(q, K2, V), V[4], atol=1e-6)
    # identical keys: uniform weights, the mean of V
    K3 = np.tile(K[0], (n, 1))
    np.testing.assert_allclose(oracle.attention_head(q, K3, V), V.astype(np.float64).mean(0), atol=2e-6)


def test_attention_rejects_empty_and_nonfinite():
    q = np.ones(4, np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.attention_head(q, np.zeros((0, 4), np.float32), np.zeros((0, 4), np.float32))
    K = np.ones((2, 4), np.float32)
    K[1, 0] = np.nan
    with pytest.raises(oracle.OracleError) as e:
        oracle.attention_head(q, K, np.ones((2, 4), np.float32))
    assert e.value.code == oracle.NUMERICAL_FAILURE


# ---------------------------------------------------------------------- SiLU

def test_silu_special_values_and_library():
    assert oracle.silu(0.0) == 0.0
    # section 9 "Adversarial SwiGLU": a negative gate leaks a small negative value
    for z in (-0.5, -3.0, -10.0, -20.0):
        assert oracle.silu(z) < 0
    assert -5e-4 < oracle.silu(-10.0) < -4e-4
    assert oracle.silu(40.0) == 40.0
    zs = np.linspace(-30, 30, 4001).astype(np.float32)
    got = np.array([oracle.silu(float(z)) for z in zs])
    want = zs.astype(np.float64) * scipy.special.expit(zs.astype(np.float64))
    np.testing.assert_allclose(got, want, rtol=4 * F32_EPS, atol=1e-30)


# ------------------------------------------------------------ dot / matvec

def test_matvec_orientation_one_hot_rows():
    # W is [out, in]: row n selects input column perm[n]; a transposed read fails this
    rows, cols = 5, 7
    perm = [6, 0, 3, 3, 1]
    W = np.zeros((rows, cols), np.float32)
    for n, k in enumerate(perm):
        W[n, k] = 1.0
    x = np.arange(1, cols + 1, dtype=np.float32) * 1.5
    np.testing.assert_array_equal(oracle.matvec(bf16(W), x), x[perm])


def test_matvec_accumulates_sequentially_in_k():
    # f32 sequential sum of (1e8, 1, -1e8, 1) is 1: the first +1 is absorbed, the last is not
    W = bf16(np.ones((1, 4)))
    x = np.array([1e8, 1.0, -1e8, 1.0], np.float32)
    assert oracle.matvec(W, x)[0] == 1.0


def test_matvec_against_float64():
    rng = np.random.default_rng(8)
    W = bf16(rng.standard_normal((64, 1024)) * 0.02)
    x = rng.standard_normal(1024).astype(np.float32)
    want = qi.bf16_to_f32(W).astype(np.float64) @ x.astype(np.float64)
    bound = 1024 * F32_EPS * (np.abs(qi.bf16_to_f32(W)).astype(np.float64) @ np.abs(x))
    assert np.all(np.abs(oracle.matvec(W, x) - want) <= bound)


def test_q8_block_extremes():
    # section 9 "Quantized Tails": one 32-element block, alternating +-127 codes
    q = np.array([[127, -127] * 16], np.int8)
    s_bits = np.array([[qi.f32_to_f16_bits(0.0078125)]], np.uint16)  # exactly representable scale
    ones = np.ones(32, np.float32)
    alt = np.array([1.0, -1.0] * 16, np.float32)
    assert oracle.matvec(q, ones, s_bits)[0] == 0.0
    assert oracle.matvec(q, alt, s_bits)[0] == 32 * 127 * 0.0078125
    # a subnormal fp16 scale still dequantises exactly (no flush to zero)
    tiny = np.array([[1]], np.uint16)  # 2^-24
    got = oracle.matvec(q, ones * 0 + np.float32(2.0 ** 20), tiny)[0]
    assert got == 0.0
    got = oracle.matvec(q, alt, tiny)[0]
    assert got == np.float32(32 * 127 * 2.0 ** -24)


def test_q8_dequant_is_exact_product():
    rng = np.random.default_rng(9)
    w = bf16(rng.standard_normal((16, 256)) * 0.02)
    q, s = qi.quantize_q8_g32(w)
    deq = q.astype(np.float64).reshape(16, 8, 32) * s.view(np.float16).astype(np.float64)[:, :, None]
    deq = deq.reshape(16, 256)
    # each dequantised weight is exactly representable in f32
    np.testing.assert_array_equal(deq.astype(np.float32).astype(np.float64), deq)
    x = rng.standard_normal(256).astype(np.float32)
    want = deq @ x.astype(np.float64)
    bound = 256 * F32_EPS * (np.abs(deq) @ np.abs(x.astype(np.float64)))
    assert np.all(np.abs(oracle.matvec(q, x, s) - want) <= bound)
    # storage: 32 int8 codes + one 2-byte scale = 34 bytes per 32 weights
    assert (q.nbytes + s.nbytes) * 32 == 34 * q.size


# ------------------------------------------------------------------- argmax

def test_argmax_ties_to_lowest_id_and_rejects_nonfinite():
    rng = np.random.default_rng(10)
    x = rng.standard_normal(1000).astype(np.float32)
    m = int(np.argmax(x))
    x[17] = x[m]
    x[900] = x[m]
    assert oracle.argmax(x) == min(17, m)
    assert oracle.argmax(np.full(5, -3.0, np.float32)) == 0
    for bad in (np.nan, np.inf, -np.inf):
        y = x.copy()
        y[500] = bad
        with pytest.raises(oracle.OracleError):
            oracle.argmax(y)


# ------------------------------------------------------------- whole model

def _model(wl, weights, **kw):
    return oracle.OracleModel(wl, weights, **kw)


def test_decode_equals_full_recomputation_bitwise():
    wl = qi.WORKLOADS["tiny"]
    w = qi.make_weights(wl)
    toks = list(qi.prompt(wl)) + [3, 4000, 8191]
    m = _model(wl, w)
    inc = np.stack([m.step(t)[0] for t in toks])
    full = m.full(toks)
    np.testing.assert_array_equal(inc, full)


def test_thread_count_does_not_change_results():
    wl = small_wl(n_layers=2)
    w = qi.make_weights(wl)
    a = _model(wl, w, nthreads=1)
    b = _model(wl, w, nthreads=7)
    for t in (1, 5, 9, 40):
        np.testing.assert_array_equal(a.step(t)[0], b.step(t)[0])


def test_gqa_equals_mha_with_duplicated_kv_heads():
    wl = small_wl(n_layers=2, n_heads=4, n_kv_heads=2)
    w = qi.make_weights(wl)
    g = wl.n_heads // wl.n_kv_heads
    d = wl.head_dim
    wl_mha = wl.with_(n_kv_heads=wl.n_heads)
    w_mha = {"embed": w["embed"], "final_norm": w["final_norm"], "layers": []}
    for lw in w["layers"]:
        nl = dict(lw)
        for m in ("k", "v"):
            heads = lw[m].reshape(wl.n_kv_heads, d, wl.hidden)
            nl[m] = np.ascontiguousarray(np.repeat(heads, g, axis=0).reshape(wl.n_heads * d, wl.hidden))
        w_mha["layers"].append(nl)
    a, b = _model(wl, w), _model(wl_mha, w_mha)
    for t in (3, 17, 0, 47, 22):
        np.testing.assert_array_equal(a.step(t)[0], b.step(t)[0])


def _structured(wl, seed=5):
    w = qi.make_weights(wl.with_(seed=seed))
    return w


def test_zero_output_projections_make_layers_identity():
    wl = small_wl(n_layers=3)
    w = _structured(wl)
    for lw in w["layers"]:
        lw["o"][:] = 0
        lw["down"][:] = 0
    m = _model(wl, w)
    for t in (2, 9, 30):
        _, hid = m.step(t, want_hidden=True)
        for l in range(wl.n_layers):
            np.testing.assert_array_equal(hid[l + 1], hid[0])
        np.testing.assert_array_equal(hid[0], qi.bf16_to_f32(w["embed"][t]))


def test_tied_head_picks_the_input_token_through_identity_layers():
    # with identity layers, logits[v] = E[v] . RMSNorm(E[t]); the self term is
    # sqrt(H)*|E[t]| ~ 20 against ~N(0, 0.64^2) for the others, so argmax == t
    wl = small_wl(n_layers=2, hidden=1024, vocab=512, n_heads=16, n_kv_heads=8, head_dim=64, intermediate=128)
    w = _structured(wl)
    for lw in w["layers"]:
        lw["o"][:] = 0
        lw["down"][:] = 0
    m = _model(wl, w)
    for t in (0, 77, 511):
        logits, _ = m.step(t)
        assert oracle.argmax(logits) == t


def test_position_zero_attention_ignores_queries_and_keys():
    # at position 0 the softmax has one term, so o = v_0 whatever q, k, QK-Norm and RoPE are
    wl = small_wl(n_layers=1)
    w1 = _structured(wl, seed=5)
    w2 = _structured(wl, seed=5)
    rng = np.random.default_rng(0)
    for name in ("q", "k", "q_norm", "k_norm"):
        w2["layers"][0][name] = bf16(rng.standard_normal(w2["layers"][0][name].shape))
    a, b = _model(wl, w1), _model(wl, w2)
    ha = a.step(7, want_hidden=True)[1]
    hb = b.step(7, want_hidden=True)[1]
    np.testing.assert_array_equal(ha, hb)
    ha = a.step(8, want_hidden=True)[1]
    hb = b.step(8, want_hidden=True)[1]
    assert not np.array_equal(ha[1], hb[1])


def test_gqa_head_routing():
    # "Scalar-Native ..." section 9: with 4 query heads and 2 KV heads, query heads 2 and 3
    # read KV head 1 only.  KV head 0 carries large positive values, KV head 1 large
    # negative ones; o_proj sums the outputs of query heads 2 and 3 into every x element.
    wl = small_wl(n_layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16)
    w = _structured(wl)
    lw = w["layers"][0]
    d, H = wl.head_dim, wl.hidden
    w["embed"][:] = bf16(np.ones((wl.vocab, H)))
    lw["input_norm"][:] = bf16(np.ones(H))
    V = np.zeros((wl.n_kv_heads * d, H), np.float32)
    V[:d] = 1000.0 / H      # v of KV head 0 = +1000 per element (h = 1)
    V[d:] = -1000.0 / H     # KV head 1 = -1000
    lw["v"][:] = bf16(V)
    O = np.zeros((H, wl.n_heads * d), np.float32)
    O[:, 2 * d:4 * d] = 1.0 / (2 * d)  # mean over heads 2 and 3
    lw["o"][:] = bf16(O)
    lw["down"][:] = 0
    m = _model(wl, w)
    for t in (1, 2, 3):
        _, hid = m.step(t, want_hidden=True)
        delta = hid[1] - hid[0]
        np.testing.assert_allclose(delta, -1000.0, rtol=1e-2)


def test_zero_gate_silences_the_mlp():
    wl = small_wl(n_layers=1)
    w = _structured(wl)
    w2 = _structured(wl)
    w["layers"][0]["gate"][:] = 0
    w2["layers"][0]["gate"][:] = 0
    w2["layers"][0]["down"][:] = 0
    a, b = _model(wl, w), _model(wl, w2)
    for t in (4, 5):
        np.testing.assert_array_equal(a.step(t, want_hidden=True)[1], b.step(t, want_hidden=True)[1])


def test_mlp_gate_takes_the_silu_and_up_scales_it():
    # "Scalar-Native ..." section 5: a = (gate * sigmoid(gate)) * up.  Build a layer whose
    # MLP input is the all-ones vector (embedding of ones, unit RMSNorm weights), whose gate
    # rows give g = -2 and up rows u = 3, and whose down projection copies a[j] to x[j]; the
    # attention contributes nothing (o_proj = 0).  Then x gains silu(-2) * 3 per element
    # (scipy's expit, not the oracle), while the swapped roles silu(3) * -2 differ by 8x.
    wl = small_wl(n_layers=1, hidden=64, intermediate=96)
    H, I = wl.hidden, wl.intermediate
    w = _structured(wl)
    lw = w["layers"][0]
    w["embed"][:] = bf16(np.ones((wl.vocab, H)))
    lw["input_norm"][:] = bf16(np.ones(H))
    lw["post_norm"][:] = bf16(np.ones(H))
    lw["o"][:] = 0
    lw["gate"][:] = bf16(np.full((I, H), -2.0 / H))
    lw["up"][:] = bf16(np.full((I, H), 3.0 / H))
    D = np.zeros((H, I), np.float32)
    D[np.arange(H), np.arange(H)] = 1.0
    lw["down"][:] = bf16(D)
    m = _model(wl, w)
    _, hid = m.step(3, want_hidden=True)
    delta = hid[1].astype(np.float64) - hid[0]
    h2 = 1.0 / math.sqrt(1.0 + wl.rms_eps)          # RMSNorm of the all-ones vector
    g, u = -2.0 * h2, 3.0 * h2
    want = g * scipy.special.expit(g) * u
    swapped = u * scipy.special.expit(u) * g
    np.testing.assert_allclose(delta, want, rtol=2e-6)
    assert abs(want - swapped) > 1.0


def _norm_routing_model(wl, q_first_half: bool):
    """A one-layer model where, at position 1, the query and the two keys are all-ones
    vectors before QK-Norm; q_norm keeps the first half of each head's dims, k_norm the
    second (or the other way round); v is -1 at position 0 and +1 at position 1; o_proj
    averages every head's output into each x element and the MLP is off."""
    H, d = wl.hidden, wl.head_dim
    w = _structured(wl)
    lw = w["layers"][0]
    E = np.ones((wl.vocab, H), np.float32)
    E[0, H // 2:] = -1.0                      # token 0: v = -1 ; token 1: v = +1
    w["embed"][:] = bf16(E)
    lw["input_norm"][:] = bf16(np.ones(H))
    first = np.zeros((1, H), np.float32)
    first[0, :H // 2] = 2.0 / H
    second = np.zeros((1, H), np.float32)
    second[0, H // 2:] = 2.0 / H
    lw["q"][:] = bf16(np.repeat(first, wl.n_heads * d, axis=0))
    lw["k"][:] = bf16(np.repeat(first, wl.n_kv_heads * d, axis=0))
    lw["v"][:] = bf16(np.repeat(second, wl.n_kv_heads * d, axis=0))
    half = np.r_[np.ones(d // 2), np.zeros(d // 2)].astype(np.float32)
    qn, kn = (half, half[::-1].copy()) if q_first_half else (half[::-1].copy(), half)
    lw["q_norm"][:] = bf16(qn)
    lw["k_norm"][:] = bf16(kn)
    lw["o"][:] = bf16(np.full((H, wl.n_heads * d), 1.0 / (wl.n_heads * d)))
    lw["down"][:] = 0
    return _model(wl, w)


def test_query_and_key_norms_route_and_keys_are_rotated():
    # QK-Norm then RoPE ("Scalar-Native ..." section 2 steps 3-4).  With q_norm on the first
    # half of the dims and k_norm on the second, each RoPE pair (i, i + d/2) holds q = (1, 0)
    # rotated by theta_i and k_0 = (0, 1) unrotated, k_1 = (0, 1) rotated by theta_i, so
    # s_0 = sum_i sin(theta_i) / sqrt(d) > 0 and s_1 = 0: the query prefers position 0 and the
    # layer adds p_1 - p_0 < 0.  Swapping which norm goes to queries and which to keys flips
    # the sign of s_0 (the layer adds a positive amount), and leaving the keys unrotated makes
    # s_1 = s_0 (the layer adds exactly 0).
    wl = small_wl(n_layers=1, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16)
    for q_first, sign in ((True, -1.0), (False, 1.0)):
        m = _norm_routing_model(wl, q_first)
        m.step(0)                               # position 0: token 0 (v = -1)
        _, hid = m.step(1, want_hidden=True)    # position 1: token 1 (v = +1)
        delta = hid[1].astype(np.float64) - hid[0]
        assert np.all(np.abs(delta - delta[0]) < 1e-6)
        assert sign * delta[0] > 0.01, (q_first, delta[0])


def test_context_overflow_leaves_length_unchanged():
    wl = small_wl(n_layers=1)
    w = _structured(wl)
    m = _model(wl, w, max_ctx=3)
    for t in (1, 2, 3):
        m.step(t)
    assert m.length == 3
    with pytest.raises(oracle.OracleError) as e:
        m.step(4)
    assert e.value.code == oracle.CONTEXT_EXCEEDED
    assert m.length == 3
    with pytest.raises(oracle.OracleError) as e:
        _model(wl, w).step(wl.vocab)
    assert e.value.code == oracle.INVALID_ARGUMENT


def test_kv_reset_and_import():
    wl = small_wl(n_layers=2)
    w = _structured(wl)
    m = _model(wl, w)
    a = [m.step(t)[0] for t in (5, 6, 7)]
    m.reset()
    assert m.length == 0
    b = [m.step(t)[0] for t in (5, 6, 7)]
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    # importing K/V planes then decoding matches attention over those planes
    k, v = qi.kv_fill(wl, 4)
    m.kv_import(k, v, 4)
    assert m.length == 4
    m.step(9)
    assert m.length == 5


def test_nonfinite_weights_are_rejected():
    wl = small_wl(n_layers=1)
    w = _structured(wl)
    w["layers"][0]["up"][3, 3] = 0x7F80  # +inf in bf16
    m = _model(wl, w)
    with pytest.raises(oracle.OracleError) as e:
        m.step(1)
    assert e.value.code == oracle.NUMERICAL_FAILURE
    assert m.length == 0


def test_int8_model_runs_and_matches_float64_dequant_on_one_row():
    wl = small_wl(n_layers=1, weight_format="int8_g32")
    w = qi.make_weights(wl)
    m = _model(wl, w)
    logits, hid = m.step(3, want_hidden=True)
    assert np.all(np.isfinite(logits))
    # the first projection's input is RMSNorm(E[3]); check q row 0 through the int8 matvec
    lw = w["layers"][0]
    h = oracle.rmsnorm(qi.bf16_to_f32(w["embed"][3]), lw["input_norm"], wl.rms_eps)
    q0 = oracle.matvec(lw["q_q8"], h, lw["q_s"])
    deq = lw["q_q8"].astype(np.float64).reshape(-1, wl.hidden // 32, 32) * \
        lw["q_s"].view(np.float16).astype(np.float64)[:, :, None]
    want = deq.reshape(-1, wl.hidden) @ h.astype(np.float64)
    np.testing.assert_allclose(q0, want, rtol=1e-4, atol=1e-6)
