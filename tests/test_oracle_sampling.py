"""Pins of the oracle's sampler ("Portable WebAssembly Runtime Architecture for TinyRustLM",
sections "Deterministic sampling contract" and "Sampling order"; repetition penalty of
"Scalar-Native Qwen3 Reference Runtime ...", section 7) against values fixed by the pages
and by the mathematics: the published PCG32 words, closed forms of the uniform draw,
greedy and tie cases, and the empirical distribution of many draws."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def u_of(word: int) -> float:
    return (word >> 8) * 2.0 ** -24


def test_draws_follow_the_published_pcg32_words():
    g = json.load(open(os.path.join(GOLDEN, "pcg32_vectors.json")))
    rng = oracle.pcg32_seed(g["seed"], g["stream"])
    for w in g["words_hex"]:
        # one candidate: the step still consumes one word, and reports its uniform
        tok, ids, cum, u = oracle.sample(np.zeros(1, np.float32), rng, 1.0)
        assert tok == 0 and u == u_of(int(w, 16))


def test_greedy_takes_the_lowest_id_on_ties_and_draws_nothing():
    x = np.array([0.5, 2.0, -1.0, 2.0], np.float32)
    rng = oracle.pcg32_seed(7, 1)
    before = rng.copy()
    tok, _, _, u = oracle.sample(x, rng, 0.0)
    assert tok == 1 and u == -1.0
    np.testing.assert_array_equal(rng, before)
    # -0 and +0 compare equal: the lower id wins
    tok, _, _, _ = oracle.sample(np.array([-1.0, 0.0, -0.0], np.float32)[[0, 2, 1]], rng, 0.0)
    assert tok == 1


def test_top_k_one_is_the_argmax_and_consumes_one_word():
    x = np.array([0.1, 0.9, 0.3, 0.9], np.float32)
    rng = oracle.pcg32_seed(3, 5)
    nxt = rng.copy()
    oracle.sample(np.zeros(1, np.float32), nxt, 1.0)  # the state after one word
    tok, ids, cum, _ = oracle.sample(x, rng, 0.8, top_k=1)
    assert tok == 1 and list(ids) == [1] and cum[0] == 1.0
    np.testing.assert_array_equal(rng, nxt)


def test_candidate_order_is_descending_value_then_ascending_id():
    x = np.array([1.0, 3.0, 3.0, 2.0, 3.0], np.float32)
    _, ids, _, _ = oracle.sample(x, oracle.pcg32_seed(1, 1), 1.0, top_k=4)
    assert list(ids) == [1, 2, 4, 3]


def test_repetition_penalty_divides_positive_and_multiplies_negative_once():
    x = np.array([2.0, -2.0, 1.0], np.float32)
    rng = oracle.pcg32_seed(1, 1)
    # penalty 2 on tokens 0 and 1: (1, -4, 1) -> tie between 0 and 2, lowest id
    assert oracle.sample(x, rng, 0.0, penalty=2.0, history=[0, 1])[0] == 0
    # penalty 4: (0.5, -8, 1) -> token 2; a token repeated in the history is penalised once
    assert oracle.sample(x, rng, 0.0, penalty=4.0, history=[0, 1, 0, 0])[0] == 2
    # a repeated negative logit moves further down: -1 * 2 = -2 < -1.5
    assert oracle.sample(np.array([-1.0, -1.5], np.float32), rng, 0.0, penalty=2.0, history=[0])[0] == 1
    # a zero logit is neither divided nor multiplied
    assert oracle.sample(np.array([0.0, -0.1], np.float32), rng, 0.0, penalty=9.0, history=[0, 1])[0] == 0
    with pytest.raises(oracle.OracleError):
        oracle.sample(x, rng, 1.0, penalty=0.0)


def test_nan_is_never_drawn_and_all_masked_is_an_error():
    x = np.array([np.nan, 0.0, np.nan, 0.0], np.float32)
    rng = oracle.pcg32_seed(11, 2)
    for _ in range(50):
        tok, ids, _, _ = oracle.sample(x, rng, 1.0)
        assert tok in (1, 3)
    with pytest.raises(oracle.OracleError):
        oracle.sample(np.full(4, -np.inf, np.float32), rng, 1.0)


def test_uniform_logits_pick_the_quantile_of_u():
    # four equal candidates: cumulative probabilities are exactly 1/4, 1/2, 3/4, 1, so
    # the draw picks candidate floor(4 u) of the id-ordered candidates
    x = np.zeros(9, np.float32)
    rng = oracle.pcg32_seed(99, 3)
    for _ in range(200):
        tok, ids, cum, u = oracle.sample(x, rng, 1.3, top_k=4)
        assert list(ids) == [0, 1, 2, 3]
        np.testing.assert_array_equal(cum, np.array([0.25, 0.5, 0.75, 1.0], np.float32))
        assert tok == int(np.floor(4 * u))


def test_top_p_keeps_the_minimal_prefix_reaching_p():
    x = np.zeros(2, np.float32)  # probabilities exactly 1/2, 1/2
    rng = oracle.pcg32_seed(5, 5)
    for _ in range(20):
        tok, ids, _, _ = oracle.sample(x, rng, 1.0, top_p=0.5)
        assert tok == 0 and list(ids) == [0]  # boundary equality keeps the prefix
    kept = set()
    for _ in range(200):
        tok, ids, _, _ = oracle.sample(x, rng, 1.0, top_p=float(np.nextafter(np.float32(0.5), np.float32(1))))
        assert list(ids) == [0, 1]
        kept.add(tok)
    assert kept == {0, 1}


def test_draw_frequencies_follow_the_tempered_softmax():
    rng_np = np.random.default_rng(0)
    x = rng_np.normal(size=6).astype(np.float32)
    T, n = 0.7, 40000
    p = np.exp((x.astype(np.float64) - x.max()) / T)
    p /= p.sum()
    rng = oracle.pcg32_seed(2024, 9)
    counts = np.zeros(6)
    for _ in range(n):
        counts[oracle.sample(x, rng, T)[0]] += 1
    sd = np.sqrt(n * p * (1 - p))
    assert np.all(np.abs(counts - n * p) < 5 * sd + 1), (counts, n * p)


def test_top_k_then_top_p_renormalise():
    rng_np = np.random.default_rng(1)
    x = rng_np.normal(size=50).astype(np.float32)
    T, k, top_p = 1.0, 10, 0.6
    order = sorted(range(50), key=lambda i: (-x[i], i))[:k]
    q = np.exp(x[order].astype(np.float64) - x[order[0]])
    q /= q.sum()
    m = int(np.searchsorted(np.cumsum(q), top_p - 1e-6)) + 1  # minimal prefix reaching p
    rng = oracle.pcg32_seed(8, 8)
    tok, ids, cum, _ = oracle.sample(x, rng, T, top_k=k, top_p=top_p)
    assert list(ids) == order[:m]
    assert abs(float(cum[-1]) - 1.0) < 1e-6
    np.testing.assert_allclose(cum, np.cumsum(q[:m] / q[:m].sum()), rtol=1e-5)
