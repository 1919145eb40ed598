"""GPU parity of on-device sampling (qw_sample_logits, qw_sample) against the oracle's sampler.

Both sides take the same seeded synthetic logits, history and PCG32 state.  The PCG32
state after every draw must match bit for bit, and so must the picked token.  The one
allowed exception is a draw u that falls within 1e-5 of a cumulative-probability
boundary of the oracle's retained candidates, or a top-p cut whose cumulative probability
lies within 1e-5 of top_p: the two sides compute exp in different libraries (a few ulp
apart), so there either neighbour of the boundary, or either cut, gives a correct pick.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402

pytestmark = pytest.mark.gpu

BOUNDARY = 1e-5


@pytest.fixture(scope="module")
def qw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw as binding
    build.build()
    return binding


def rng_tensor(state: np.ndarray):
    return torch.from_numpy(state.astype(np.uint64).view(np.int64).copy()).cuda()


def rng_host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


def top_p_alternatives(x, state_before, T, k, p, pen, hist, u):
    """Picks the oracle would make had its top-p cut kept one candidate more or fewer, for
    cuts whose cumulative probability lies within BOUNDARY of top_p (the two sides sum exp
    values from different libraries, so such a cut may fall on either side)."""
    if p >= 1.0:
        return set()
    st = state_before.copy()
    _, ids, cum, _ = oracle.sample(x, st, T, top_k=k, top_p=1.0, penalty=pen, history=hist)
    out = set()
    for n in range(1, len(ids) + 1):
        if abs(float(cum[n - 1]) - p) > BOUNDARY and not (n >= 2 and abs(float(cum[n - 2]) - p) <= BOUNDARY):
            continue
        z = float(cum[n - 1])
        j = next((i for i in range(n) if float(cum[i]) / z > u), n - 1)
        out.add(int(ids[j]))
    return out


def check_pick(gpu_tok, ora, what, alternatives=()):
    tok, ids, cum, u = ora
    if gpu_tok == tok:
        return 0
    if gpu_tok in alternatives:
        return 1
    near = [j for j in range(len(cum)) if abs(float(cum[j]) - u) <= BOUNDARY]
    assert near, f"{what}: GPU picked {gpu_tok}, oracle {tok} (u={u:.7f} not at a boundary)"
    j = near[0]
    assert gpu_tok in (int(ids[j]), int(ids[min(j + 1, len(ids) - 1)])), what
    return 1


@pytest.mark.parametrize("V", [100, 8192, 151936])
@pytest.mark.parametrize("params", [
    (0.0, 1, 1.0, 1.0),
    (1.0, 1, 1.0, 1.0),
    (0.7, 40, 1.0, 1.0),
    (1.0, 64, 0.9, 1.0),
    (1.5, 20, 0.5, 1.3),
    (0.8, 64, 1.0, 1.1),
])
def test_sample_logits_matches_oracle(qw, V, params):
    T, k, p, pen = params
    g = np.random.default_rng(V * 31 + int(T * 10) + k)
    sp = qw.Sampling(T, k, p, pen)
    state = oracle.pcg32_seed(1234 + V, k)
    rng = rng_tensor(state)
    tok = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    scratch = torch.empty(qw.lib().qw_sample_scratch_bytes(V), dtype=torch.uint8, device="cuda")
    boundary = 0
    for step in range(25):
        x = (g.standard_normal(V) * 2.0).astype(np.float32)
        hist = g.integers(0, V, size=int(g.integers(0, 40))).astype(np.int32)
        before = state.copy()
        ora = oracle.sample(x, state, T, top_k=k, top_p=p, penalty=pen, history=hist)
        qw.sample_logits(torch.from_numpy(x).cuda(), sp, rng, tok,
                         history=torch.from_numpy(hist).cuda() if hist.size else None, scratch=scratch)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(rng_host(rng), state)  # one word per sampled step, none for greedy
        got = int(tok.item())
        alt = top_p_alternatives(x, before, T, k, p, pen, hist, ora[3]) if got != ora[0] else set()
        boundary += check_pick(got, ora, f"V={V} {params} step {step}", alt)
    assert boundary <= 2


def test_sample_edge_cases(qw):
    V = 4096
    sp = qw.Sampling(1.0, 8, 1.0, 1.0)
    state = oracle.pcg32_seed(5, 5)
    rng = rng_tensor(state)
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    # NaN logits are never drawn
    x = np.full(V, np.nan, np.float32)
    x[[10, 700, 3000]] = 0.0
    for _ in range(20):
        qw.sample_logits(torch.from_numpy(x).cuda(), sp, rng, tok)
        assert int(tok.item()) in (10, 700, 3000)
    # every logit masked: no token
    qw.sample_logits(torch.full((V,), float("-inf"), device="cuda"), sp, rng, tok)
    assert int(tok.item()) == -1
    # a history id outside the vocabulary: no token
    bad = torch.tensor([1, V + 5], dtype=torch.int32, device="cuda")
    qw.sample_logits(torch.zeros(V, device="cuda"), qw.Sampling(1.0, 8, 1.0, 1.2), rng, tok, history=bad)
    assert int(tok.item()) == -1
    # greedy: ties (including -0 against +0) go to the lowest id
    y = np.full(V, -1.0, np.float32)
    y[900] = 0.0
    y[77] = -0.0
    qw.sample_logits(torch.from_numpy(y).cuda(), qw.Sampling(0.0, 1, 1.0, 1.0), rng, tok)
    assert int(tok.item()) == 77


def test_sample_rejects_bad_parameters(qw):
    V = 256
    rng = rng_tensor(oracle.pcg32_seed(1, 1))
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.zeros(V, device="cuda")
    for params in [(1.0, 0, 1.0, 1.0), (1.0, 65, 1.0, 1.0), (1.0, 8, 0.0, 1.0), (1.0, 8, 1.5, 1.0),
                   (1.0, 8, 1.0, 0.0), (-1.0, 8, 1.0, 1.0), (float("nan"), 8, 1.0, 1.0)]:
        with pytest.raises(qw.QwError) as e:
            qw.sample_logits(x, qw.Sampling(*params), rng, tok)
        assert e.value.code == qw.INVALID_ARGUMENT, params


def test_model_sampler_feeds_decode(qw):
    import qw_inputs as qi
    wl = qi.WORKLOADS["tiny"]
    dev = qw.weights_to_device(qi.make_weights(wl), int8=False)
    m = qw.Model(wl, dev)
    greedy = m.prefill(qi.prompt(wl))
    # temperature 0 is the model's own greedy pick
    assert m.sample(qw.Sampling(0.0, 1, 1.0, 1.0)) == greedy
    m.sampler_seed(42, 54)
    st = m.sampler_state()
    np.testing.assert_array_equal(np.array(st, np.uint64), oracle.pcg32_seed(42, 54))
    # the model-bound call equals the standalone call on the same logits and state
    sp = qw.Sampling(0.9, 32, 0.95, 1.2)
    hist = torch.from_numpy(qi.prompt(wl).astype(np.int32)).cuda()
    rng = rng_tensor(np.array(st, np.uint64))
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    qw.sample_logits(m.logits(), sp, rng, tok, history=hist)
    picked = m.sample(sp, history=hist)
    assert picked == int(tok.item())
    assert tuple(int(v) for v in rng_host(rng)) == m.sampler_state()
    # decode_step(-1) consumes the sampled token: same logits as feeding it explicitly
    m.decode_step(-1, want_token=False)
    a = m.logits().cpu().numpy()
    m2 = qw.Model(wl, dev)
    m2.prefill(qi.prompt(wl))
    m2.decode_step(picked, want_token=False)
    np.testing.assert_array_equal(a, m2.logits().cpu().numpy())
    m.close()
    m2.close()
