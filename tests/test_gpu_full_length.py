"""Parity against the oracle at each full-size workload's own length (slow: minutes of CPU).

Every workload runs the path its bench line times: the batched prefill of the whole prompt
(or the imported cache), then every decode step of the workload, teacher-forced with the
oracle's greedy picks so both sides stay position-aligned.  At every position: residual
stream after each layer (relative L2), logits (max-abs), and the greedy pick where the
oracle's top-2 margin exceeds 0.1.  The prefill workload also compares every K/V row its
2048-row prompt appends.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import qw_inputs as qi  # noqa: E402
from _helpers import check_position, rel_l2  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# Per (layer, KV head) plane of appended K or V rows: the prefill projections see
# fp16-rounded activations (relative rounding 2^-11), so a plane agrees to a few 1e-4.
KV_PLANE_REL_L2 = 2e-3


@pytest.fixture(scope="module")
def qw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from runtime_qwen3_decode_gb300 import build, qw as binding
    build.build()
    return binding


def _kv_planes(m, ref, wl, n):
    """Worst relative L2 over the (layer, KV head) planes of the first n cache rows."""
    ke, ve = m.kv_export(n)
    ke, ve = ke.float().cpu().numpy(), ve.float().cpu().numpy()
    worst = 0.0
    for l in range(wl.n_layers):
        for h in range(wl.n_kv_heads):
            ko = np.empty((n, wl.head_dim), np.float32)
            vo = np.empty_like(ko)
            for p in range(n):
                ko[p], vo[p] = ref.kv_row(l, h, p)
            for got, want, what in ((ke[l, h], ko, "K"), (ve[l, h], vo, "V")):
                r = rel_l2(got, want)
                worst = max(worst, r)
                assert r <= KV_PLANE_REL_L2, f"{what} layer {l} head {h}: rel L2 {r:.3g}"
    return worst


def _run_workload(qw, wl, check_kv=False):
    host = qi.make_weights(wl)
    n_ctx = wl.kv_prefill + wl.prompt_len + wl.decode_steps
    ref = oracle.OracleModel(wl, host, max_ctx=n_ctx + 1)
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    del host
    m = qw.Model(wl, dev, max_ctx=n_ctx + 1)
    m.set_debug(qw.DEBUG_HIDDEN)
    worst = {"logits_max_abs": 0.0, "hidden_rel_l2_max": 0.0, "positions": 0}

    def note(st):
        worst["logits_max_abs"] = max(worst["logits_max_abs"], st["logits_max_abs"])
        worst["hidden_rel_l2_max"] = max(worst["hidden_rel_l2_max"], st.get("hidden_rel_l2_max", 0.0))
        worst["positions"] += 1

    if wl.kv_prefill:
        k, v = qi.kv_fill(wl, wl.kv_prefill)
        ref.kv_import(k, v, wl.kv_prefill)
        m.kv_import(torch.from_numpy(k.view(np.int16)).cuda(), torch.from_numpy(v.view(np.int16)).cuda(),
                    wl.kv_prefill)
        del k, v
    if wl.prompt_len:
        prompt = qi.prompt(wl)
        ora = oracle.run_sequence(ref, prompt, 0, want_hidden=True)
        pick = m.prefill(prompt)
        note(check_position(m.logits().cpu().numpy(), ora["logits"][0], m.debug_hidden().cpu().numpy(),
                            ora["hidden"][0], pick, ora["picks"][0], what=f"{wl.name} prefill last row"))
        if check_kv:
            worst["kv_plane_rel_l2_max"] = _kv_planes(m, ref, wl, wl.prompt_len)
        nxt = ora["picks"][0]
    else:
        nxt = qi.first_decode_token(wl)
    for s in range(wl.decode_steps):
        ologits, ohid = ref.step(nxt, want_hidden=True)
        opick = oracle.argmax(ologits)
        gpick = m.decode_step(nxt)
        note(check_position(m.logits().cpu().numpy(), ologits, m.debug_hidden().cpu().numpy(), ohid, gpick, opick,
                            what=f"{wl.name} decode step {s}"))
        nxt = opick
    assert m.kv_length == ref.length == n_ctx
    m.close()
    ref.close()
    return worst


def test_decode_workload_128_prompt_384_steps(qw):
    print(_run_workload(qw, qi.WORKLOADS["qwen3_0p6b_decode"]))


def test_prefill_workload_2048_rows_then_16_steps(qw):
    print(_run_workload(qw, qi.WORKLOADS["qwen3_0p6b_prefill2048"], check_kv=True))


def test_long_context_workload_32k_cache_64_steps(qw):
    print(_run_workload(qw, qi.WORKLOADS["qwen3_0p6b_ctx32k"]))


def test_int8_workload_256_prompt_768_steps(qw):
    print(_run_workload(qw, qi.WORKLOADS["qwen3_0p6b_int8"]))
