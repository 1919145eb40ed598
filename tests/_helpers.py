"""Shared test helpers: parity tolerances and GPU/oracle comparison."""
from __future__ import annotations

import numpy as np

# Parity bar for floating point (per position compared):
#   residual stream after each layer: relative L2 <= 2e-3
#   logits: max |gpu - oracle| <= 5e-2
#   greedy token identical wherever the oracle's top-2 margin exceeds 0.1
HIDDEN_REL_L2 = 2e-3
LOGITS_MAX_ABS = 5e-2
MARGIN = 0.1
# DIAGNOSTIC bar, used by one labelled diagnostic test only (never a workload's parity):
# a bf16 K/V cache on both sides (not one of the workloads' prefill configurations): each
# side rounds its own K/V rows to bf16, and an element whose two unrounded values straddle
# a rounding boundary ends one bf16 ulp (2^-8 relative) apart.  With only one side rounding
# the cache, the per-layer hidden error was measured at 2.6e-3 to 4.3e-3 on the tiny
# model, so twice the bar bounds the case where both round.
HIDDEN_REL_L2_BF16_KV = 4e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def top2_margin(logits) -> float:
    part = np.partition(np.asarray(logits, np.float64), -2)[-2:]
    return float(part[1] - part[0])


def check_position(gpu_logits, ora_logits, gpu_hidden=None, ora_hidden=None, gpu_pick=None, ora_pick=None,
                   what="", hidden_tol=HIDDEN_REL_L2):
    """Assert the parity bar at one position; returns a dict of the measured errors."""
    g = np.asarray(gpu_logits, np.float32)
    o = np.asarray(ora_logits, np.float32)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU logits"
    err = float(np.abs(g - o).max())
    out = {"logits_max_abs": err}
    assert err <= LOGITS_MAX_ABS, f"{what}: logits max-abs {err:.4g} > {LOGITS_MAX_ABS}"
    if gpu_hidden is not None and ora_hidden is not None:
        rels = [rel_l2(gh, oh) for gh, oh in zip(gpu_hidden, ora_hidden)]
        out["hidden_rel_l2_max"] = max(rels)
        bad = [(i, r) for i, r in enumerate(rels) if r > hidden_tol]
        assert not bad, f"{what}: hidden rel L2 above {hidden_tol} at (layer+1, value) {bad[:4]}"
    m = top2_margin(o)
    out["margin"] = m
    if gpu_pick is not None and ora_pick is not None and m > MARGIN:
        assert gpu_pick == ora_pick, f"{what}: greedy pick {gpu_pick} != oracle {ora_pick} (margin {m:.3f})"
    return out
