"""Per-phase timeline of one decode step (debug tracing of the persistent decode kernel).

Usage: python -m runtime_qwen3_decode_gb300.timeline [--workload NAME] [--pos P] [--json FILE]

Builds a model with seeded synthetic weights, imports a synthetic K/V cache of P
positions, runs a few decode steps with QW_DEBUG_TRACE and prints, per phase kind,
where the time goes: the wait for the previous phase (sync), the work, and how far
the producer's copies ran ahead.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

KINDS = ("qkv", "attn", "oproj", "gateup", "down")


def analyse(tr: np.ndarray, n_layers: int) -> dict:
    """tr: [phases, ctas, 8] int64 ns."""
    t0 = tr[0, :, 0].min()
    tr = tr.astype(np.float64) - t0
    out = {"step_us": float(tr[-1, :, 3].max() / 1e3)}
    rows = {k: {"sync_us": [], "work_med_us": [], "work_max_us": [], "crit_us": [], "lead_us": []}
            for k in KINDS + ("head",)}
    for ph in range(tr.shape[0]):
        kind = "head" if ph == 5 * n_layers else KINDS[ph % 5]
        t = tr[ph]
        prev_arrive = tr[ph - 1, :, 3].max() if ph else t[:, 0].min()
        rows[kind]["sync_us"].append((np.median(t[:, 1]) - prev_arrive) / 1e3)
        work = t[:, 2] - t[:, 1]
        rows[kind]["work_med_us"].append(np.median(work) / 1e3)
        rows[kind]["work_max_us"].append(work.max() / 1e3)
        rows[kind]["crit_us"].append((t[:, 3].max() - prev_arrive) / 1e3)
        issued = t[:, 4] > 0
        if issued.any():
            rows[kind]["lead_us"].append(float(np.median((t[issued, 1] - t[issued, 4]) / 1e3)))
    out["phases"] = {k: {m: float(np.mean(v)) if v else None for m, v in r.items()} | {"count": len(r["sync_us"])}
                     for k, r in rows.items()}
    return out


def main():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch

    import qw_inputs as qi
    from runtime_qwen3_decode_gb300 import build, qw

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3_0p6b_decode")
    ap.add_argument("--pos", type=int, default=128)
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--json", default=None)
    args = ap.parse_args()
    build.build()
    wl = qi.WORKLOADS[args.workload]
    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    del host
    m = qw.Model(wl, dev, max_ctx=args.pos + args.steps + 1)
    if args.pos:
        k, v = qi.kv_fill(wl, args.pos)
        m.kv_import(torch.from_numpy(k.view(np.int16)).cuda(), torch.from_numpy(v.view(np.int16)).cuda(), args.pos)
    m.set_debug(qw.DEBUG_TRACE)
    tok = qi.first_decode_token(wl)
    res = []
    for _ in range(args.steps):
        tok = m.decode_step(tok)
        tr = m.debug_trace().cpu().numpy()
        res.append(analyse(tr, wl.n_layers))
    last = res[-1]
    print(f"workload {wl.name}  pos {args.pos}  ctas {m.query(qw.QUERY_DECODE_CTAS)}  "
          f"step {last['step_us']:.1f} us")
    print(f"{'phase':8s} {'n':>3s} {'sync':>8s} {'work_med':>9s} {'work_max':>9s} {'crit':>8s} {'lead':>8s}  (us)")
    for k, r in last["phases"].items():
        print(f"{k:8s} {r['count']:3d} {r['sync_us']:8.2f} {r['work_med_us']:9.2f} {r['work_max_us']:9.2f} "
              f"{r['crit_us']:8.2f} {r['lead_us'] if r['lead_us'] is not None else float('nan'):8.2f}")
    if args.json:
        with open(args.json, "w") as f:
            json.dump({"workload": wl.name, "pos": args.pos, "steps": res}, f)


if __name__ == "__main__":
    main()
