"""Benchmark: batch-1 decode tokens/s of the Qwen3-0.6B-shape decoder on one GB300.

Workload (default "qwen3_0p6b_decode"): full Qwen3-0.6B shape, random-init bf16
weights from the seeded generator, a 128-token uniform-random prompt prefilled, then
greedy decode.  One timed step = one decode token (one pass of the whole decode hot
path: embedding gather, 28 layers, final norm, tied lm_head, argmax).  Inputs are
resident in HBM before the timed region; the 1.19 GB of weights streamed per token
are larger than L2, so no flush is needed between steps.

Output: one JSON line (rank 0).  `--impl reference` times the CPU oracle instead
(the reference arm: the plain fp32 restatement of the same forward on host cores).
Multi-GPU runs (torchrun) are independent replicas, one sequence per GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import qw_inputs as qi  # noqa: E402

METRIC = "batch-1 decode tokens/s (Qwen3-0.6B shape); achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 7900.0


# ------------------------------------------------------------------ byte model

def weight_bytes(wl) -> int:
    """Bytes of weights one decode token reads once (incl. the tied head and one embedding row)."""
    H, d, Hq, Hkv, I, V = wl.hidden, wl.head_dim, wl.n_heads, wl.n_kv_heads, wl.intermediate, wl.vocab
    mats = [Hq * d * H, 2 * Hkv * d * H, H * Hq * d, 3 * I * H]  # q, k+v, o, gate+up+down
    n = sum(mats)
    if wl.weight_format == "int8_g32":
        per_layer = n + 2 * (n // 32)  # int8 codes + fp16 scales
    else:
        per_layer = 2 * n
    per_layer += 2 * (2 * H + 2 * d)  # norms
    return wl.n_layers * per_layer + 2 * V * H + 2 * H + 2 * H  # + lm_head + final norm + embedding row


def kv_bytes_per_pos(wl) -> int:
    esz = 4 if wl.kv_format == "f32" else 2
    return wl.n_layers * wl.n_kv_heads * wl.head_dim * 2 * esz  # K and V rows of one position


def token_bytes(wl, pos: int) -> int:
    """Algorithmic HBM bytes of the decode step at position pos: weights once, the pos cached
    K/V rows read, this position's K/V written, f32 logits written."""
    return weight_bytes(wl) + kv_bytes_per_pos(wl) * (pos + 1) + 4 * wl.vocab


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense 16-bit tensor-core peak in TFLOP/s (burst: the prefill is timed on its own).
    fp16 and bf16 share kind::f16 and its nominal rate, so the bf16 figure applies."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured bf16 burst (fp16 runs at the same nominal rate)"
    return 1900.0, "fallback"


def prefill_flops(wl, T: int) -> int:
    """Algorithmic flops of a T-row prefill: the projections and MLP of every row, the
    causal QK^T and PV over non-masked (query, key) pairs, and the head of the last row."""
    H, d, Hq, Hkv, I, V = wl.hidden, wl.head_dim, wl.n_heads, wl.n_kv_heads, wl.intermediate, wl.vocab
    per_layer = Hq * d * H + 2 * Hkv * d * H + H * Hq * d + 3 * I * H
    gemm = 2 * T * wl.n_layers * per_layer
    attn = wl.n_layers * 4 * Hq * d * (T * (T + 1) // 2)
    return gemm + attn + 2 * V * H


DECODE_SOURCES = ("decode.cu", "decode_g1.cu", "decode_g2.cu", "decode_kernel.cuh", "topology.cu", "qw_internal.h")


def kernel_traffic(workload: str):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu capture of this
    workload, if the kernel's sources are unchanged since."""
    p = os.path.join(ROOT, "profiles", "decode_step_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_sha256_16") != decode_source_sha():
        return None
    return d.get("dram_bytes_per_launch")


def decode_source_sha():
    """First 16 hex digits of the SHA-256 over the decode kernel's sources, in DECODE_SOURCES order."""
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "runtime_qwen3_decode_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_threads() -> int:
    """Host cores this process may run on (the oracle's explicit thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_plan(n_decode: int, warmup: int, nthreads: int) -> dict:
    """The CPU oracle on the plan the bench states: the whole tiny workload (8-token prompt,
    8 greedy steps), then the Qwen3-0.6B-shape decode workload's 128-token prompt token by
    token and `warmup` + `n_decode` greedy decode steps after it.  Weight generation is not
    timed.  Runs in a process of its own (see cpu_plan_child) so that no CUDA context, torch
    thread pool or clock sampler shares the cores with it."""
    import oracle

    out = {"cores": nthreads}
    tiny = qi.WORKLOADS["tiny"]
    ref = oracle.OracleModel(tiny, qi.make_weights(tiny), nthreads=nthreads)
    t = time.perf_counter()
    oracle.run_sequence(ref, qi.prompt(tiny), tiny.decode_steps)
    out["tiny_whole_s"] = time.perf_counter() - t
    ref.close()

    wl = qi.WORKLOADS["qwen3_0p6b_decode"]
    ref = oracle.OracleModel(wl, qi.make_weights(wl), max_ctx=wl.prompt_len + warmup + n_decode + 1,
                             nthreads=nthreads)
    prompt = qi.prompt(wl)
    t = time.perf_counter()
    for i, tok in enumerate(prompt):
        lg, _ = ref.step(int(tok), want_logits=i == len(prompt) - 1)
    out["prefill_s"] = time.perf_counter() - t
    out["prefill_tokens"] = len(prompt)
    tok = oracle.argmax(lg)
    for _ in range(warmup):
        lg, _ = ref.step(tok)
        tok = oracle.argmax(lg)
    t = time.perf_counter()
    for _ in range(n_decode):
        lg, _ = ref.step(tok)
        tok = oracle.argmax(lg)
    out["decode_s"] = time.perf_counter() - t
    out["decode_steps"] = n_decode
    out["decode_positions"] = [wl.prompt_len + warmup, wl.prompt_len + warmup + n_decode - 1]
    out["value"] = n_decode / out["decode_s"]
    ref.close()
    return out


def cpu_plan_child(n_decode: int, warmup: int) -> dict:
    """oracle_plan in a fresh interpreter (no torch, no CUDA): the same program the reference
    arm runs, so the two CPU numbers come from identical conditions."""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-plan", "--steps", str(n_decode),
                        "--warmup", str(warmup)], capture_output=True, text=True, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"CPU oracle plan failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def plan_sample(plan: dict) -> str:
    return (f"oracle on {plan['cores']} host threads: tiny workload whole ({plan['tiny_whole_s']:.2f} s); "
            f"Qwen3-0.6B shape {plan['prefill_tokens']}-token prompt token by token "
            f"({plan['prefill_s']:.1f} s, {plan['prefill_tokens'] / plan['prefill_s']:.2f} tok/s) then "
            f"{plan['decode_steps']} timed greedy decode steps at positions {plan['decode_positions'][0]}.."
            f"{plan['decode_positions'][1]} ({plan['decode_s']:.1f} s)")


# -------------------------------------------------------------------- arms

def run_reference(args, wl):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    plan = oracle_plan(args.steps, args.warmup, cpu_threads())
    rate = plan["value"]
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * plan["decode_s"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "qwen3_0p6b_decode", "prompt": 128, "decode_steps": 384},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": plan["cores"], "kind": "oracle",
                             "sample": plan_sample(plan), "plan": plan},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def measure_prefill(qw, wl, reps: int, warmup: int, gpu: int):
    """Batched prefill of the workload's whole prompt: median device time over reps
    (CUDA events on the model's stream, after warm-up), plus one host-synchronous call."""
    import torch

    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    prompt = qi.prompt(wl)
    T = len(prompt)
    model = qw.Model(wl, dev, max_ctx=T + 1)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        model.kv_reset()
        model.prefill(prompt, want_token=False)
    model.sync()
    clocks = ClockSampler(gpu)
    clocks.start()
    times = []
    for _ in range(reps):
        model.kv_reset()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        model.prefill(prompt, want_token=False)
        e1.record(stream)
        model.sync()
        times.append(e0.elapsed_time(e1))
    clk = clocks.stop()
    model.kv_reset()
    torch.cuda.synchronize()
    t = time.perf_counter()
    model.prefill(prompt)  # host token ids in, greedy pick back to the host
    e2e_s = time.perf_counter() - t
    model.close()
    del dev
    ms = statistics.median(times)
    flops = prefill_flops(wl, T)
    tf = flops / (ms / 1e3) / 1e12
    peak, kind = measured_tensor_peak()
    return {"workload": wl.name, "tokens": T, "ms": ms, "ms_all": times, "tokens_per_s": T / (ms / 1e3),
            "dtype": "fp16 operands, f32 accumulation (tcgen05 kind::f16)",
            "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_kind": kind, "traffic": None,
                         "note": "whole prefill (GEMMs, attention, row kernels, head) against the GEMM peak"},
            "e2e": {"value": T / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * T, "d2h_bytes_per_step": 16,
                    "how": "qw_prefill(tokens_host, &next_token_host), host-synchronous"},
            "clocks": clk}


def measure_decode(qw, wl, K: int, W: int, gpu: int, ws: int = 1, with_e2e: bool = True):
    """Decode of one workload: W warm-up tokens, then exactly K timed tokens (CUDA events on the
    model's stream, a barrier and a synchronize on both sides).  A new sequence starts (reset +
    prefill or K/V import, inside the timed region) whenever the workload's decode budget is
    used up.  Returns the measured numbers and the model's byte accounting."""
    import torch

    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    del host
    prompt = qi.prompt(wl)
    per_seq = wl.decode_steps
    n0 = wl.kv_prefill + wl.prompt_len  # positions in the cache when decoding starts
    max_ctx = n0 + per_seq + 1
    model = qw.Model(wl, dev, max_ctx=max_ctx)
    stream = torch.cuda.current_stream()
    kd = vd = None
    if wl.kv_prefill:
        kh, vh = qi.kv_fill(wl, wl.kv_prefill)
        kd = torch.from_numpy(kh.view(np.int16)).cuda()
        vd = torch.from_numpy(vh.view(np.int16)).cuda()
        del kh, vh

    def start_sequence():
        """Fresh cache for a new sequence; returns the first decode input (-1: the prefill's pick)."""
        model.kv_reset()
        if wl.kv_prefill:
            model.kv_import(kd, vd, wl.kv_prefill)
        if wl.prompt_len:
            model.prefill(prompt, want_token=False)
            return -1
        return qi.first_decode_token(wl)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    toks = torch.zeros(max(K, 1), dtype=torch.int32, device="cuda")
    positions = []
    state = {"next_in": start_sequence(), "done": 0}

    def run_tokens(n, out=None, record=False):
        i = 0
        while i < n:
            if state["done"] == per_seq:
                state["next_in"] = start_sequence()
                state["done"] = 0
            m = min(n - i, per_seq - state["done"])
            if record:
                positions.extend(range(model.kv_length, model.kv_length + m))
            model.generate(m, state["next_in"], out[i:i + m] if out is not None else None)
            state["next_in"] = -1
            state["done"] += m
            i += m

    run_tokens(W)
    model.sync()
    clocks = ClockSampler(gpu)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run_tokens(K, toks, record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    model.sync()
    ms = t0.elapsed_time(t1)
    if ws > 1:
        import torch.distributed as dist
        tt = torch.tensor([ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())

    e2e = None
    if with_e2e:
        # end to end through the public call: host token in, host token out, every step
        model.kv_reset()
        tok = qi.first_decode_token(wl)
        if wl.kv_prefill:
            model.kv_import(kd, vd, wl.kv_prefill)
        if wl.prompt_len:
            tok = model.prefill(prompt)
        n_e2e = min(K, per_seq)
        torch.cuda.synchronize()
        t_e = time.perf_counter()
        for _ in range(n_e2e):
            tok = model.decode_step(tok)
        e2e = {"value": n_e2e / (time.perf_counter() - t_e), "unit": UNIT, "h2d_bytes_per_step": 4,
               "d2h_bytes_per_step": 16,
               "how": "qw_decode_step(token_from_host, &next_token_host) per token, host-synchronous"}
    model.close()
    del kd, vd, dev
    torch.cuda.empty_cache()
    peak, peak_kind = measured_peaks()
    bytes_timed = sum(token_bytes(wl, p) for p in positions)
    achieved = bytes_timed / (ms / 1000.0) / 1e9
    return {"ms": ms, "K": K, "W": W, "positions": positions, "value": K * ws / (ms / 1000.0),
            "bytes_per_token_mean": bytes_timed / max(1, len(positions)), "achieved": achieved, "peak": peak,
            "peak_kind": peak_kind, "clocks": clk, "e2e": e2e, "n0": n0}


def decode_sub(qw, wl, K: int, W: int, gpu: int) -> dict:
    """A secondary decode workload's figures for the bench line (same method as the headline)."""
    r = measure_decode(qw, wl, K, W, gpu, with_e2e=False)
    return {"workload": wl.name, "value": r["value"], "unit": UNIT, "steps": K, "warmup": W,
            "ms_per_step": r["ms"] / K, "positions_timed": [r["positions"][0], r["positions"][-1]],
            "weights": wl.weight_format, "kv_cache": wl.kv_format,
            "roofline": {"bound": "hbm", "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
                         "frac": r["achieved"] / r["peak"], "peak_kind": r["peak_kind"],
                         "bytes_per_token": r["bytes_per_token_mean"],
                         "bytes_per_token_at_first_pos": token_bytes(wl, r["positions"][0]),
                         "traffic": kernel_traffic(wl.name)},
            "clocks": r["clocks"]}


def measure_batch(qw, wl, B: int, K: int, W: int, gpu: int) -> dict:
    """Batched decode (qw_batch_*): B sequences of the workload's shape, each with its own
    seeded prompt of the workload's length, prefilled, then W untimed and K timed steps of all B
    (CUDA events on the model's stream, a synchronize on both sides)."""
    import torch

    host = qi.make_weights(wl)
    dev = qw.weights_to_device(host, int8=wl.weight_format == "int8_g32")
    del host
    n_ctx = wl.prompt_len + W + K + 1
    model = qw.Model(wl, dev, max_ctx=n_ctx)
    batch = qw.Batch(model, B, n_ctx)
    g = np.random.default_rng(1000 + B)
    for s in range(B):
        batch.prefill(s, g.integers(0, wl.vocab, size=wl.prompt_len), want_token=False)
    for _ in range(W):
        batch.step(B, want_tokens=False)
    model.sync()
    batch.sync()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(gpu)
    clocks.start()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    first = batch.length(0)
    t0.record(stream)
    for _ in range(K):
        batch.step(B, want_tokens=False)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    batch.sync()
    ms = t0.elapsed_time(t1)
    positions = range(first, first + K)
    step_bytes = [weight_bytes(wl) + B * (kv_bytes_per_pos(wl) * (p + 1) + 4 * wl.vocab) for p in positions]
    peak, peak_kind = measured_peaks()
    achieved = sum(step_bytes) / (ms / 1000.0) / 1e9
    batch.close()
    model.close()
    del dev
    torch.cuda.empty_cache()
    return {"workload": wl.name, "batch": B, "value": B * K / (ms / 1000.0), "unit": "tokens/s (all sequences)",
            "per_sequence": K / (ms / 1000.0), "steps": K, "warmup": W, "ms_per_step": ms / K,
            "positions_timed": [positions[0], positions[-1]],
            "compute": "fp16 tensor-core operands for the projections and MLP (M = batch), f32 accumulation; "
                       "per-sequence split attention and the lm_head on CUDA cores",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "bytes_per_step_at_first_pos": step_bytes[0]},
            "clocks": clk}


def run_ours(args, wl):
    import torch

    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from runtime_qwen3_decode_gb300 import build as qbuild
    from runtime_qwen3_decode_gb300 import qw

    qbuild.build()
    W, K = args.warmup, args.steps
    r = measure_decode(qw, wl, K, W, local, ws)
    if rank != 0:
        return 0
    positions = r["positions"]
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": r["ms"] / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.weight_format == "bf16" else "int8",
        "data": "synthetic (seeded random-init weights, uniform-random prompt)",
        "config": {"workload": wl.name, "prompt": wl.prompt_len, "decode_steps": wl.decode_steps,
                   "positions_timed": [positions[0], positions[-1]] if positions else None,
                   "compute": "bf16 weights x f32 activations, f32 accumulation",
                   "l2": "no flush: inputs larger than L2 (weights streamed per token)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "achieved": r["achieved"], "peak": r["peak"], "unit": "GB/s",
                     "frac": r["achieved"] / r["peak"], "peak_kind": r["peak_kind"],
                     "frac_of_nominal_7.9TBs": r["achieved"] / NOMINAL_HBM_GBS,
                     "bytes_per_token_mean": r["bytes_per_token_mean"],
                     "bytes_per_token_at_first_pos": token_bytes(wl, positions[0]) if positions else None,
                     "kernel": "qw::decode_kernel (one persistent launch per token)",
                     "traffic": kernel_traffic(wl.name)},
        "e2e": r["e2e"],
        "gpu_launches": K,
        "clocks": r["clocks"],
    }
    if not args.no_extra and ws == 1:
        for key, name, k_sub in (("decode_ctx32k", "qwen3_0p6b_ctx32k", 56), ("decode_int8", "qwen3_0p6b_int8", 248)):
            sub = qi.WORKLOADS[name]
            if sub.name != wl.name:
                line[key] = decode_sub(qw, sub, min(k_sub, sub.decode_steps - W), W, local)
        # the int8 workload with int8 activations too (Q8 x Q8; its prompt runs through the decode path)
        q8 = qi.WORKLOADS["qwen3_0p6b_int8"].with_(act_format="q8")
        line["decode_q8q8"] = decode_sub(qw, q8, 248, W, local)
        line["decode_q8q8"]["activations"] = "int8, per 32-element block, quantized in the kernel"
    if not args.no_extra and ws == 1:
        for B in (8,):
            line[f"decode_batch{B}"] = measure_batch(qw, qi.WORKLOADS["qwen3_0p6b_decode"], B, 64, W, local)
    if not args.no_prefill:
        line["prefill"] = measure_prefill(qw, qi.WORKLOADS[args.prefill_workload], args.prefill_reps,
                                          max(3, min(W, 5)), local)
    if not args.no_cpu_baseline and ws == 1:
        plan = cpu_plan_child(args.cpu_steps, 2)
        line["cpu_baseline"] = {"value": plan["value"], "unit": UNIT, "cores": plan["cores"], "kind": "oracle",
                                "sample": plan_sample(plan), "plan": plan}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed decode tokens (default: the workload's "
                    "decode budget minus the warm-up)")
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_0p6b_decode", choices=sorted(qi.WORKLOADS))
    ap.add_argument("--cpu-steps", type=int, default=32, help="timed oracle decode steps of the CPU baseline")
    ap.add_argument("--cpu-plan", action="store_true", help=argparse.SUPPRESS)  # the baseline's child process
    ap.add_argument("--no-extra", action="store_true", help="skip the 32K-context and int8 decode sub-objects")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-workload", default="qwen3_0p6b_prefill2048", choices=sorted(qi.WORKLOADS))
    ap.add_argument("--prefill-reps", type=int, default=5)
    ap.add_argument("--no-prefill", action="store_true")
    args = ap.parse_args()
    if args.cpu_plan:
        print(json.dumps(oracle_plan(args.steps, args.warmup, cpu_threads())), flush=True)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    wl = qi.WORKLOADS[args.workload]
    if args.steps is None:
        args.steps = max(1, wl.decode_steps - args.warmup)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
