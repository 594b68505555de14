#!/usr/bin/env python3
"""DSA forward benchmark on GB300: query tokens/s at S = 32768, top-2048
(DeepSeek-V3.2 shapes: 128 heads, d_qk 576, d_v 512, indexer 64 x 128), plus
the tensor-core fraction of the indexer + attention stages.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over one synthetic batch: indexer
scores -> top-k (streamed in row waves through a workspace ring) -> sparse
attention, through the library's C ABI.  N > 1 (torchrun): every rank runs an
independent replica problem of its own (weak scaling, no collective on the
data path); value = all ranks' tokens / the slowest rank's time.

--impl reference times the C++ CPU oracle (fp64 loops, std::thread workers on
all host cores) on a bounded sample of query rows of the same workload per
step.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "DSA fwd query tokens/s @S=32K top-2048; % of GB300 bf16 tensor-core peak"
UNIT = "query tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank's step time, all-reduced with MAX
    (the job's time is its slowest replica's)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t)


def job_value(world: int, rows_per_rank: int, ms: float) -> float:
    """Whole-job throughput: the query rows all ranks processed / the job's time."""
    return world * rows_per_rank / (ms * 1e-3)


def replica_seed(rank: int) -> int:
    """Each rank draws its own replica problem (weak scaling)."""
    return rank


def algorithmic(wl, pos):
    """Work the method must do (causal / selected pairs only)."""
    n = pos.astype(np.float64) + 1.0
    sel = np.minimum(n, wl["topk"])
    f_idx = 2.0 * wl["H_I"] * wl["d_I"] * n.sum()
    f_attn = 2.0 * wl["H"] * (wl["d_qk"] + wl["d_v"]) * sel.sum()
    topk_bytes = 4.0 * n.sum() + 4.0 * wl["topk"] * pos.size
    return f_idx, f_attn, topk_bytes


def algorithmic_bwd(wl, pos):
    """Backward work: attention backward 2*H*(3*d_qk + 2*d_v) flops per selected
    pair (S and dP recomputed, dQ, dK, dV) and the indexer KL pass
    (2*H*d_qk + 3*2*H_I*d_I) per selected pair (the probability recompute, the
    indexer logits, dq_I and dk_I)."""
    sel = np.minimum(pos.astype(np.float64) + 1.0, wl["topk"]).sum()
    f_bwd = 2.0 * wl["H"] * (3 * wl["d_qk"] + 2 * wl["d_v"]) * sel
    f_kl = (2.0 * wl["H"] * wl["d_qk"] + 3 * 2.0 * wl["H_I"] * wl["d_I"]) * sel
    return f_bwd, f_kl


def time_calls(fn, steps, warmup, stream):
    """Mean ms of fn() over `steps` calls after `warmup`, CUDA events on `stream`."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def fp8_indexer_stage(dsa, dev, wl, x, waves, steps, peak_tc):
    """The FP8 (E4M3) indexer on the same rows as the step, outside the timed
    step: the quantization of q_I and k_I, then every wave of scores.  Its
    tensor peak is the bf16 peak x 2 (the nominal FP8 / BF16 ratio)."""
    S = wl["S"]
    p = dsa.make_params(B=1, S_q=S, S_k=S, H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"], H_I=wl["H_I"],
                        d_I=wl["d_I"], topk=wl["topk"], scale=wl["scale"], dtype="bf16", flags=1)
    q8 = torch.empty(1, S, wl["H_I"], wl["d_I"], dtype=torch.uint8, device=dev)
    sq = torch.empty(1, S, wl["H_I"], device=dev)
    k8 = torch.empty(1, S, wl["d_I"], dtype=torch.uint8, device=dev)
    sk = torch.empty(1, S, device=dev)
    ring = torch.empty(max(n for _, n in waves), S, device=dev)
    st = torch.cuda.current_stream(dev)
    t_q = time_calls(lambda: dsa.indexer_quantize_fp8(p, x["q_I"], x["k_I"], q8, sq, k8, sk), steps, 2, st)

    def scores():
        for r0, n in waves:
            dsa.indexer_scores_fp8(p, q8, sq, k8, sk, x["w"], r0, n, ring)
    t_s = time_calls(scores, steps, 2, st)
    assert dsa.get_status() == 0
    f_idx, _, _ = algorithmic(wl, np.arange(S))
    tflops = f_idx / (t_s * 1e-3) / 1e12
    return {"quantize_ms": t_q, "scores_ms": t_s, "tflops": tflops, "peak_fp8": 2 * peak_tc,
            "frac": tflops / (2 * peak_tc),
            "note": "E4M3 q_I, k_I with one fp32 scale per 128-vector; outside the timed step"}


def fused_topk_stage(dsa, dev, wl, x, idx_ref, steps):
    """The fused indexer + streaming top-k (dsa_indexer_topk) over the step's
    rows, outside the timed step, and the whole forward with it
    (DSA_FLAG_FUSED_TOPK); its indices are checked against the step's."""
    S, k = wl["S"], wl["topk"]
    p = dsa.make_params(B=1, S_q=S, S_k=S, H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"], H_I=wl["H_I"],
                        d_I=wl["d_I"], topk=k, scale=wl["scale"], dtype="bf16",
                        flags=dsa.DSA_FLAG_FUSED_TOPK)
    st = torch.cuda.current_stream(dev)
    ws = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_INDEXER_TOPK), dtype=torch.uint8, device=dev)
    idx = torch.empty(1, S, k, dtype=torch.int32, device=dev)
    t_sel = time_calls(lambda: dsa.indexer_topk(p, x["q_I"], x["k_I"], x["w"], 0, S, idx, ws), steps, 2, st)
    same = bool(torch.equal(idx, idx_ref))
    out = torch.empty(1, S, wl["H"], wl["d_v"], dtype=torch.bfloat16, device=dev)
    m = torch.empty(1, S, wl["H"], device=dev)
    l = torch.empty_like(m)
    t_fwd = time_calls(lambda: dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], idx, out, m, l,
                                           ws), steps, 2, st)
    assert dsa.get_status() == 0
    return {"indexer_topk_ms": t_sel, "forward_ms": t_fwd, "forward_tokens_per_s": S / (t_fwd * 1e-3),
            "equals_unfused": same,
            "note": "indexer + top-k fused (candidate lists instead of the score ring); outside the "
                    "timed step, no L2 flush between calls"}


def backward_stage(dsa, dev, steps, peak_tc, workload="dsv32_S16384_train", rows=None):
    """The training-shape backward (S = 16384, top-2048, all rows): the forward,
    the attention backward (dq, dkv), the indexer KL-loss backward, each timed
    alone, and dsa_backward (both in one call sharing the recompute of P).
    `workload` picks another shape and `rows` the last `rows` query rows
    against all S keys (a context-parallel shard), for profiling on a small
    device footprint."""
    wl = synth.WORKLOADS[workload]
    S, k, H = wl["S"], wl["topk"], wl["H"]
    S_q = S if rows is None else int(rows)
    x = synth.make_inputs(wl, device=dev, with_dout=True, S_q=S_q)
    p = dsa.make_params(B=1, S_q=S_q, S_k=S, H=H, d_qk=wl["d_qk"], d_v=wl["d_v"], H_I=wl["H_I"],
                        d_I=wl["d_I"], topk=k, scale=wl["scale"], dtype="bf16",
                        q_row_offset=S - S_q)
    ring = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD), dtype=torch.uint8, device=dev)
    idx = torch.empty(1, S_q, k, dtype=torch.int32, device=dev)
    out = torch.empty(1, S_q, H, wl["d_v"], dtype=torch.bfloat16, device=dev)
    m = torch.empty(1, S_q, H, device=dev)
    l = torch.empty_like(m)
    dq = torch.empty(1, S_q, H, wl["d_qk"], dtype=torch.bfloat16, device=dev)
    dkv = torch.zeros(1, S, wl["d_qk"], device=dev)
    ws_b = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_ATTN_BWD), dtype=torch.uint8, device=dev)
    loss = torch.zeros(1, device=dev)
    dq_I = torch.empty(1, S_q, wl["H_I"], wl["d_I"], dtype=torch.bfloat16, device=dev)
    dk_I = torch.zeros(1, S, wl["d_I"], device=dev)
    dw = torch.empty(1, S_q, wl["H_I"], device=dev)
    ws_k = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_KL_BWD), dtype=torch.uint8, device=dev)
    ws_all = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_BACKWARD), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fwd = lambda: dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], idx, out, m, l, ring)
    bwd = lambda: dsa.sparse_attn_bwd(p, x["q"], x["kv"], idx, out, x["dO"], m, l, dq, dkv, ws_b)
    kl = lambda: dsa.indexer_kl_loss_bwd(p, x["q"], x["kv"], x["q_I"], x["k_I"], x["w"], idx, m, l,
                                         loss, dq_I, dk_I, dw, ws_k)
    both = lambda: dsa.backward(p, x["q"], x["kv"], idx, out, x["dO"], m, l, x["q_I"], x["k_I"],
                                x["w"], dq, dkv, loss, dq_I, dk_I, dw, ws_all)
    t_fwd = time_calls(fwd, steps, 1, stream)
    t_bwd = time_calls(bwd, steps, 1, stream)
    t_kl = time_calls(kl, steps, 1, stream)
    t_both = time_calls(both, steps, 1, stream)
    # dsa_backward in row passes (wave_rows): the workspace holds one pass
    W = min(2048, S_q)
    p_w = dsa.make_params(B=1, S_q=S_q, S_k=S, H=H, d_qk=wl["d_qk"], d_v=wl["d_v"], H_I=wl["H_I"],
                          d_I=wl["d_I"], topk=k, scale=wl["scale"], dtype="bf16",
                          q_row_offset=S - S_q, wave_rows=W)
    ws_w = torch.empty(dsa.workspace_size(p_w, dsa.DSA_CALL_BACKWARD), dtype=torch.uint8, device=dev)
    both_w = lambda: dsa.backward(p_w, x["q"], x["kv"], idx, out, x["dO"], m, l, x["q_I"], x["k_I"],
                                  x["w"], dq, dkv, loss, dq_I, dk_I, dw, ws_w)
    t_both_w = time_calls(both_w, steps, 1, stream)
    assert dsa.get_status() == 0, "device status after the backward"
    f_bwd, f_kl = algorithmic_bwd(wl, np.arange(S - S_q, S))
    return {"workload": wl["name"], "rows": S_q, "calls_timed": steps,
            "forward_ms": t_fwd, "attn_bwd_ms": t_bwd, "kl_bwd_ms": t_kl,
            "backward_ms": t_both,
            "backward_ms_in_passes": t_both_w, "pass_rows": W,
            "backward_tflops": (f_bwd + f_kl) / (t_both * 1e-3) / 1e12,
            "attn_bwd_tflops": f_bwd / (t_bwd * 1e-3) / 1e12,
            "kl_bwd_tflops": f_kl / (t_kl * 1e-3) / 1e12,
            "attn_bwd_frac": f_bwd / (t_bwd * 1e-3) / 1e12 / peak_tc,
            "workspace_bytes": {"attn_bwd": ws_b.numel(), "kl_bwd": ws_k.numel(),
                                "backward": ws_all.numel(), "backward_in_passes": ws_w.numel()},
            "note": "outside the timed forward step; dkv / dk_I accumulate over calls"}


def topk_stage(dsa, dev, wl, steps, warmup, peaks):
    """Top-k alone on the last wave of the workload (rows at the end of the
    sequence, the longest ones) over seeded N(0, 8^2) scores; a profiling aid."""
    S, k = wl["S"], wl["topk"]
    R = min(2048, S)
    p = dsa.make_params(B=1, S_q=R, S_k=S, H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"],
                        H_I=wl["H_I"], d_I=wl["d_I"], topk=k, scale=wl["scale"], dtype="bf16",
                        q_row_offset=S - R)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    sc = torch.randn(R, S, device=dev, generator=g) * 8.0
    idx = torch.empty(R, k, dtype=torch.int32, device=dev)
    ms = time_calls(lambda: dsa.topk(p, sc, 0, R, idx), steps, warmup, torch.cuda.current_stream(dev))
    assert dsa.get_status() == 0
    _, _, byts = algorithmic(wl, np.arange(S - R, S))
    return {"stage": "topk", "workload": wl["name"], "rows": R, "ms": ms,
            "gbs": byts / (ms * 1e-3) / 1e9, "hbm_frac": byts / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 50 ms from before
    the warm-up on; only the samples stamped inside the timed region count."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.t0 = self.t1 = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        # wait (at most 5 s) for the first sample, so the sampler runs when
        # the timed region starts
        t_end = time.time() + 5.0
        while self.p is not None and time.time() < t_end and os.path.getsize(self.f.name) == 0:
            time.sleep(0.02)

    def start_window(self):
        self.t0 = time.time()

    def end_window(self):
        self.t1 = time.time()

    @staticmethod
    def _stamp(text):
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 9]
        os.unlink(self.f.name)
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None and
                  (ts := self._stamp(r[0])) is not None and self.t0 <= ts <= self.t1]
        window = bool(inside)
        rows = inside if inside else rows
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "samples_in_timed_region": window}


def kernel_traffic(kernel_file, summary):
    """DRAM bytes per launch recorded by an ncu capture, valid only while the
    kernel source is unchanged (sha256 prefix recorded beside the number)."""
    path = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "sparse_attention_long_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "kernel_sha256")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sha256") != h:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ oracle arm
def oracle_inputs(wl, rows, seed=0):
    """The workload's inputs restricted to the sampled query rows (the
    generator is counter based, so rows are drawn directly)."""
    S, H, dqk, HI, dI = wl["S"], wl["H"], wl["d_qk"], wl["H_I"], wl["d_I"]

    def rows_of(name, width, scale):
        parts = [synth.normal_flat(int(t) * width, width, seed, synth.STREAM[name]) for t in rows]
        return (torch.stack(parts) * scale).to(torch.bfloat16)

    return dict(q_I=rows_of("q_I", HI * dI, 1.0).view(1, len(rows), HI, dI),
                w=rows_of("w", HI, 1.0 / 8).view(1, len(rows), HI),
                q=rows_of("q", H * dqk, 1.0).view(1, len(rows), H, dqk),
                k_I=synth.normal((1, S, dI), "k_I", seed),
                kv=synth.normal((1, S, dqk), "kv", seed))


def host_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def oracle_f64(x):
    """The sampled inputs widened once to float64 (exact) for the C++ oracle."""
    return {n: t.double().numpy() for n, t in x.items()}


def oracle_step(wl, x64, rows, threads):
    """Indexer -> top-k -> attention for the given global rows, C++ oracle
    (fp64 loops, one row per task on `threads` std::thread workers)."""
    from oracle import cpp
    cpp.dsa_forward(x64["q_I"], x64["k_I"], x64["w"], x64["q"], x64["kv"], wl["topk"], wl["scale"],
                    wl["d_v"], q_row_index=np.asarray(rows, dtype=np.int64), threads=threads)


def sample_rows(S, n, seed=0):
    rng = np.random.default_rng(seed)
    a = max(1, n // 4)
    rows = np.concatenate([np.arange(a), np.arange(S - a, S), rng.integers(0, S, n - 2 * a)])
    return np.unique(rows)[:n]


def cpu_baseline(wl, budget_s=15.0):
    """The C++ oracle as it stands, on all host cores, on sampled query rows
    (the first, the last and uniform rows of the workload)."""
    from oracle import cpp
    cpp.build()
    threads = host_threads()
    rows_all = sample_rows(wl["S"], 4096, seed=0)
    x = oracle_f64(oracle_inputs(wl, rows_all))
    chunk = 2 * threads
    done, t0 = 0, time.perf_counter()
    while done < rows_all.size and time.perf_counter() - t0 < budget_s:
        sel = slice(done, min(done + chunk, rows_all.size))
        xs = dict(x, q_I=x["q_I"][:, sel], w=x["w"][:, sel], q=x["q"][:, sel])
        oracle_step(wl, xs, rows_all[sel], threads)
        done = sel.stop
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} query rows of the S={wl['S']} workload (first/last/uniform): indexer "
                      f"over all causal keys + top-k + attention, C++ fp64 oracle on {threads} "
                      f"std::thread workers, {dt:.1f} s"}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import cpp
    cpp.build()
    threads = host_threads()
    rows_per_step = 2 * threads
    rows_all = sample_rows(wl["S"], rows_per_step * (args.steps + args.warmup), seed=1)
    x = oracle_f64(oracle_inputs(wl, rows_all))
    times = []
    for i in range(args.warmup + args.steps):
        sel = slice(i * rows_per_step, min((i + 1) * rows_per_step, rows_all.size))
        if sel.start >= sel.stop:
            sel = slice(0, rows_per_step)
        xs = dict(x, q_I=x["q_I"][:, sel], w=x["w"][:, sel], q=x["q"][:, sel])
        t0 = time.perf_counter()
        oracle_step(wl, xs, rows_all[sel], threads)
        if i >= args.warmup:
            times.append((time.perf_counter() - t0, sel.stop - sel.start))
    tot = sum(t for t, _ in times)
    value = sum(n for _, n in times) / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl["name"], "S": wl["S"], "topk": wl["topk"],
                       "rows_per_step": rows_per_step},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{rows_per_step} query rows per step of the S={wl['S']} "
                                       f"workload, C++ fp64 oracle on {threads} std::thread workers"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- our arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv32_S32768", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-bwd", action="store_true", help="skip the training-shape backward timing")
    ap.add_argument("--rows", type=int, default=None,
                    help="with --stage bwd: the last N query rows against all keys (profiling)")
    ap.add_argument("--stage", default=None, choices=["topk", "bwd", "fp8idx", "fused"],
                    help="time one stage alone (a profiling aid; prints its own JSON line)")
    args = ap.parse_args()
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_long_gb300 as dsa
    if args.stage == "topk":
        print(json.dumps(topk_stage(dsa, dev, wl, args.steps, args.warmup, load_peaks())), flush=True)
        return
    if args.stage == "fp8idx":
        S0 = wl["S"]
        xi = synth.make_inputs(wl, device=dev)
        p0 = dsa.make_params(B=1, S_q=S0, S_k=S0, H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"], H_I=wl["H_I"],
                             d_I=wl["d_I"], topk=wl["topk"], scale=wl["scale"], dtype="bf16")
        W0 = dsa.wave_rows(p0)
        wv = [(r0, min(W0, S0 - r0)) for r0 in range(0, S0, W0)]
        r = fp8_indexer_stage(dsa, dev, wl, xi, wv, args.steps, load_peaks()["bf16_tflops"])
        print(json.dumps(dict(stage="fp8idx", workload=wl["name"], **r)), flush=True)
        return
    if args.stage == "fused":
        S0, k0 = wl["S"], wl["topk"]
        xi = synth.make_inputs(wl, device=dev)
        p0 = dsa.make_params(B=1, S_q=S0, S_k=S0, H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"], H_I=wl["H_I"],
                             d_I=wl["d_I"], topk=k0, scale=wl["scale"], dtype="bf16",
                             flags=dsa.DSA_FLAG_CAUSAL_ONLY)  # as dsa_forward's ring
        ring0 = torch.empty(dsa.workspace_size(p0, dsa.DSA_CALL_FORWARD), dtype=torch.uint8, device=dev)
        idx0 = torch.empty(1, S0, k0, dtype=torch.int32, device=dev)
        W0 = dsa.wave_rows(p0)
        sc0 = torch.empty(W0, S0, device=dev)
        def plain():
            for r0 in range(0, S0, W0):
                n0 = min(W0, S0 - r0)
                dsa.indexer_scores(p0, xi["q_I"], xi["k_I"], xi["w"], r0, n0, sc0)
                dsa.topk(p0, sc0, r0, n0, idx0[0, r0:r0 + n0])
        t_plain = time_calls(plain, args.steps, 2, torch.cuda.current_stream(dev))
        del ring0
        r = fused_topk_stage(dsa, dev, wl, xi, idx0, args.steps)
        print(json.dumps(dict(stage="fused", workload=wl["name"], indexer_then_topk_ms=t_plain, **r)),
              flush=True)
        return
    if args.stage == "bwd":
        wname = args.workload if args.workload != "dsv32_S32768" else "dsv32_S16384_train"
        bwd = backward_stage(dsa, dev, args.steps, load_peaks()["bf16_tflops_sustained"], wname,
                             args.rows)
        print(json.dumps(dict(stage="bwd", **bwd)), flush=True)
        return

    S, k = wl["S"], wl["topk"]
    x = synth.make_inputs(wl, device=dev, seed=replica_seed(rank))  # each rank: its own replica
    mk = lambda **kw: dsa.make_params(B=1, S_q=S, S_k=S, H=wl["H"], d_qk=wl["d_qk"], d_v=wl["d_v"],
                                      H_I=wl["H_I"], d_I=wl["d_I"], topk=k, scale=wl["scale"],
                                      dtype="bf16", **kw)
    p = mk()
    p_causal = mk(flags=dsa.DSA_FLAG_CAUSAL_ONLY)
    W = dsa.wave_rows(p)
    ring = torch.empty(dsa.workspace_size(p, dsa.DSA_CALL_FORWARD) // 4, device=dev)
    idx = torch.empty(1, S, k, dtype=torch.int32, device=dev)
    out = torch.empty(1, S, wl["H"], wl["d_v"], dtype=torch.bfloat16, device=dev)
    m = torch.empty(1, S, wl["H"], device=dev)
    l = torch.empty_like(m)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    waves = [(r0, min(W, S - r0)) for r0 in range(0, S, W)]

    def step(ev=None):
        for i, (r0, n) in enumerate(waves):
            if ev: ev["idx"][i][0].record(stream)
            dsa.indexer_scores(p_causal, x["q_I"], x["k_I"], x["w"], r0, n, ring)
            if ev: ev["idx"][i][1].record(stream)
            dsa.topk(p, ring, r0, n, idx.view(S, k)[r0:r0 + n])
            if ev: ev["topk"][i][1].record(stream)
        if ev: ev["attn"][0].record(stream)
        dsa.sparse_attn_fwd(p, x["q"], x["kv"], idx, out, m, l)
        if ev: ev["attn"][1].record(stream)

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    assert dsa.get_status() == 0, "device status after warm-up"

    E = lambda: torch.cuda.Event(enable_timing=True)
    evs = [dict(idx=[(E(), E()) for _ in waves], topk=[(None, E()) for _ in waves], attn=(E(), E()))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start_window()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        step(evs[s])
        flush.zero_()          # L2 flush between steps (outside the per-stage events)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks.end_window()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    assert dsa.get_status() == 0, "device status after the timed steps"

    t_idx = t_topk = t_attn = 0.0
    per_step = []                       # ms of each timed step (for the median)
    for e in evs:
        t0 = t_idx + t_topk + t_attn
        for i in range(len(waves)):
            t_idx += e["idx"][i][0].elapsed_time(e["idx"][i][1])
            t_topk += e["idx"][i][1].elapsed_time(e["topk"][i][1])
        t_attn += e["attn"][0].elapsed_time(e["attn"][1])
        per_step.append(t_idx + t_topk + t_attn - t0)
    K = args.steps
    t_idx, t_topk, t_attn = t_idx / K, t_topk / K, t_attn / K      # ms per step
    ms_step = t_idx + t_topk + t_attn
    ms_step = max_over_ranks(ms_step, world, dev)

    f_idx, f_attn, topk_bytes = algorithmic(wl, np.arange(S))
    peaks = load_peaks()
    # The denominator follows the clocks seen during the timed region: the
    # burst peak when the SMs ran at their maximum clock with no power cap,
    # else the sustained one; both fractions are reported.
    burst = bool(clk and clk.get("sm_mhz") and clk.get("sm_max_mhz") and
                 clk["sm_mhz"] >= clk["sm_max_mhz"] - 1 and "sw_power_cap" not in clk.get("reasons", []))
    peak_key = "bf16_tflops" if burst else "bf16_tflops_sustained"
    peak_tc = peaks[peak_key]
    value = job_value(world, S, ms_step)
    attn_tflops = f_attn / (t_attn * 1e-3) / 1e12
    tensor_frac = (f_idx + f_attn) / ((t_idx + t_attn) * 1e-3) / 1e12 / peak_tc
    tensor_frac_sust = (f_idx + f_attn) / ((t_idx + t_attn) * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"]
    # the attention's gather: every selected kv row crosses into shared memory
    # once per CTA pair (each CTA its 288 of the 576 columns): 2 * 576 bytes
    gather_bytes = 2.0 * wl["d_qk"] * np.minimum(np.arange(S) + 1.0, k).sum()

    # end to end through dsa_forward with pinned host buffers
    e2e = None
    if not args.no_e2e:
        host_in = {n: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for n, v in x.items()}
        for n in host_in:
            host_in[n].copy_(x[n])
        host_out = dict(idx=torch.empty(idx.shape, dtype=idx.dtype, pin_memory=True),
                        out=torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                        m=torch.empty(m.shape, pin_memory=True), l=torch.empty(l.shape, pin_memory=True))
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())

        # The step is cut into row chunks (dsa_forward with q_row_offset, as a
        # context-parallel shard would call it) so that the host->device copy
        # of the next chunk and the device->host copy of the previous one
        # overlap the compute of the current chunk on three streams.  Rows are
        # independent, so the results equal one whole-sequence call bit for
        # bit.  Chunks run from the last rows to the first: causal rows get
        # cheaper towards the start while their copies do not, so the heavy
        # chunks hide the copies of the light ones.  Each chunk but the last
        # (the lightest) is two indexer waves, so no wave of a chunk runs
        # with idle SMs.  The device inputs are double-buffered across steps
        # (a data loader's prefetch): step s copies into buffer s % 2 once
        # step s - 2's compute has released it, so the next step's copies run
        # under this step's compute, and the first chunk's copy-in and the
        # last chunk's copy-out overlap the neighbouring steps.
        c_rows = 2 * dsa.wave_rows(p)
        if S >= 4 * c_rows:
            sizes = [c_rows] * (S // c_rows) + ([S % c_rows] if S % c_rows else [])
        else:
            sizes = [S]
        bounds = []
        r1 = S
        for n_rows in sizes:                 # descending rows
            bounds.append((r1 - n_rows, r1))
            r1 -= n_rows
        nch = len(bounds)
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        pc = []
        for (r0, r1) in bounds:
            pr = mk(q_row_offset=r0)
            pr.S_q = r1 - r0
            pc.append(pr)
        rows = lambda t, c: t[:, bounds[c][0]:bounds[c][1]]
        xs = (x, {n: torch.empty_like(v) for n, v in x.items()})
        prev = {"cmp": [None, None], "out": [None] * nch, "step": 0}

        def e2e_step():
            e_kv, e_in, e_done, e_out = E(), [E() for _ in range(nch)], [E() for _ in range(nch)], \
                [E() for _ in range(nch)]
            buf = prev["step"] % 2
            xb = xs[buf]
            with torch.cuda.stream(s_in):
                if prev["cmp"][buf] is not None:  # step - 2 no longer reads this input buffer
                    s_in.wait_event(prev["cmp"][buf])
                xb["k_I"].copy_(host_in["k_I"], non_blocking=True)
                xb["kv"].copy_(host_in["kv"], non_blocking=True)
                e_kv.record(s_in)
                for c in range(nch):
                    for n in ("q_I", "w", "q"):
                        rows(xb[n], c).copy_(rows(host_in[n], c), non_blocking=True)
                    e_in[c].record(s_in)
            s_cmp.wait_event(e_kv)
            for c in range(nch):
                s_cmp.wait_event(e_in[c])
                if prev["out"][c] is not None:  # the previous step's outputs are copied out
                    s_cmp.wait_event(prev["out"][c])
                dsa.forward(pc[c], rows(xb["q_I"], c), xb["k_I"], rows(xb["w"], c), rows(xb["q"], c),
                            xb["kv"], rows(idx, c), rows(out, c), rows(m, c), rows(l, c), ring,
                            stream=s_cmp)
                e_done[c].record(s_cmp)
            with torch.cuda.stream(s_out):
                for c in range(nch):
                    s_out.wait_event(e_done[c])
                    for n, t in (("idx", idx), ("out", out), ("m", m), ("l", l)):
                        rows(host_out[n], c).copy_(rows(t, c), non_blocking=True)
                    e_out[c].record(s_out)
            prev["cmp"][buf], prev["out"] = e_done[-1], e_out
            prev["step"] += 1
            return e_out[-1]

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        ke = max(3, K // 2)
        a, b = E(), E()
        a.record(s_in)
        for _ in range(ke):
            last = e2e_step()
        s_out.wait_event(last)
        b.record(s_out)
        torch.cuda.synchronize()
        ms_e2e = a.elapsed_time(b) / ke
        ms_e2e = max_over_ranks(ms_e2e, world, dev)
        # the chunked path returns what one whole-sequence call returns
        ref = dict(idx=torch.empty_like(idx), out=torch.empty_like(out), m=torch.empty_like(m),
                   l=torch.empty_like(l))
        dsa.forward(p, x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], ref["idx"], ref["out"],
                    ref["m"], ref["l"], ring)
        torch.cuda.synchronize()
        same = all(torch.equal(ref[n].cpu(), host_out[n]) for n in ref)
        del xs, ref  # the second input buffer
        e2e = {"value": job_value(world, S, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "row_chunks": nch,
               "equals_whole_call": same}
        assert dsa.get_status() == 0

    fp8i = fused = None
    if rank == 0:
        fp8i = fp8_indexer_stage(dsa, dev, wl, x, waves, max(2, min(K, 5)), peak_tc)
        fused = fused_topk_stage(dsa, dev, wl, x, idx, max(2, min(K, 5)))
    bwd = None
    if not args.no_bwd and rank == 0:
        del x, out, ring, idx, m, l, flush
        torch.cuda.empty_cache()
        bwd = backward_stage(dsa, dev, max(2, min(K, 5)), peak_tc)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if world == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl)
    launches_per_step = len(waves) * 2 + 1
    traffic = kernel_traffic("attn_fwd_tc.cu", "attn_fwd_tc_dsv32.md")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step,
        "ms_per_step_median": float(np.median(per_step)), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl["name"], "B": 1, "S": S, "topk": k, "H": wl["H"],
                   "d_qk": wl["d_qk"], "d_v": wl["d_v"], "H_I": wl["H_I"], "d_I": wl["d_I"],
                   "wave_rows": W, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (q 4.8 GB) and a 256 MiB L2 flush between steps"},
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_tc_kernel",
                     "achieved": attn_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak_tc,
                     "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                     "peak_source": f"{peaks['source']} {peak_key} (of measured; clocks "
                                    f"{'at max, no power cap' if burst else 'below max or capped'})",
                     "traffic": traffic},
        "tensor_frac_indexer_plus_attention": tensor_frac,
        "tensor_frac_indexer_plus_attention_of_sustained": tensor_frac_sust,
        "stages": {"indexer_ms": t_idx, "topk_ms": t_topk, "attention_ms": t_attn,
                   "indexer_tflops": f_idx / (t_idx * 1e-3) / 1e12,
                   "attention_tflops": attn_tflops,
                   "topk_gbs": topk_bytes / (t_topk * 1e-3) / 1e9,
                   "topk_hbm_frac": topk_bytes / (t_topk * 1e-3) / 1e9 / peaks["hbm_gbs"],
                   "gather_bytes": gather_bytes,
                   "gather_gbs": gather_bytes / (t_attn * 1e-3) / 1e9,
                   "gather_note": "selected kv rows L2 -> shared memory inside the attention "
                                  "kernel (kv is L2-resident); 2 x 576 B per selected pair"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "wall_s_timed": t_wall,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "backward": bwd,
        "fp8_indexer": fp8i,
        "fused_topk": fused,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
