#!/usr/bin/env python3
"""Decode-step benchmark of the single-launch MoE megakernel on GB300.

Workload (one "step" = one decode step of every sequence through all layers,
the LM head included, in one kernel launch): the deep MoE decoder -- 92 MLA
layers, d_model 2048, 64 routed experts top-8 + 1 shared, vocab 64000, about
59 GB of bf16 weights -- at batch 1 with 8192 cached positions, seeded
synthetic weights and KV. Batch 8 is measured in the same run and reported
under "extra". Weights (59 GB) are far larger than L2, so no flush is needed
between steps.

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth import configs  # noqa: E402

METRIC = "decode tokens/s at batch 1/8; achieved HBM GB/s as % of GB300 peak"
UNIT = "tokens/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def workload_name(cfg, B, T, ctx):
    return f"{cfg['name']}-moe-{cfg['n_layers']}L-{'mla' if cfg['attn_kind'] else 'gqa'}-b{B}-t{T}-ctx{ctx}"


def algorithmic_bytes(cfg, B, T, positions, route_idx=None):
    """bf16 bytes the step must move: every non-routed weight, the union of
    the routed experts actually selected (per layer), the LM head, B*T
    embedding rows, the cached KV read (positions before the step) and the KV
    written for the new positions."""
    d, L, V = cfg["d_model"], cfg["n_layers"], cfg["vocab"]
    per = 2 * d
    if cfg["attn_kind"] == 0:
        hq, hkv, hd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
        per += d * hq * hd * 2 + d * hkv * hd * 2
        row = 2 * hkv * hd
    else:
        H, ql, kl = cfg["n_q_heads"], cfg["q_lora_rank"], cfg["kv_lora_rank"]
        nope, rope, vd = cfg["qk_nope_dim"], cfg["qk_rope_dim"], cfg["v_head_dim"]
        per += ql * d + ql + H * (nope + rope) * ql + (kl + rope) * d + kl + H * (nope + vd) * kl + d * H * vd
        row = kl + rope
    E = cfg["n_routed_experts"]
    if E:
        per += E * d
    if cfg["n_shared_experts"]:
        per += 3 * d * cfg["shared_ffn_dim"]
    elems = L * per + V * d + d + B * T * d
    if E:
        expert = 3 * d * cfg["ffn_dim"]
        for l in range(L):
            elems += len(set(np.asarray(route_idx[l]).ravel().tolist())) * expert
    kv_read = sum(int(p) for p in positions) * row * L
    kv_write = B * T * row * L
    return 2 * (elems + kv_read + kv_write)


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None
        self.lines = []

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.p = None
        return self

    def _read(self):
        for line in self.p.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(ws, v):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(cfg, B, T, ctx, sample_layers=23, steps=1, warmup=0):
    """Time the oracle (single thread, fp32 accumulation as the reference step
    is defined) on `sample_layers` layers of the workload and scale to the
    full layer count. Weights and cache are generated before timing; each
    timed step decodes the next position."""
    import oracle
    import synth
    sub = configs.scaled(cfg, n_layers=min(sample_layers, cfg["n_layers"]))
    nl = sub["n_layers"]
    m = oracle.Model(sub)
    kv = oracle.KV(m, B, ctx + (steps + warmup + 1) * T + 1)
    kv.prefill(cfg["seed"], ctx)
    tok = synth.tokens(cfg["seed"], 0, B, T, cfg["vocab"])
    # generate every tensor the step touches (untimed), then time whole steps
    for _ in range(max(1, warmup)):
        oracle.decode(m, kv, tok, [ctx] * B, precision=32)
    times = []
    for i in range(steps):
        t0 = time.perf_counter()
        oracle.decode(m, kv, tok, [ctx + (i + 1) * T] * B, precision=32)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    step_s = dt * cfg["n_layers"] / nl
    return {"value": B * T / step_s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"decode step of {nl} of {cfg['n_layers']} layers (batch {B}, ctx {ctx}) timed "
                      f"{steps}x, median {dt:.2f} s, scaled x{cfg['n_layers'] / nl:g}",
            "seconds_per_step": step_s}


def run_reference(args, cfg, B, T, ctx, ws, rank):
    if rank != 0:
        return
    cb = cpu_baseline(cfg, B, T, ctx, sample_layers=8, steps=max(1, args.steps), warmup=1)
    v = cb["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / v * B * T,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": workload_name(cfg, B, T, ctx), "batch": B, "tokens_per_seq": T, "ctx": ctx},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def timed_steps(model, kv, tok_d, pos_list, logits, K, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for p in pos_list[:K]:
        model.decode_step(kv, tok_d, p, logits, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / K


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--config", default="deep", choices=list(configs.ALL))
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--extra-batch", type=int, default=8, help="second batch size measured in the same run (0: off)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override layer count (profiling runs only)")
    args = ap.parse_args()

    cfg = configs.ALL[args.config]
    if args.layers:
        cfg = configs.scaled(cfg, n_layers=args.layers)
    B, T, ctx = args.batch, cfg["T"], cfg["ctx"]
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, cfg, B, T, ctx, ws, rank)
        return

    import torch

    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload

    torch.cuda.set_device(local)
    Bmax = max(B, args.extra_batch or 0)
    K, W = args.steps, max(3, args.warmup)
    max_ctx = ctx + (K + W + 2) * T + 8
    model = workload.load_synthetic(cfg, max_batch=Bmax, max_tokens_per_seq=T, max_ctx=max_ctx)
    kv = mk.KVCache(model, Bmax, max_ctx)
    workload.prefill(kv, cfg, ctx, batch=Bmax)
    info = model.info()
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()

    def measure(Bm, with_clocks):
        tok = workload.tokens(cfg, 0, Bm, T)
        tok_d = torch.from_numpy(tok).cuda()
        pos_list = [torch.full((Bm,), ctx + i * T, dtype=torch.int32, device="cuda") for i in range(K + W)]
        logits = torch.empty((Bm * T, cfg["vocab"]), dtype=torch.float32, device="cuda")
        for i in range(W):
            model.decode_step(kv, tok_d, pos_list[i], logits)
        model.check()
        idx = model.routing(Bm * T)[0] if cfg["n_routed_experts"] else None
        barrier(ws)
        clk = Clocks(local) if with_clocks else None
        if clk:
            clk.__enter__()
        ms = timed_steps(model, kv, tok_d, pos_list[W:], logits, K, stream)
        if clk:
            clk.__exit__()
        model.check()
        ms = allmax(ws, ms)
        nbytes = algorithmic_bytes(cfg, Bm, T, [ctx + (W + K // 2) * T] * Bm, idx)
        # end to end through the public call with host buffers: pinned tokens and
        # positions copied in, logits copied out, every step
        tok_h = torch.from_numpy(tok).pin_memory()
        pos_h = torch.full((Bm,), ctx + W * T, dtype=torch.int32).pin_memory()
        out_h = torch.empty((Bm * T, cfg["vocab"]), dtype=torch.float32).pin_memory()
        pos_d = torch.empty(Bm, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            tok_d.copy_(tok_h, non_blocking=True)
            pos_d.copy_(pos_h, non_blocking=True)
            model.decode_step(kv, tok_d, pos_d, logits)
            out_h.copy_(logits, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        model.check()
        e2e_ms = allmax(ws, e0.elapsed_time(e1) / K)
        return dict(ms=ms, bytes=nbytes, e2e_ms=e2e_ms, clocks=clk.summary() if clk else None,
                    h2d=tok.nbytes + 4 * Bm, d2h=4 * Bm * T * cfg["vocab"])

    main_r = measure(B, True)
    extra = {}
    if args.extra_batch and args.extra_batch != B:
        r8 = measure(args.extra_batch, False)
        gbs8 = r8["bytes"] / (r8["ms"] * 1e-3) / 1e9
        extra[f"batch{args.extra_batch}"] = {
            "value": ws * args.extra_batch * T / (r8["ms"] * 1e-3), "ms_per_step": r8["ms"],
            "hbm_gbs": gbs8, "frac_of_peak": gbs8 / peak, "bytes_per_step": r8["bytes"],
            "e2e_value": ws * args.extra_batch * T / (r8["e2e_ms"] * 1e-3)}
    if rank != 0:
        return
    ms = main_r["ms"]
    value = ws * B * T / (ms * 1e-3)
    gbs = main_r["bytes"] / (ms * 1e-3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as f:
                tr = json.load(f)
            if tr.get("workload") == workload_name(cfg, B, T, ctx) and tr.get("kernel_build") == kernel_hash():
                traffic = tr.get("bytes_per_launch")
        except Exception:
            traffic = None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded bf16 N(0,0.02) weights, N(0,1) KV)",
        "config": {"workload": workload_name(cfg, B, T, ctx), "batch": B, "tokens_per_seq": T, "ctx": ctx,
                   "layers": cfg["n_layers"], "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (all weights streamed every step)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": traffic, "peak_kind": f"{peak_kind} (hbm_gbs)",
                     "algorithmic_bytes_per_step": main_r["bytes"]},
        "clocks": main_r["clocks"],
        "e2e": {"value": ws * B * T / (main_r["e2e_ms"] * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": main_r["h2d"], "d2h_bytes_per_step": main_r["d2h"]},
        "gpu_launches": K,
        "kernel": {"grid": info.grid_ctas, "threads": info.threads_per_cta, "smem": info.smem_bytes,
                   "weight_bytes": info.weight_bytes},
        "extra": extra,
    }
    if not args.no_cpu_baseline and ws == 1:
        cb = cpu_baseline(cfg, B, T, ctx)
        cb.pop("seconds_per_step", None)
        line["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)


def kernel_hash():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "moe_decode_megakernel_02_gb300", "csrc")
    for n in sorted(os.listdir(d)):
        with open(os.path.join(d, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
