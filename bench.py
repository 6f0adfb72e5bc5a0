#!/usr/bin/env python3
"""Decode-step benchmark of the single-launch MoE megakernel on GB300.

Workload (one "step" = one decode step of every sequence through all layers,
the LM head included, in one kernel launch): the deep MoE decoder -- 92 MLA
layers, d_model 2048, 64 routed experts top-8 + 1 shared, vocab 64000, about
59 GB of bf16 weights -- at batch 1 with 8192 cached positions, seeded
synthetic weights and KV. Every timed step decodes the next position with its
own token ids. Weights (59 GB) are far larger than L2, so no flush is needed
between steps.

The same run measures, under "extra", the deep model at batch 2, 4 and 8,
the speculative verify step (batch 8 x 7 tokens), the mid MoE model at batch
1, 4 and 8 and the dense model at batch 1 and 8 (`--extra` chooses).

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
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
    """Bytes the step must move: every non-routed weight, the union of the
    routed experts actually selected (per layer), the LM head, B*T embedding
    rows, the cached KV read (positions before the step) and the KV written
    for the new positions; 2 bytes per element, and for MXFP8 expert weights
    1 + 1/32 (a code, and a scale byte per 32 codes)."""
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
    ex = 0  # expert weight elements
    if cfg["n_shared_experts"]:
        ex += L * 3 * d * cfg["shared_ffn_dim"]
    elems = L * per + V * d + d + B * T * d
    if E:
        expert = 3 * d * cfg["ffn_dim"]
        for l in range(L):
            ex += len(set(np.asarray(route_idx[l]).ravel().tolist())) * expert
    kv_read = sum(int(p) for p in positions) * row * L
    kv_write = B * T * row * L
    ex_bytes = ex * 33 // 32 if cfg.get("expert_format", 0) == 1 else 2 * ex
    return 2 * (elems + kv_read + kv_write) + ex_bytes


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
            time.sleep(0.3)  # the first sample lands before the timed region starts
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
        sm, mx, reasons, power = [], 0.0, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(power) if power else None}


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


def host_facts():
    """Core count and CPU model of this host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def cpu_baseline(cfg, B, T, ctx, sample_layers=23, steps=3):
    """Time the oracle (one thread pinned to one core, fp32 accumulation as the
    step is defined) on `sample_layers` layers of the workload and scale to
    the full layer count. Weights and cache are generated before timing (with
    every core); each timed step decodes the next position with its own
    token ids."""
    import oracle
    import synth
    sub = configs.scaled(cfg, n_layers=min(sample_layers, cfg["n_layers"]))
    nl = sub["n_layers"]
    m = oracle.Model(sub)
    kv = oracle.KV(m, B, ctx + (steps + 2) * T + 1)
    kv.prefill(cfg["seed"], ctx)
    tok = synth.tokens(cfg["seed"], 0, B, T, cfg["vocab"])
    # generate every tensor the step touches (untimed), then time whole steps
    oracle.decode(m, kv, tok, [ctx] * B, precision=32)
    facts = host_facts()
    cores = sorted(os.sched_getaffinity(0))
    pin = cores[0]
    os.sched_setaffinity(0, {pin})  # this thread only: the oracle's arithmetic is single-threaded
    times = []
    try:
        for i in range(steps):
            t = synth.tokens(cfg["seed"], i + 1, B, T, cfg["vocab"])
            pos = [ctx + (i + 1) * T] * B
            # the step's routed experts are generated on first use: run it
            # once untimed, then time the same step (it rewrites the same
            # cache rows with the same values)
            oracle.decode(m, kv, t, pos, precision=32)
            t0 = time.perf_counter()
            oracle.decode(m, kv, t, pos, precision=32)
            times.append(time.perf_counter() - t0)
    finally:
        os.sched_setaffinity(0, set(cores))
    dt = statistics.median(times)
    step_s = dt * cfg["n_layers"] / nl
    return {"value": B * T / step_s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"decode steps of {nl} of {cfg['n_layers']} layers (batch {B}, ctx {ctx}), {steps} timed, "
                      f"median {dt:.2f} s, scaled x{cfg['n_layers'] / nl:g} to the full depth; one thread pinned to "
                      f"core {pin} of {facts['nproc']} ({facts['cpu_model']})",
            "host": facts, "scaled": True, "layer_fraction": nl / cfg["n_layers"], "seconds_per_step": step_s}


def run_reference(args, cfg, B, T, ctx, ws, rank):
    if rank != 0:
        return
    cb = cpu_baseline(cfg, B, T, ctx, sample_layers=8, steps=max(1, args.steps if args.steps <= 5 else 3))
    v = cb["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / v * B * T,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": workload_name(cfg, B, T, ctx), "batch": B, "tokens_per_seq": T, "ctx": ctx,
                       "layers": cfg["n_layers"], "parallelism": f"replicas x{args.gpus}"},
            "scaled": True, "layer_fraction": cb["layer_fraction"],
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": cb["sample"],
                             "host": cb["host"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(model, kv, cfg, Bm, T, ctx, K, W, ws, stream, with_clocks, local, want_accept=False,
            entry="decode_step"):
    """W warm-up steps, then K timed steps (CUDA events on the launch stream),
    each at the next position(s) with its own token ids; then the same K steps
    replayed untimed to read each one's routing (for its algorithmic bytes);
    then K end-to-end steps through the public call with host buffers.
    `entry`: decode_step (one launch per step) or decode_step_unfused (one
    launch per stage, the comparison path)."""
    import torch
    step = getattr(model, entry)
    V = cfg["vocab"]
    toks = [torch.from_numpy(workload_tokens(cfg, i, Bm, T)).cuda() for i in range(W + K)]
    pos_list = [torch.full((Bm,), ctx + i * T, dtype=torch.int32, device="cuda") for i in range(W + K)]
    logits = torch.empty((Bm * T, V), dtype=torch.float32, device="cuda")
    acc = torch.zeros(Bm, dtype=torch.int32, device="cuda") if want_accept else None
    for i in range(W):
        step(kv, toks[i], pos_list[i], logits, acc)
    model.check()
    barrier(ws)
    clk = Clocks(local) if with_clocks else None
    if clk:
        clk.__enter__()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(W, W + K):
        step(kv, toks[i], pos_list[i], logits, acc, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / K
    if clk:
        clk.__exit__()
    model.check()
    barrier(ws)
    ms = allmax(ws, ms)
    # the timed steps again, untimed, for their routing and acceptance
    nbytes, accepted = [], []
    for i in range(W, W + K):
        step(kv, toks[i], pos_list[i], logits, acc)
        idx = model.routing(Bm * T)[0] if cfg["n_routed_experts"] else None
        nbytes.append(algorithmic_bytes(cfg, Bm, T, [ctx + i * T] * Bm, idx))
        if want_accept:
            accepted.append(int(acc.sum().item()))
    model.check()
    # end to end through the public call with host buffers: pinned token ids
    # and positions copied in, logits copied out, every step, positions
    # advancing as in the timed loop
    tok_h = torch.stack([t.cpu() for t in toks[W:]]).pin_memory()
    pos_h = torch.stack([p.cpu() for p in pos_list[W:]]).pin_memory()
    out_h = torch.empty((Bm * T, V), dtype=torch.float32).pin_memory()
    tok_d = torch.empty((Bm, T), dtype=torch.int32, device="cuda")
    pos_d = torch.empty(Bm, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        tok_d.copy_(tok_h[i], non_blocking=True)
        pos_d.copy_(pos_h[i], non_blocking=True)
        step(kv, tok_d, pos_d, logits, acc)
        out_h.copy_(logits, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    model.check()
    e2e_ms = allmax(ws, e0.elapsed_time(e1) / K)
    return dict(ms=ms, bytes=float(np.mean(nbytes)), e2e_ms=e2e_ms, clocks=clk.summary() if clk else None,
                h2d=Bm * T * 4 + 4 * Bm, d2h=4 * Bm * T * V,
                accepted=float(np.mean(accepted)) if accepted else None)


def workload_tokens(cfg, step, B, T):
    from moe_decode_megakernel_02_gb300 import workload
    return workload.tokens(cfg, step, B, T)


def kernel_hash():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "moe_decode_megakernel_02_gb300", "csrc")
    for n in sorted(os.listdir(d)):
        with open(os.path.join(d, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--config", default="deep", choices=list(configs.ALL) + ["deep_mxfp8"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--extra", default="all", choices=["none", "batch8", "all"],
                    help="other measurements in the same run (batch8: the deep model at batch 8 only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override layer count (profiling runs only)")
    args = ap.parse_args()

    cfg = configs.DEEP_MXFP8 if args.config == "deep_mxfp8" else configs.ALL[args.config]
    if args.config == "deep_mxfp8":
        args.extra = "none"
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
    K, W = args.steps, max(3, args.warmup)
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()

    def load(c, Bmax, Tm):
        max_ctx = c["ctx"] + 2 * (K + W + 2) * Tm + 8
        model = workload.load_synthetic(c, max_batch=Bmax, max_tokens_per_seq=Tm, max_ctx=max_ctx)
        kv = mk.KVCache(model, Bmax, max_ctx)
        workload.prefill(kv, c, c["ctx"], batch=Bmax)
        return model, kv

    def extra_line(c, r, Bm, Tm):
        gbs = r["bytes"] / (r["ms"] * 1e-3) / 1e9
        out = {"workload": workload_name(c, Bm, Tm, c["ctx"]), "value": ws * Bm * Tm / (r["ms"] * 1e-3),
               "unit": "positions/s" if Tm > 1 else UNIT, "ms_per_step": r["ms"], "hbm_gbs": gbs,
               "frac_of_peak": gbs / peak, "bytes_per_step": r["bytes"],
               "e2e_value": ws * Bm * Tm / (r["e2e_ms"] * 1e-3)}
        if r["accepted"] is not None:
            out["accepted_tokens_per_s"] = ws * r["accepted"] / (r["ms"] * 1e-3)
            out["mean_accept_length"] = r["accepted"] / Bm
        return out

    extra = {}
    deep_batches = [b for b in (2, 4, 8) if b != B] if args.extra == "all" else ([8] if args.extra == "batch8" else [])
    Bmax = max([B] + deep_batches)
    model, kv = load(cfg, Bmax, T)
    info = model.info()
    main_r = measure(model, kv, cfg, B, T, ctx, K, W, ws, stream, True, local)
    for Bm in deep_batches:
        r = measure(model, kv, cfg, Bm, T, ctx, K, W, ws, stream, False, local)
        extra[f"{cfg['name']}_b{Bm}"] = extra_line(cfg, r, Bm, T)
    if args.extra == "all":
        # the same step as one launch per stage (CUDA graph, programmatic
        # dependent launch): what the single launch buys on this GPU
        for Bm in sorted({B, 8}):
            r = measure(model, kv, cfg, Bm, T, ctx, K, W, ws, stream, False, local, entry="decode_step_unfused")
            extra[f"{cfg['name']}_b{Bm}_unfused"] = extra_line(cfg, r, Bm, T)
    del kv, model
    torch.cuda.empty_cache()
    if args.extra == "all" and not args.layers and args.config == "deep":
        # the speculative verify step: batch 8 x 7 tokens (1 + 6 random drafts)
        vc = configs.VERIFY
        model, kv = load(vc, 8, vc["T"])
        r = measure(model, kv, vc, 8, vc["T"], vc["ctx"], K, W, ws, stream, False, local, want_accept=True)
        extra["verify_b8_t7"] = extra_line(vc, r, 8, vc["T"])
        del kv, model
        torch.cuda.empty_cache()
        for name, batches in (("mid", (1, 4, 8)), ("dense", (1, 8))):
            c = configs.ALL[name]
            model, kv = load(c, max(batches), 1)
            for Bm in batches:
                r = measure(model, kv, c, Bm, 1, c["ctx"], K, W, ws, stream, False, local)
                extra[f"{name}_b{Bm}"] = extra_line(c, r, Bm, 1)
            del kv, model
            torch.cuda.empty_cache()
        # the deep model with MXFP8 expert weights, batch 1 and 8 (a
        # different model: its experts hold other values; bytes counted at
        # 1 + 1/32 per expert weight)
        c = configs.DEEP_MXFP8
        model, kv = load(c, 8, 1)
        for Bm in (1, 8):
            r = measure(model, kv, c, Bm, 1, c["ctx"], K, W, ws, stream, False, local)
            extra[f"deep_mxfp8_b{Bm}"] = extra_line(c, r, Bm, 1)
        del kv, model
        torch.cuda.empty_cache()
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
        "data": "synthetic (seeded bf16 N(0,0.02) weights, N(0,1) KV, per-step token ids)",
        "config": {"workload": workload_name(cfg, B, T, ctx), "batch": B, "tokens_per_seq": T, "ctx": ctx,
                   "layers": cfg["n_layers"], "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (all weights streamed every step)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": traffic, "peak_kind": f"{peak_kind} (hbm_gbs)",
                     "algorithmic_bytes_per_step": main_r["bytes"],
                     "bytes_note": "mean over the timed steps, each counted from its own routing"},
        "clocks": main_r["clocks"],
        "e2e": {"value": ws * B * T / (main_r["e2e_ms"] * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": main_r["h2d"], "d2h_bytes_per_step": main_r["d2h"]},
        "gpu_launches": K,
        "kernel": {"grid": info.grid_ctas, "threads": info.threads_per_cta, "smem": info.smem_bytes,
                   "ring_slots": info.ring_slots, "weight_bytes": info.weight_bytes, "build": kernel_hash()},
        "extra": extra,
    }
    if not args.no_cpu_baseline and ws == 1:
        cb = cpu_baseline(cfg, B, T, ctx)
        cb.pop("seconds_per_step", None)
        line["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
