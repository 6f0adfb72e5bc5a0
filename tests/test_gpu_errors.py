"""Error reporting and the stage trace on the GPU, without any fault.

Bad inputs: the kernel checks every token id and position of the step before
it reads or writes anything with them (each CTA reaches the same verdict and
leaves); the host sees MK_ERR_INVALID_ARG from mk_step_status, which resets
the device state, and the next step with good inputs matches the oracle.

Trace: with MK_TRACE=1 at load, every CTA records (stage << 16 | layer,
items, t_wait, t_ready, t_end) for each stage it takes part in; the records
must cover every stage of every layer and be ordered in time.
"""
import numpy as np
import pytest

import parity
from synth import configs

pytestmark = pytest.mark.gpu


def _tiny_setup(monkeypatch=None):
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    cfg = configs.TINY
    ctx = cfg["ctx"]
    model = workload.load_synthetic(cfg, max_batch=2, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv = mk.KVCache(model, 2, ctx + 8)
    workload.prefill(kv, cfg, ctx)
    logits = torch.empty((2, cfg["vocab"]), dtype=torch.float32, device="cuda")
    return cfg, ctx, model, kv, logits


def _oracle_logits(cfg, ctx, tok):
    import oracle
    om = oracle.Model(cfg)
    okv = oracle.KV(om, len(tok), ctx + 8)
    okv.prefill(cfg["seed"], ctx)
    return oracle.decode(om, okv, tok, [ctx] * len(tok))["logits"].reshape(len(tok), -1)


@pytest.mark.parametrize("what", ["token", "negative_token", "position", "negative_position"])
def test_out_of_range_inputs_are_reported_and_the_next_step_recovers(what):
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    cfg, ctx, model, kv, logits = _tiny_setup()
    tok = workload.tokens(cfg, 0, 2, 1)
    bad_tok, bad_pos = tok.copy(), np.array([ctx, ctx], dtype=np.int32)
    if what == "token":
        bad_tok[1, 0] = cfg["vocab"]
    elif what == "negative_token":
        bad_tok[0, 0] = -1
    elif what == "position":
        bad_pos[1] = ctx + 8  # one past the cache's last position
    else:
        bad_pos[0] = -3
    model.decode_step(kv, torch.from_numpy(bad_tok).cuda(), torch.from_numpy(bad_pos).cuda(), logits)
    with pytest.raises(mk.MKError) as e:
        model.check()
    assert e.value.code == mk.ERR_INVALID_ARG and "out of range" in str(e.value)
    # the state was reset: the next step runs and matches the oracle
    model.decode_step(kv, torch.from_numpy(tok).cuda(), torch.tensor([ctx, ctx], dtype=torch.int32, device="cuda"),
                      logits)
    model.check()
    err = np.abs(logits.cpu().numpy().astype(np.float64) - _oracle_logits(cfg, ctx, tok))
    assert err.max() <= parity.MAX_ABS and err.mean() <= parity.MEAN_ABS


@pytest.mark.parametrize("name,B", [("mid", 1), ("deep", 2)])
def test_trace_covers_every_stage_of_every_layer(monkeypatch, name, B):
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import tracing, workload
    monkeypatch.setenv("MK_TRACE", "1")
    cfg = configs.scaled(configs.ALL[name], n_layers=3)
    ctx = 700
    model = workload.load_synthetic(cfg, max_batch=B, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv = mk.KVCache(model, B, ctx + 8)
    workload.prefill(kv, cfg, ctx)
    logits = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device="cuda")
    model.decode_step(kv, torch.from_numpy(workload.tokens(cfg, 0, B, 1)).cuda(),
                      torch.full((B,), ctx, dtype=torch.int32, device="cuda"), logits)
    model.check()
    per_cta = model.trace()
    G = model.info().grid_ctas
    assert len(per_cta) == G
    seen = set()
    for recs in per_cta:
        assert 0 < len(recs) < mk.TRACE_CAP
        for r in recs:
            code = int(r["code"])
            assert not code & 0x80000000  # item-level records only with MK_TRACE >= 2
            assert r["t_wait"] <= r["t_ready"] <= r["t_end"], r
            seen.add((code & 0xFFFF, tracing.stage_name(code)))
    L = cfg["n_layers"]
    mla = cfg["attn_kind"] == 1
    # (MLA: the absorbed-query and value up-projection stages, QLAT and UV,
    # run on their own only when they are not folded into QB and the combine)
    want = ["A", "ATTN", "COMB", "O", "FFN", "ROUTE"] + (["QB", "APP"] if mla else [])
    if B == 1:
        want.append("ROUTER")  # steps of two or more tokens fold the router into O
    for l in range(L):
        for st in want:
            assert (l, st) in seen, f"layer {l}: no {st} record"
    assert (L, "INIT") in seen and (L, "LM") in seen
    summ = tracing.summary(per_cta, L)
    assert summ["layer_us"] is not None and summ["layer_us"] > 0
    print(name, B, "layer us", summ["layer_us"], "stage spans", summ["stage_span_us"])


@pytest.mark.parametrize("model_first", [True, False])
def test_model_and_caches_free_in_either_order(model_first):
    # a model freed while its caches are alive (as happens when the garbage
    # collector finalises a cycle holding both) gives up its device memory
    # at once; the caches keep working on their own memory and the model's
    # host record goes with the last of them -- no write into freed memory
    import ctypes
    import gc
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    cfg = configs.TINY
    ctx = 40
    model = workload.load_synthetic(cfg, max_batch=2, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv1, kv2 = mk.KVCache(model, 2, ctx + 8), mk.KVCache(model, 2, ctx + 8)
    workload.prefill(kv1, cfg, ctx)
    rows = kv1.read(0, 1, 0, ctx)
    if model_first:
        model.close()
        assert np.array_equal(kv1.read(0, 1, 0, ctx), rows)  # the cache's own memory is intact
        kv1.close()
        kv2.close()
    else:
        kv2.close()
        kv1.close()
        model.close()
    # freed chunks are consolidated and handed out again: corrupted heap
    # metadata would abort the process here
    gc.collect()
    junk = [bytearray(n) for n in (24, 48, 96, 200, 1000, 5000) for _ in range(200)]
    del junk
    ctypes.CDLL("libc.so.6").malloc_trim(0)


@pytest.mark.parametrize("name,B,T", [("deep", 2, 1), ("verify", 8, 7), ("dense", 8, 1)])
def test_debug_mode_checks_pass_and_parity_holds(monkeypatch, name, B, T):
    # MK_DEBUG=1: shared-memory canaries at the end of every ring slot and
    # after the staging area (written when a CTA starts, compared when it
    # leaves) and the expert units' token-map check; a clean step reports
    # MK_OK and still matches the oracle (the deep and verify cases stream
    # MLA chunks, 64-row tensor-core tiles and expert down tiles through
    # the ring; dense B 8 the split-panel norm inputs)
    monkeypatch.setenv("MK_DEBUG", "1")
    cfg = configs.scaled(configs.ALL[name], n_layers=2)
    ctx = min(cfg["ctx"], 2000)
    g, _ = parity.run_gpu(cfg, B, T, 1, ctx, want_accept=T > 1)
    o = parity.run_oracle(cfg, g, ctx, B, T)
    rep = parity.compare(cfg, g, o, B, T)
    print(name, B, T, "debug mode", rep)


def test_debug_mode_scratch_guard_report(monkeypatch):
    # MK_DEBUG=1: the scratch guards hold after a clean step; with
    # MK_FAULT=corrupt_guard the host overwrites one before the check, the
    # step reports MK_ERR_STATE naming the guard, and (the guard restored)
    # the next step reports MK_OK and matches the oracle
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    import oracle

    monkeypatch.setenv("MK_DEBUG", "1")
    cfg = configs.TINY
    ctx = cfg["ctx"]
    model = workload.load_synthetic(cfg, max_batch=1, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv = mk.KVCache(model, 1, ctx + 8)
    workload.prefill(kv, cfg, ctx)
    tok = workload.tokens(cfg, 0, 1, 1)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float32, device="cuda")
    pos = torch.tensor([ctx], dtype=torch.int32, device="cuda")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    model.check()
    monkeypatch.setenv("MK_FAULT", "corrupt_guard")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    with pytest.raises(mk.MKError) as e:
        model.check()
    assert e.value.code == mk.ERR_STATE and "scratch guard" in str(e.value)
    monkeypatch.delenv("MK_FAULT")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    model.check()
    om = oracle.Model(cfg)
    okv = oracle.KV(om, 1, ctx + 8)
    okv.prefill(cfg["seed"], ctx)
    ref = oracle.decode(om, okv, tok, [ctx])["logits"].reshape(1, -1)
    err = np.abs(logits.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= parity.MAX_ABS and err.mean() <= parity.MEAN_ABS
