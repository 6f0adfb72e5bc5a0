"""Failure detection on the GPU without a fault: a wait that runs out.

With MK_TEST_STALL set, the step's first wait targets a counter that nothing
signals; after the wait limit (MK_WAIT_NS, short here) the kernel records a
timeout and every CTA leaves. The host sees MK_ERR_TIMEOUT from
mk_step_status, which also resets the device state, and the next step runs
normally and still matches the oracle.
"""
import numpy as np
import pytest

import parity
from synth import configs

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_next_step_recovers(monkeypatch):
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    import oracle

    cfg = configs.TINY
    ctx = cfg["ctx"]
    monkeypatch.setenv("MK_WAIT_NS", "50000000")  # 50 ms, read when the weights load
    model = workload.load_synthetic(cfg, max_batch=1, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv = mk.KVCache(model, 1, ctx + 8)
    workload.prefill(kv, cfg, ctx)
    tok = workload.tokens(cfg, 0, 1, 1)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float32, device="cuda")
    pos = torch.tensor([ctx], dtype=torch.int32, device="cuda")

    monkeypatch.setenv("MK_TEST_STALL", "1")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    with pytest.raises(mk.MKError) as e:
        model.check()
    assert e.value.code == mk.ERR_TIMEOUT

    monkeypatch.delenv("MK_TEST_STALL")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    model.check()
    om = oracle.Model(cfg)
    okv = oracle.KV(om, 1, ctx + 8)
    okv.prefill(cfg["seed"], ctx)
    ref = oracle.decode(om, okv, tok, [ctx])["logits"].reshape(1, -1)
    err = np.abs(logits.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= parity.MAX_ABS and err.mean() <= parity.MEAN_ABS


def test_skipped_signal_times_out_and_the_next_step_recovers(monkeypatch):
    # host-side injection (MK_FAULT=skip_signal): no CTA signals the end of
    # layer 0's first projection, so the stages that read that projection
    # run into their wait limit; nothing faults, the step reports a timeout
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    import oracle

    cfg = configs.TINY
    ctx = cfg["ctx"]
    monkeypatch.setenv("MK_WAIT_NS", "50000000")
    model = workload.load_synthetic(cfg, max_batch=1, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv = mk.KVCache(model, 1, ctx + 8)
    workload.prefill(kv, cfg, ctx)
    tok = workload.tokens(cfg, 0, 1, 1)
    logits = torch.empty((1, cfg["vocab"]), dtype=torch.float32, device="cuda")
    pos = torch.tensor([ctx], dtype=torch.int32, device="cuda")

    monkeypatch.setenv("MK_FAULT", "skip_signal")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    with pytest.raises(mk.MKError) as e:
        model.check()
    assert e.value.code == mk.ERR_TIMEOUT and "timed out" in str(e.value)

    monkeypatch.delenv("MK_FAULT")
    model.decode_step(kv, torch.from_numpy(tok).cuda(), pos, logits)
    model.check()
    om = oracle.Model(cfg)
    okv = oracle.KV(om, 1, ctx + 8)
    okv.prefill(cfg["seed"], ctx)
    ref = oracle.decode(om, okv, tok, [ctx])["logits"].reshape(1, -1)
    err = np.abs(logits.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= parity.MAX_ABS and err.mean() <= parity.MEAN_ABS
