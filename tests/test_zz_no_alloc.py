"""The allocation-free decode entry point, mk_decode_step_noalloc.

It serves callers that may not allocate device memory on their call path --
code running inside a host framework that owns a fixed memory pool, or a
serving thread that must stay out of the driver's allocator -- by taking the
step's scratch from a static device array of the library. Checked through the
C ABI against the regular mk_decode_step on identical inputs for two calls in
a row (the static array keeps the previous call's contents), plus the size
limit. The file is collected last so that a failure here comes after the rest
of the GPU suite has run.
"""
import numpy as np
import pytest

import parity
from synth import configs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,B", [("tiny", 1), ("mid", 2)])
def test_noalloc_matches_regular_entry_point(name, B):
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    cfg = configs.ALL[name]
    if name == "mid":
        cfg = configs.scaled(cfg, n_layers=2)
    ctx = min(cfg["ctx"], 300)
    model = workload.load_synthetic(cfg, max_batch=B, max_tokens_per_seq=1, max_ctx=ctx + 8)
    kv_a, kv_b = mk.KVCache(model, B, ctx + 8), mk.KVCache(model, B, ctx + 8)
    workload.prefill(kv_a, cfg, ctx)
    workload.prefill(kv_b, cfg, ctx)
    la = torch.empty((B, cfg["vocab"]), dtype=torch.float32, device="cuda")
    lb = torch.full((B, cfg["vocab"]), float("nan"), dtype=torch.float32, device="cuda")
    for step in range(2):
        tok = torch.from_numpy(workload.tokens(cfg, step, B, 1)).cuda()
        pos = torch.full((B,), ctx + step, dtype=torch.int32, device="cuda")
        model.decode_step(kv_a, tok, pos, la)
        model.check()
        model.decode_step_noalloc(kv_b, tok, pos, lb)
        assert torch.isfinite(lb).all()
        d = (la - lb).abs()
        assert d.max().item() <= parity.MAX_ABS and d.mean().item() <= parity.MEAN_ABS, (step, d.max().item())
        # both calls appended the same cache rows
        fa = (kv_a.read(0, 0, ctx + step, 1).astype(np.uint32) << 16).view(np.float32)
        fb = (kv_b.read(0, 0, ctx + step, 1).astype(np.uint32) << 16).view(np.float32)
        assert np.abs(fa - fb).max() <= 0.05


def test_noalloc_rejects_models_beyond_the_static_scratch():
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    # positions up to 300k: the RoPE table alone is ~77 MB of step scratch
    cfg = configs.scaled(configs.DEEP, n_layers=2)
    model = workload.load_synthetic(cfg, max_batch=8, max_tokens_per_seq=1, max_ctx=300_000)
    assert model.info().scratch_bytes > 64 << 20
    kv = mk.KVCache(model, 8, 80)
    tok = torch.zeros((8, 1), dtype=torch.int32, device="cuda")
    pos = torch.full((8,), 10, dtype=torch.int32, device="cuda")
    logits = torch.empty((8, cfg["vocab"]), dtype=torch.float32, device="cuda")
    with pytest.raises(mk.MKError) as e:
        model.decode_step_noalloc(kv, tok, pos, logits)
    assert e.value.code == mk.ERR_UNSUPPORTED and "static scratch" in str(e.value)
