"""The allocation-free decode entry point, mk_decode_step_noalloc.

It serves callers that may not allocate device memory on their call path --
code running inside a host framework that owns a fixed memory pool, or a
serving thread that must stay out of the driver's allocator -- by taking the
step's scratch from a static device array of the library. Checked through the
C ABI against the regular mk_decode_step on identical inputs for two calls in
a row (the static array keeps the previous call's contents), with a check that
the model's own scratch is neither read nor written by it, plus the size
limit. The file is collected last so that a failure here comes after the rest
of the GPU suite has run.
"""
import numpy as np
import pytest

import parity
from synth import configs

pytestmark = pytest.mark.gpu


def _rows_f32(kv, layer, seq, pos, n):
    return (kv.read(layer, seq, pos, n).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("name,B,T", [("tiny", 1, 1), ("mid", 2, 1), ("deep", 2, 2), ("deep_mxfp8", 1, 1)])
def test_noalloc_matches_regular_entry_point(name, B, T):
    # deep, T 2: MLA (the query, absorbed-query, latent-output and new-latent
    # buffers) and the verify extras (row argmaxes, acceptance); larger
    # batch x tokens products of the deep model need more step scratch than
    # the static array holds (the attention partials grow with them)
    import torch
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    cfg = configs.DEEP_MXFP8 if name == "deep_mxfp8" else configs.ALL[name]
    if name != "tiny":
        cfg = configs.scaled(cfg, n_layers=2)
    ctx = min(cfg["ctx"], 300)
    cap = ctx + 2 * T + 8
    model = workload.load_synthetic(cfg, max_batch=B, max_tokens_per_seq=T, max_ctx=cap)
    kv_r, kv_n, kv_x = (mk.KVCache(model, B, cap) for _ in range(3))
    for kv in (kv_r, kv_n, kv_x):
        workload.prefill(kv, cfg, ctx)
    V = cfg["vocab"]
    la = torch.empty((B * T, V), dtype=torch.float32, device="cuda")
    lb = torch.full((B * T, V), float("nan"), dtype=torch.float32, device="cuda")
    lx = torch.empty((B * T, V), dtype=torch.float32, device="cuda")
    acc_r = torch.zeros(B, dtype=torch.int32, device="cuda") if T > 1 else None
    acc_n = torch.zeros(B, dtype=torch.int32, device="cuda") if T > 1 else None
    am_r = torch.zeros(B * T, dtype=torch.int32)
    am_n = torch.zeros(B * T, dtype=torch.int32)
    for step in range(2):
        tok = torch.from_numpy(workload.tokens(cfg, step, B, T)).cuda()
        other = torch.from_numpy(workload.tokens(cfg, step + 100, B, T)).cuda()
        pos = torch.full((B,), ctx + step * T, dtype=torch.int32, device="cuda")
        model.decode_step(kv_r, tok, pos, la, acc_r)
        model.check()
        if T > 1:
            model.last_argmax(am_r)
        # another step with other tokens leaves unrelated data in the model's
        # own scratch: a pointer the allocation-free path failed to move to
        # its static array would read that data and change the result
        model.decode_step(kv_x, other, pos, lx, acc_r.clone() if T > 1 else None)
        model.check()
        before = model.scratch()
        model.decode_step_noalloc(kv_n, tok, pos, lb, acc_n)
        # ... and nothing of the allocation-free step lands there
        assert np.array_equal(before, model.scratch()), "mk_decode_step_noalloc wrote into the model's scratch"
        assert torch.isfinite(lb).all()
        d = (la - lb).abs()
        assert d.max().item() <= parity.MAX_ABS and d.mean().item() <= parity.MEAN_ABS, (step, d.max().item())
        if T > 1:
            model.last_argmax(am_n)
            assert torch.equal(acc_r.cpu(), acc_n.cpu()), (acc_r, acc_n)
            top = torch.topk(la, 2, dim=1).values
            clear = ((top[:, 0] - top[:, 1]) > 2 * d.max(dim=1).values).cpu()
            assert torch.equal(am_r[clear], am_n[clear])
        # both calls appended the same cache rows (every layer and sequence;
        # bf16 values, which may differ by rounding of the summation order)
        for l in range(cfg["n_layers"]):
            for b in range(B):
                fa = _rows_f32(kv_r, l, b, ctx + step * T, T)
                fb = _rows_f32(kv_n, l, b, ctx + step * T, T)
                assert np.all(np.abs(fa - fb) <= 1e-3 + np.abs(fa) / 64), (l, b)
        if cfg["n_routed_experts"]:
            with pytest.raises(mk.MKError) as e:
                model.routing(B * T)
            assert e.value.code == mk.ERR_STATE


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
