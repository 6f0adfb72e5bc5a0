"""GPU parity: the CUDA megakernel (through the C ABI) against the CPU oracle.

Every case runs both sides on the same seeded weights, KV and tokens and
applies the parity bar in tests/parity.py: routed experts identical where the
oracle's router margin exceeds 1e-3, logits within max-abs 2e-2 / mean-abs
2e-3 of the fp64 oracle. Sizes span several tiles per stage and ragged tails
(partial last KV chunk, vocab not a multiple of the tile, sequences at
different positions).
"""
import numpy as np
import pytest

import parity
from synth import configs

pytestmark = pytest.mark.gpu


def _run(cfg, B, T, steps, ctx, lazy=False, **kw):
    g, _ = parity.run_gpu(cfg, B, T, steps, ctx, **kw)
    o = parity.run_oracle(cfg, g, ctx, B, T, lazy=lazy)
    rep = parity.compare(cfg, g, o, B, T)
    print(cfg["name"], B, T, rep)
    return g, o, rep


def test_generator_device_matches_host():
    import torch
    import synth
    n = 1 << 20
    for kind, sigma, mean in ((synth.WQ, 0.02, 0.0), (synth.ATTN_NORM, 0.02, 1.0), (synth.KV_LATENT, 1.0, 0.0)):
        tid = synth.tensor_id(kind, 3, 1)
        d = torch.empty(n, dtype=torch.int16, device="cuda")
        synth.fill_bf16_cuda(d.data_ptr(), n, 1234, tid, sigma, mean, 17)
        torch.cuda.synchronize()
        h = synth.fill_bf16_host(n, 1234, tid, sigma, mean, 17)
        assert np.array_equal(d.cpu().numpy().view(np.uint16), h)


def test_tiny_sixteen_steps():
    cfg = configs.TINY
    _run(cfg, 1, 1, cfg["steps"], cfg["ctx"])


def test_tiny_batch_ragged_positions():
    cfg = configs.TINY
    pos0 = np.array([64, 1, 130], dtype=np.int32)
    _run(cfg, 3, 1, 3, 131, positions_fn=lambda s: pos0 + s)


def test_mid_batch1():
    cfg = configs.MID
    _run(cfg, 1, 1, 2, cfg["ctx"])


@pytest.mark.parametrize("B", [3, 4, 6, 8])
def test_mid_batched(B):
    # 3: the one-token register path run once per token; 6: the shared
    # expert in token groups of 4 and 2; every batch: routed experts on
    # their own tokens only
    cfg = configs.MID
    _run(cfg, B, 1, 1, cfg["ctx"])


def test_deep_reduced_layers_batch1():
    cfg = configs.scaled(configs.DEEP, n_layers=3)
    _run(cfg, 1, 1, 2, cfg["ctx"])


def test_deep_reduced_layers_batch2_ragged():
    cfg = configs.scaled(configs.DEEP, n_layers=2)
    pos0 = np.array([8192, 1000], dtype=np.int32)
    _run(cfg, 2, 1, 1, 8192, positions_fn=lambda s: pos0 + s)


def test_dense_reduced_layers():
    cfg = configs.scaled(configs.DENSE, n_layers=2)
    _run(cfg, 1, 1, 1, cfg["ctx"])
    _run(cfg, 8, 1, 1, cfg["ctx"])


def test_paged_cache_with_permuted_block_table():
    cfg = configs.scaled(configs.MID, n_layers=2)
    rng = np.random.default_rng(3)

    def table(pps, B=2):
        return rng.permutation(B * pps).astype(np.int32).reshape(B, pps)

    _run(cfg, 2, 1, 2, 700, block_table=table)


def test_verify_step_reduced_layers():
    cfg = configs.scaled(configs.VERIFY, n_layers=2)
    g, o, rep = _run(cfg, 8, 7, 1, 2000, want_accept=True)
    assert np.all((g[0]["accept"] >= 1) & (g[0]["accept"] <= 7))


@pytest.mark.parametrize("name,B", [("mid", 4), ("deep", 2)])
def test_separate_router_stage(monkeypatch, name, B):
    # the schedule with its own router stage (used for one token, or when the
    # output projection splits K); by default steps of two or more tokens fold
    # the router into the output projection
    monkeypatch.setenv("MK_ROUTER_STAGE", "1")
    cfg = configs.scaled(configs.ALL[name], n_layers=2)
    _run(cfg, B, 1, 1, cfg["ctx"])
