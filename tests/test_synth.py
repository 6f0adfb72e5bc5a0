"""Pins of the seeded input generator (synth/), CPU only.

The generator is shared by the oracle and the CUDA-path harness, so it is
pinned to things outside itself: published SplitMix64 test vectors, torch's
bf16 rounding, the exact moments of the Irwin-Hall(12) sum, and structural
properties of the recipe.
"""
import os

import numpy as np
import pytest
import torch

import synth
from synth import configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64.txt")


def test_splitmix64_published_vectors():
    lib = synth.host_lib()
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert rows
    for seed, *draws in rows:
        got = [lib.synth_draw(int(seed), j) for j in range(3)]
        assert got == [int(x) for x in draws]


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 3,
                           np.float32([0.0, -0.0, 1.0, 65504.0, 1e-40, -1e-38, 3.0e38]),
                           # exact ties: low 16 bits 0x8000 with even and odd kept bits
                           np.array([0x3f808000, 0x3f818000, 0xbf808000, 0x40008000], dtype=np.uint32).view(np.float32)])
    lib = synth.host_lib()
    mine = np.array([lib.synth_bf16_rne(float(v)) for v in vals], dtype=np.uint16)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_normal_moments_irwin_hall():
    # S = sum of 12 uniform 16-bit draws; (S - 6*65535)/65535 has mean 0 and
    # variance 12 * (65536^2 - 1) / (12 * 65535^2) = (65536^2-1)/65535^2.
    n = 1 << 20
    x = synth.bf16_to_f32(synth.fill_bf16_host(n, 7, synth.tensor_id(synth.KV_K, 3, 1), 1.0)).astype(np.float64)
    var = (65536.0 ** 2 - 1) / 65535.0 ** 2
    # bf16 rounding adds variance ~ (2^-8)^2 * E[x^2] / 12 relative; negligible at this tolerance
    assert abs(x.mean()) < 5 * np.sqrt(var / n)
    assert abs(x.var() - var) < 6 * np.sqrt(2 * var ** 2 / n) + 1e-4
    assert x.min() >= -6.0 and x.max() <= 6.0
    # kurtosis of Irwin-Hall(12) standardised: 3 - 6/(5*12) = 2.9
    k = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(k - 2.9) < 0.02


def test_fill_is_index_addressable_and_thread_invariant():
    tid = synth.tensor_id(synth.WQ, 2, 0)
    full = synth.fill_bf16_host(300000, 5, tid, 0.02, threads=1)
    par = synth.fill_bf16_host(300000, 5, tid, 0.02, threads=8)
    part = synth.fill_bf16_host(1000, 5, tid, 0.02, index0=123456)
    assert np.array_equal(full, par)
    assert np.array_equal(full[123456:124456], part)


def test_gain_recipe_mean_one():
    g = synth.bf16_to_f32(synth.fill_bf16_host(4096, 1, synth.tensor_id(synth.ATTN_NORM, 0), 0.02, 1.0))
    assert abs(g.mean() - 1.0) < 0.003 and 0.015 < g.std() < 0.025


def test_tensor_ids_distinct_and_streams_differ():
    ids = {synth.tensor_id(k, l, e) for k in range(1, 44) for l in range(-1, 93) for e in (0, 1, 63)}
    assert len(ids) == 43 * 94 * 3
    a = synth.fill_bf16_host(64, 1, synth.tensor_id(synth.GATE, 0, 0), 0.02)
    b = synth.fill_bf16_host(64, 1, synth.tensor_id(synth.GATE, 0, 1), 0.02)
    assert not np.array_equal(a, b)


def test_tokens_in_range_and_spread():
    V = 1024
    t = [synth.token(0, s, b, 0, V) for s in range(64) for b in range(32)]
    assert min(t) >= 0 and max(t) < V and len(set(t)) > 500


@pytest.mark.parametrize("name", list(configs.ALL))
def test_weight_specs_cover_model(name):
    cfg = configs.ALL[name]
    total = sum(r * c for _, _, _, r, c, _, _ in synth.weight_tensors(cfg))
    assert 2 * total == configs.weight_bytes(cfg)
    if name == "deep":
        assert 58e9 < 2 * total < 61e9  # about 59 GB of bf16 weights
