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


def _e4m3_values():
    """Every FP8 E4M3 code's value from the format's definition (OCP MX v1.0):
    sign bit, 4 exponent bits of bias 7, 3 mantissa bits; exponent field 0
    holds the subnormals m * 2^-9; codes 0x7F / 0xFF are NaN."""
    out = np.empty(256)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            out[c] = np.nan
            continue
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        out[c] = -v if s else v
    return out


def test_e4m3_values_closed_form():
    v = _e4m3_values()
    assert v[0x38] == 1.0 and v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x07] == 7 * 2.0 ** -9 and v[0xB8] == -1.0 and v[0x30] == 0.5 and v[0x3C] == 1.5
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes 0 .. 0x7E are increasing in value


def test_e4m3_rne_nearest_even_brute_force():
    # every representable value maps to its own code; every midpoint between
    # neighbours goes to the one with the even code; random values go to the
    # nearest code (brute force over the 127 non-negative finite values)
    v = _e4m3_values()
    pos = v[:0x7F]
    for c in range(0x7F):
        assert synth.e4m3_rne(float(pos[c])) == c
        assert synth.e4m3_rne(float(-pos[c])) == (0x80 | c)
    for c in range(0x7E):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)
        assert float(mid) == (pos[c] + pos[c + 1]) / 2  # exact in fp32
        want = c if c % 2 == 0 else c + 1
        assert synth.e4m3_rne(float(mid)) == want, hex(c)
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.standard_normal(4000) * 16, rng.uniform(-0.03, 0.03, 2000),
                         rng.uniform(-460, 460, 2000)]).astype(np.float32)
    for x in xs:
        a = abs(float(x))
        d = np.abs(pos - a)
        best = np.flatnonzero(d == d.min())
        c = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        if x < 0 or (x == 0 and np.signbit(x)):
            c |= 0x80
        assert synth.e4m3_rne(float(x)) == c, (float(x), c)
    # saturation and NaN
    assert synth.e4m3_rne(464.0) == 0x7E and synth.e4m3_rne(1e9) == 0x7E and synth.e4m3_rne(-1e9) == 0xFE
    assert synth.e4m3_rne(float("nan")) == 0x7F


def test_e4m3_rne_matches_torch():
    # torch's float8_e4m3fn conversion (round to nearest even) inside the
    # finite range
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.standard_normal(20000) * 16, rng.uniform(-447, 447, 5000),
                         rng.uniform(-0.02, 0.02, 5000)]).astype(np.float32)
    mine = np.array([synth.e4m3_rne(float(x)) for x in xs], dtype=np.uint8)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_mxfp8_recipe_codes_and_scales():
    # codes: sigma-16 normal draws rounded to E4M3 (mean 0, std about 16, no
    # saturation); scales: E8M0 bytes 117 and 118 (2^-10, 2^-9), both frequent
    v = _e4m3_values()
    codes = synth.fill_e4m3_host(1 << 16, 1234, synth.tensor_id(synth.GATE, 0, 3))
    x = v[codes]
    assert not np.isnan(x).any() and np.abs(x).max() <= 96
    assert abs(x.mean()) < 0.3 and abs(x.std() - 16.0) < 0.3
    part = synth.fill_e4m3_host(100, 1234, synth.tensor_id(synth.GATE, 0, 3), index0=5000)
    assert np.array_equal(part, codes[5000:5100])
    sc = synth.fill_e8m0_host(1 << 14, 1234, synth.tensor_id(synth.GATE_SCALE, 0, 3))
    assert set(np.unique(sc)) == {117, 118}
    assert 0.45 < (sc == 118).mean() < 0.55
    d = configs.DEEP
    for k in synth.F8_KINDS:
        r, c, _, _ = synth.weight_spec(d, k)
        rs, cs, _, _ = synth.weight_spec(d, synth.SCALE_OF[k])
        assert (rs, cs) == (r, c // 32)
