"""Pins of the oracle's building blocks (CPU only).

Each block is checked against something other than itself: a closed form, a
library routine the oracle does not use (scipy softmax/expit, numpy complex
exponentials, numpy stable argsort), exact rational arithmetic, or an
invariant that a dropped term / wrong sign / wrong index would break.
"""
import numpy as np
import pytest
from scipy.special import expit, softmax as sp_softmax

import oracle
import synth


def bf16(x):
    """float array -> bf16 bits via torch-free truncation-safe path (used only to build inputs)."""
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rmsnorm_closed_form():
    # x = c * ones -> out_i = g_i * c / sqrt(c^2 + eps)
    rng = np.random.default_rng(1)
    g = bf16(1 + 0.02 * rng.standard_normal(64))
    gf = synth.bf16_to_f32(g).astype(np.float64)
    for c in (3.0, -0.5, 1e-3):
        out = oracle.rmsnorm(np.full(64, c), g, 1e-6)
        assert np.allclose(out, gf * c / np.sqrt(c * c + 1e-6), rtol=1e-14, atol=0)
    # alternating signs have the same mean square
    x = np.tile([2.0, -2.0], 32)
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), gf * np.sign(x), rtol=1e-14)


def test_rope_against_complex_rotation():
    rng = np.random.default_rng(2)
    for dim in (4, 64, 128):
        x = rng.standard_normal(dim)
        half = dim // 2
        for pos in (0, 1, 77, 8191):
            z = (x[:half] + 1j * x[half:]) * np.exp(1j * pos * 1e4 ** (-2.0 * np.arange(half) / dim))
            out = oracle.rope(x, pos, 1e4)
            assert np.allclose(out[:half], z.real, atol=1e-12)
            assert np.allclose(out[half:], z.imag, atol=1e-12)


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    assert np.array_equal(oracle.rope(q, 0, 1e4), q)
    assert np.isclose(np.linalg.norm(oracle.rope(q, 1234, 1e4)), np.linalg.norm(q), rtol=1e-13)
    a = oracle.rope(q, 10, 1e4) @ oracle.rope(k, 3, 1e4)
    b = oracle.rope(q, 510, 1e4) @ oracle.rope(k, 503, 1e4)
    assert np.isclose(a, b, rtol=1e-10)


def test_softmax_against_scipy():
    rng = np.random.default_rng(4)
    for n in (1, 2, 64, 1000):
        x = rng.standard_normal(n) * 5
        p = oracle.softmax(x)
        assert np.allclose(p, sp_softmax(x), rtol=1e-13, atol=1e-300)
        assert abs(p.sum() - 1) < 1e-12
        assert np.allclose(oracle.softmax(x + 100.0), p, rtol=1e-12)


def test_topk_against_stable_sort_and_invariants():
    rng = np.random.default_rng(5)
    for n, k in ((8, 2), (64, 6), (64, 8), (5, 5)):
        for _ in range(50):
            lg = rng.standard_normal(n)
            idx, w, margin = oracle.topk(lg, k)
            p = sp_softmax(lg)
            ref = np.argsort(-p, kind="stable")[:k]
            assert np.array_equal(idx, ref)
            assert len(set(idx.tolist())) == k
            assert np.isclose(w.sum(), 1.0, atol=1e-14)
            assert np.allclose(w, p[ref] / p[ref].sum(), rtol=1e-13)
            unsel = np.setdiff1d(np.arange(n), idx)
            assert all(p[i] >= p[j] for i in idx for j in unsel)
            srt = np.sort(lg)[::-1]
            if k < n:
                assert np.isclose(margin, srt[k - 1] - srt[k], rtol=0, atol=1e-15)
            else:
                assert np.isinf(margin)


def test_topk_ties_pick_lower_index():
    lg = np.array([0.5, 1.0, 1.0, 0.2, 1.0, 1.0])
    idx, w, margin = oracle.topk(lg, 3)
    assert idx.tolist() == [1, 2, 4]
    assert margin == 0.0
    assert np.allclose(w, 1 / 3)


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    for z in (-30.0, -2.5, -0.1, 0.3, 1.0, 7.0, 40.0):
        assert np.isclose(oracle.silu(z), z * expit(z), rtol=1e-14, atol=1e-300)
        assert np.isclose(oracle.silu(z) - oracle.silu(-z), z, rtol=1e-13, atol=1e-13)
    assert np.isclose(oracle.silu(50.0), 50.0, rtol=1e-15)


def test_attend_special_cases_and_library():
    rng = np.random.default_rng(6)
    hd = 16
    q = rng.standard_normal(hd)
    V = bf16(rng.standard_normal((1, hd)))
    K = bf16(rng.standard_normal((1, hd)))
    # one cached position: output is that position's value exactly
    assert np.array_equal(oracle.attend(q, K, V, 0.25), synth.bf16_to_f32(V[0]).astype(np.float64))
    # identical keys: uniform weights, output = mean of the values
    K4 = np.repeat(K, 5, axis=0)
    V4 = bf16(rng.standard_normal((5, hd)))
    assert np.allclose(oracle.attend(q, K4, V4, 0.25), synth.bf16_to_f32(V4).astype(np.float64).mean(0), rtol=1e-13)
    # general case against scipy softmax and a numpy matrix product
    Kn, Vn = bf16(rng.standard_normal((37, hd))), bf16(rng.standard_normal((37, hd)))
    Kf, Vf = synth.bf16_to_f32(Kn).astype(np.float64), synth.bf16_to_f32(Vn).astype(np.float64)
    ref = sp_softmax(Kf @ q * 0.25) @ Vf
    assert np.allclose(oracle.attend(q, Kn, Vn, 0.25), ref, rtol=1e-12, atol=1e-14)


def test_router_folded_into_output_rows_equals_norm_then_matmul():
    # the GPU path for two or more tokens: each CTA adds its rows' share of
    # sum_i Wr[e,i] g_i x_i and of sum_i x_i^2 into one of 8 copies; the reader
    # sums the copies and scales by 1/rms. Same logits as RMSNorm then Wr.
    rng = np.random.default_rng(7)
    d, E, eps = 2048, 64, 1e-6
    x = rng.standard_normal(d) * 3
    g = bf16(1 + 0.02 * rng.standard_normal(d))
    Wr = synth.bf16_to_f32(bf16(0.02 * rng.standard_normal((E, d)))).astype(np.float64)
    plain = Wr @ oracle.rmsnorm(x, g, eps)
    gf = synth.bf16_to_f32(g).astype(np.float64)
    acc = np.zeros((8, E + 1))
    rows = np.array_split(np.arange(d), 152)  # one row range per CTA
    for cta, r in enumerate(rows):
        acc[cta % 8, :E] += Wr[:, r] @ (gf[r] * x[r])
        acc[cta % 8, E] += x[r] @ x[r]
    tot = acc.sum(0)
    folded = tot[:E] / np.sqrt(tot[E] / d + eps)
    assert np.allclose(folded, plain, rtol=1e-12, atol=1e-12)
    # top-k unchanged by the common positive scale
    assert np.array_equal(oracle.topk(folded, 8)[0], oracle.topk(tot[:E], 8)[0])


def test_e4m3_value_against_torch_and_closed_forms():
    # every code against torch's float8_e4m3fn decoding (a library routine
    # the oracle does not use), plus values fixed by the format's definition
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], ref[~nan])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0xC0) == -2.0


def test_mx_dequant_blocks_and_scales():
    # element (r, j) = value(code) * 2^(E[r, j // 32] - 127): built here from
    # torch's decoding and numpy's ldexp with the scales repeated per block;
    # a wrong block index, bias or row stride breaks the comparison
    import torch
    rng = np.random.default_rng(8)
    rows, cols = 5, 96
    q = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    sc = rng.integers(100, 140, (rows, cols // 32), dtype=np.uint8)
    dec = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = np.ldexp(dec, np.repeat(sc.astype(np.int64) - 127, 32, axis=1))
    assert np.array_equal(oracle.mx_dequant(q, sc, rows, cols), ref)
    # scale byte 127 is the identity
    one = np.full((rows, cols // 32), 127, dtype=np.uint8)
    assert np.array_equal(oracle.mx_dequant(q, one, rows, cols), dec)


def _tiny_mx():
    from synth import configs
    return configs.scaled(configs.TINY, n_layers=1, expert_format=oracle.MXFP8)


def test_mxfp8_model_expert_weights_are_the_dequantised_codes():
    # the MXFP8 model's expert tensors equal the generator's codes decoded by
    # torch and scaled by 2^(E - 127), exactly (as bf16 bits); every other
    # tensor is the bf16 model's
    import torch
    from synth import configs
    cfg = _tiny_mx()
    mx, bf = oracle.Model(cfg), oracle.Model(configs.scaled(cfg, expert_format=oracle.BF16))
    for kind, layer, e in [(synth.GATE, 0, 0), (synth.UP, 0, 5), (synth.DOWN, 0, 7), (synth.SH_DOWN, 0, 0)]:
        r, c, _, _ = synth.weight_spec(cfg, kind)
        q = synth.fill_e4m3_host(r * c, cfg["seed"], synth.tensor_id(kind, layer, e))
        sc = synth.fill_e8m0_host(r * c // 32, cfg["seed"], synth.tensor_id(synth.SCALE_OF[kind], layer, e))
        dec = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        want = np.ldexp(dec, np.repeat(sc.astype(np.int64) - 127, 32))
        got = synth.bf16_to_f32(mx.get_tensor(kind, layer, e)).astype(np.float64)
        assert np.array_equal(got, want)
    for kind in (synth.WQ, synth.WO, synth.ROUTER, synth.FFN_NORM):
        assert np.array_equal(mx.get_tensor(kind, 0, 0), bf.get_tensor(kind, 0, 0))


def test_mxfp8_model_is_the_bf16_model_with_those_weights():
    # a decode step of the MXFP8 model equals, bit for bit, the bf16 model's
    # step once its expert tensors are set to the MXFP8 model's values: the
    # format changes the weights and nothing else
    from synth import configs
    cfg = _tiny_mx()
    mx, bf = oracle.Model(cfg), oracle.Model(configs.scaled(cfg, expert_format=oracle.BF16))
    for kind in (synth.SH_GATE, synth.SH_UP, synth.SH_DOWN):
        bf.set_tensor(kind, 0, 0, mx.get_tensor(kind, 0, 0))
    for e in range(cfg["n_routed_experts"]):
        for kind in (synth.GATE, synth.UP, synth.DOWN):
            bf.set_tensor(kind, 0, e, mx.get_tensor(kind, 0, e))
    outs = []
    for m in (mx, bf):
        kv = oracle.KV(m, 1, 40)
        kv.prefill(cfg["seed"], 32)
        outs.append(oracle.decode(m, kv, np.array([[7]], dtype=np.int32), [32])["logits"])
    assert np.array_equal(outs[0], outs[1])
