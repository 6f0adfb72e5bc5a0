"""Model-level pins of the oracle decode step (CPU only).

Each test checks the composed step against something independent:
 - brute force: incremental decode with a KV cache equals a from-scratch
   recompute with an explicit causal attention matrix (no cache object);
 - algebra: absorbed MLA equals the plain decompress-K/V form in fp64;
 - structure: a T-token verify block equals T single-token steps; a batch row
   equals a batch-1 run; E=1/k=1 MoE equals the dense MLP;
 - reductions to numpy: with layer outputs zeroed the step is
   LM_head(RMSNorm(embedding)); a first token attends only to itself, so the
   attention output is its own V; a uniform router with k=E averages experts;
 - precision: fp32 accumulation stays far inside the parity tolerance of fp64;
 - acceptance: drafts planted equal to the greedy tokens are all accepted.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
import synth
from synth import configs

MLA_SMALL = configs.scaled(
    configs.DEEP, name="mla_small", n_layers=2, d_model=64, vocab=50, n_q_heads=2,
    q_lora_rank=32, kv_lora_rank=16, qk_nope_dim=8, qk_rope_dim=4, v_head_dim=8,
    n_routed_experts=4, top_k=2, ffn_dim=16, shared_ffn_dim=16, seed=11, ctx=8)
GQA_SMALL = configs.scaled(configs.TINY, name="gqa_small", d_model=64, vocab=60, n_q_heads=4, n_kv_heads=2,
                           head_dim=16, n_routed_experts=4, top_k=2, ffn_dim=32, shared_ffn_dim=32, ctx=8)


def f32(u):
    return synth.bf16_to_f32(np.asarray(u, dtype=np.uint16)).astype(np.float64)


def bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def np_rms(x, g, eps):
    return x / np.sqrt((x * x).mean() + eps) * g


def run_steps(cfg, B, T, steps, ctx, precision=64, absorbed=True, tok_fn=None):
    m = oracle.Model(cfg)
    kv = oracle.KV(m, B, ctx + steps * T + 1)
    kv.prefill(cfg["seed"], ctx)
    outs = []
    for s in range(steps):
        tok = tok_fn(s) if tok_fn else synth.tokens(cfg["seed"], s, B, T, cfg["vocab"])
        outs.append(oracle.decode(m, kv, tok, [ctx + s * T] * B, precision=precision, mla_absorbed=absorbed))
    return outs


@pytest.mark.parametrize("cfg", [GQA_SMALL, MLA_SMALL], ids=["gqa", "mla"])
def test_incremental_equals_full_recompute(cfg):
    P = 7
    tok = np.array([[synth.token(cfg["seed"], 0, 0, t, cfg["vocab"]) for t in range(P)]], dtype=np.int32)
    m = oracle.Model(cfg)
    full = oracle.full_recompute(m, tok, precision=64)
    for absorbed in (False, True):
        kv = oracle.KV(m, 1, P)
        inc = np.stack([oracle.decode(m, kv, tok[:, p:p + 1], [p], mla_absorbed=absorbed)["logits"][0, 0]
                        for p in range(P)])
        assert np.abs(inc - full[0]).max() < 1e-12
    full32 = oracle.full_recompute(m, tok, precision=32)
    kv = oracle.KV(m, 1, P)
    inc32 = np.stack([oracle.decode(m, kv, tok[:, p:p + 1], [p], precision=32)["logits"][0, 0] for p in range(P)])
    assert np.abs(inc32 - full32[0]).max() < 1e-5


def test_mla_absorbed_equals_unabsorbed_fp64():
    a = run_steps(MLA_SMALL, 2, 1, 3, MLA_SMALL["ctx"], absorbed=True)
    b = run_steps(MLA_SMALL, 2, 1, 3, MLA_SMALL["ctx"], absorbed=False)
    for x, y in zip(a, b):
        assert np.abs(x["logits"] - y["logits"]).max() < 1e-10
        assert np.array_equal(x["route_idx"], y["route_idx"])


@pytest.mark.parametrize("cfg", [GQA_SMALL, MLA_SMALL], ids=["gqa", "mla"])
def test_verify_block_equals_sequential_steps(cfg):
    T, ctx = 5, cfg["ctx"]
    tok = synth.tokens(cfg["seed"], 0, 2, T, cfg["vocab"])
    m = oracle.Model(cfg)
    kv = oracle.KV(m, 2, ctx + T)
    kv.prefill(cfg["seed"], ctx)
    blk = oracle.decode(m, kv, tok, [ctx, ctx])
    kv2 = oracle.KV(m, 2, ctx + T)
    kv2.prefill(cfg["seed"], ctx)
    for t in range(T):
        one = oracle.decode(m, kv2, tok[:, t:t + 1], [ctx + t, ctx + t])
        assert np.abs(one["logits"][:, 0] - blk["logits"][:, t]).max() < 1e-12
        ridx = blk["route_idx"].reshape(cfg["n_layers"], 2, T, -1)[:, :, t]
        assert np.array_equal(one["route_idx"].reshape(cfg["n_layers"], 2, -1), ridx)
    # caches identical after both paths
    for l in range(cfg["n_layers"]):
        for b in range(2):
            assert np.array_equal(kv.read(l, b, 0, ctx + T), kv2.read(l, b, 0, ctx + T))


def test_batch_rows_equal_single_runs():
    cfg = GQA_SMALL
    ctx = cfg["ctx"]
    tok = synth.tokens(cfg["seed"], 0, 3, 1, cfg["vocab"])
    pos = [ctx, ctx + 2, ctx + 5]
    m = oracle.Model(cfg)
    kv = oracle.KV(m, 3, ctx + 8)
    kv.prefill(cfg["seed"], ctx + 6)
    both = oracle.decode(m, kv, tok, pos)
    for b in range(3):
        kv1 = oracle.KV(m, 1, ctx + 8)
        # sequence b's prefill stream is tensor (layer, seq=b): copy it into a batch-1 cache
        for l in range(cfg["n_layers"]):
            kv1.write(l, 0, 0, kv.read(l, b, 0, pos[b]))
        one = oracle.decode(m, kv1, tok[b:b + 1], [pos[b]])
        assert np.abs(one["logits"][0] - both["logits"][b]).max() < 1e-12


def test_single_expert_moe_equals_dense_mlp():
    moe = configs.scaled(GQA_SMALL, n_routed_experts=1, top_k=1, n_shared_experts=0)
    dense = configs.scaled(GQA_SMALL, n_routed_experts=0, top_k=0, n_shared_experts=1, shared_ffn_dim=32)
    mm, md = oracle.Model(moe), oracle.Model(dense)
    for l in range(moe["n_layers"]):
        for src, dst in ((synth.GATE, synth.SH_GATE), (synth.UP, synth.SH_UP), (synth.DOWN, synth.SH_DOWN)):
            md.set_tensor(dst, l, 0, mm.get_tensor(src, l, 0))
    tok = synth.tokens(1, 0, 1, 1, moe["vocab"])
    outs = []
    for m in (mm, md):
        kv = oracle.KV(m, 1, 16)
        kv.prefill(5, 8)
        outs.append(oracle.decode(m, kv, tok, [8]))
    assert np.abs(outs[0]["logits"] - outs[1]["logits"]).max() < 1e-13
    assert np.all(outs[0]["route_w"] == 1.0)


def _zero(m, kind, layer, expert=0):
    n = m.get_tensor(kind, layer, expert).size
    m.set_tensor(kind, layer, expert, np.zeros(n, dtype=np.uint16))


def test_zeroed_layers_reduce_to_embedding_head():
    cfg = GQA_SMALL
    m = oracle.Model(cfg)
    for l in range(cfg["n_layers"]):
        _zero(m, synth.WO, l)
        _zero(m, synth.SH_DOWN, l)
        for e in range(cfg["n_routed_experts"]):
            _zero(m, synth.DOWN, l, e)
    tok = np.array([[17]], dtype=np.int32)
    kv = oracle.KV(m, 1, 16)
    out = oracle.decode(m, kv, tok, [3])["logits"][0, 0]
    d = cfg["d_model"]
    E = f32(m.get_tensor(synth.EMBED)).reshape(-1, d)
    W = f32(m.get_tensor(synth.LM_HEAD)).reshape(-1, d)
    g = f32(m.get_tensor(synth.FINAL_NORM))
    ref = W @ np_rms(E[17], g, cfg["rms_eps"])
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_first_token_attends_to_itself_gqa():
    # position 0 with an empty cache: softmax over one key, output = own V
    # (rounded to bf16 like the cache). With the FFN zeroed the whole step is
    # a few numpy matrix products; RoPE at position 0 is the identity.
    cfg = configs.scaled(GQA_SMALL, n_layers=1)
    m = oracle.Model(cfg)
    _zero(m, synth.SH_DOWN, 0)
    for e in range(cfg["n_routed_experts"]):
        _zero(m, synth.DOWN, 0, e)
    d, Hq, Hkv, hd = cfg["d_model"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    tok = np.array([[5]], dtype=np.int32)
    kv = oracle.KV(m, 1, 4)
    out = oracle.decode(m, kv, tok, [0])["logits"][0, 0]
    x = f32(m.get_tensor(synth.EMBED)).reshape(-1, d)[5]
    xn = np_rms(x, f32(m.get_tensor(synth.ATTN_NORM, 0)), cfg["rms_eps"])
    k = f32(m.get_tensor(synth.WK, 0)).reshape(-1, d) @ xn
    v = f32(m.get_tensor(synth.WV, 0)).reshape(-1, d) @ xn
    row = kv.read(0, 0, 0, 1)[0]
    assert np.array_equal(row[:Hkv * hd], bf16(k)) and np.array_equal(row[Hkv * hd:], bf16(v))
    vb = f32(bf16(v)).reshape(Hkv, hd)
    o = np.concatenate([vb[h // (Hq // Hkv)] for h in range(Hq)])  # contiguous head groups
    x1 = x + f32(m.get_tensor(synth.WO, 0)).reshape(d, -1) @ o
    ref = f32(m.get_tensor(synth.LM_HEAD)).reshape(-1, d) @ np_rms(x1, f32(m.get_tensor(synth.FINAL_NORM)),
                                                                   cfg["rms_eps"])
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_uniform_router_with_all_experts_averages_swiglu():
    cfg = configs.scaled(GQA_SMALL, n_layers=1, top_k=4, n_shared_experts=0)
    m = oracle.Model(cfg)
    _zero(m, synth.WO, 0)
    _zero(m, synth.ROUTER, 0)
    d, f = cfg["d_model"], cfg["ffn_dim"]
    tok = np.array([[9]], dtype=np.int32)
    kv = oracle.KV(m, 1, 4)
    res = oracle.decode(m, kv, tok, [1])
    x = f32(m.get_tensor(synth.EMBED)).reshape(-1, d)[9]
    xn = np_rms(x, f32(m.get_tensor(synth.FFN_NORM, 0)), cfg["rms_eps"])
    y = np.zeros(d)
    for e in range(4):
        g = f32(m.get_tensor(synth.GATE, 0, e)).reshape(f, d) @ xn
        u = f32(m.get_tensor(synth.UP, 0, e)).reshape(f, d) @ xn
        y += 0.25 * (f32(m.get_tensor(synth.DOWN, 0, e)).reshape(d, f) @ (g * expit(g) * u))
    x1 = x + y
    ref = f32(m.get_tensor(synth.LM_HEAD)).reshape(-1, d) @ np_rms(x1, f32(m.get_tensor(synth.FINAL_NORM)),
                                                                   cfg["rms_eps"])
    assert np.allclose(res["logits"][0, 0], ref, rtol=1e-10, atol=1e-12)
    assert res["route_idx"][0, 0].tolist() == [0, 1, 2, 3] and np.allclose(res["route_w"], 0.25)


def test_tiny_fp32_close_to_fp64_and_router_invariants():
    cfg = configs.TINY
    o64 = run_steps(cfg, 1, 1, cfg["steps"], cfg["ctx"], precision=64)
    o32 = run_steps(cfg, 1, 1, cfg["steps"], cfg["ctx"], precision=32)
    worst = 0.0
    for a, b in zip(o64, o32):
        flips = (a["route_idx"] != b["route_idx"]).any()
        if not flips:
            worst = max(worst, np.abs(a["logits"] - b["logits"]).max())
        ri, rw, rm = a["route_idx"], a["route_w"], a["route_margin"]
        assert np.all(np.sort(ri, -1)[..., 1:] != np.sort(ri, -1)[..., :-1])
        assert np.allclose(rw.sum(-1), 1.0) and np.all(rw > 0) and np.all(rm >= 0)
        assert np.all(np.diff(rw, axis=-1) <= 1e-15)  # weights sorted descending
    assert worst < 2e-4  # far inside the 2e-2 parity bound


@pytest.mark.parametrize("cfg", [GQA_SMALL, MLA_SMALL], ids=["gqa", "mla"])
def test_acceptance_of_planted_greedy_drafts(cfg):
    T, ctx = 5, cfg["ctx"]
    m = oracle.Model(cfg)
    # build drafts greedily with single-token steps: token t+1 = argmax at t
    kv = oracle.KV(m, 1, ctx + T)
    kv.prefill(cfg["seed"], ctx)
    seq = [int(synth.token(cfg["seed"], 0, 0, 0, cfg["vocab"]))]
    for t in range(T - 1):
        lg = oracle.decode(m, kv, np.array([[seq[-1]]]), [ctx + t])["logits"][0, 0]
        seq.append(int(np.argmax(lg)))
    for bad_at, expect in ((None, T), (3, 3), (1, 1)):
        s = list(seq)
        if bad_at is not None:
            s[bad_at] = (s[bad_at] + 1) % cfg["vocab"]
        kv2 = oracle.KV(m, 1, ctx + T)
        kv2.prefill(cfg["seed"], ctx)
        out = oracle.decode(m, kv2, np.array([s], dtype=np.int32), [ctx])
        assert out["accept"][0] == expect


def np_rope(x, pos, theta=1e4):
    half = x.size // 2
    z = (x[:half] + 1j * x[half:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(half) / x.size))
    return np.concatenate([z.real, z.imag])


def _ffn_off(m, cfg, l=0):
    if cfg["n_shared_experts"]:
        _zero(m, synth.SH_DOWN, l)
    for e in range(cfg["n_routed_experts"]):
        _zero(m, synth.DOWN, l, e)


def test_two_position_gqa_against_numpy():
    """One layer, one cached position written by hand, query at position 1:
    scores scaled by 1/sqrt(hd), RoPE at the query position, contiguous GQA
    groups, softmax over both positions -- all rebuilt with numpy/scipy."""
    from scipy.special import softmax as sp_softmax
    cfg = configs.scaled(GQA_SMALL, n_layers=1)
    m = oracle.Model(cfg)
    _ffn_off(m, cfg)
    d, Hq, Hkv, hd = cfg["d_model"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    rng = np.random.default_rng(8)
    row0 = bf16(rng.standard_normal(2 * Hkv * hd))
    kv = oracle.KV(m, 1, 4)
    kv.write(0, 0, 0, row0[None])
    out = oracle.decode(m, kv, np.array([[7]], dtype=np.int32), [1])["logits"][0, 0]
    x = f32(m.get_tensor(synth.EMBED)).reshape(-1, d)[7]
    xn = np_rms(x, f32(m.get_tensor(synth.ATTN_NORM, 0)), cfg["rms_eps"])
    q = (f32(m.get_tensor(synth.WQ, 0)).reshape(-1, d) @ xn).reshape(Hq, hd)
    k1 = (f32(m.get_tensor(synth.WK, 0)).reshape(-1, d) @ xn).reshape(Hkv, hd)
    v1 = (f32(m.get_tensor(synth.WV, 0)).reshape(-1, d) @ xn).reshape(Hkv, hd)
    K = np.stack([f32(row0[:Hkv * hd]).reshape(Hkv, hd), f32(bf16(np.stack([np_rope(k, 1) for k in k1])))])
    V = np.stack([f32(row0[Hkv * hd:]).reshape(Hkv, hd), f32(bf16(v1))])
    o = []
    for h in range(Hq):
        g = h // (Hq // Hkv)
        a = sp_softmax(K[:, g] @ np_rope(q[h], 1) / np.sqrt(hd))
        o.append(a @ V[:, g])
    x1 = x + f32(m.get_tensor(synth.WO, 0)).reshape(d, -1) @ np.concatenate(o)
    ref = f32(m.get_tensor(synth.LM_HEAD)).reshape(-1, d) @ np_rms(x1, f32(m.get_tensor(synth.FINAL_NORM)),
                                                                   cfg["rms_eps"])
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-11)


def test_two_position_mla_against_numpy():
    """MLA with one hand-written cached latent and the query at position 1,
    rebuilt with numpy: q path (W_dq, q-norm, W_uq, RoPE on the rope part),
    latent path (W_dkv, kv-norm, RoPE on k_rope, bf16 append), K_nope / V
    decompressed with W_ukv, scores scaled by 1/sqrt(nope + rope)."""
    from scipy.special import softmax as sp_softmax
    cfg = configs.scaled(MLA_SMALL, n_layers=1)
    m = oracle.Model(cfg)
    _ffn_off(m, cfg)
    d, H, ql, kl = cfg["d_model"], cfg["n_q_heads"], cfg["q_lora_rank"], cfg["kv_lora_rank"]
    nope, rd, vd = cfg["qk_nope_dim"], cfg["qk_rope_dim"], cfg["v_head_dim"]
    rng = np.random.default_rng(9)
    lat0 = bf16(rng.standard_normal(kl + rd))
    kv = oracle.KV(m, 1, 4)
    kv.write(0, 0, 0, lat0[None])
    for absorbed in (False, True):
        kvx = oracle.KV(m, 1, 4)
        kvx.write(0, 0, 0, lat0[None])
        out = oracle.decode(m, kvx, np.array([[3]], dtype=np.int32), [1], mla_absorbed=absorbed)["logits"][0, 0]
        x = f32(m.get_tensor(synth.EMBED)).reshape(-1, d)[3]
        xn = np_rms(x, f32(m.get_tensor(synth.ATTN_NORM, 0)), cfg["rms_eps"])
        cq = np_rms(f32(m.get_tensor(synth.WDQ, 0)).reshape(ql, d) @ xn, f32(m.get_tensor(synth.Q_NORM, 0)),
                    cfg["rms_eps"])
        q = (f32(m.get_tensor(synth.WUQ, 0)).reshape(-1, ql) @ cq).reshape(H, nope + rd)
        kva = f32(m.get_tensor(synth.WDKV, 0)).reshape(kl + rd, d) @ xn
        c1 = np_rms(kva[:kl], f32(m.get_tensor(synth.KV_NORM, 0)), cfg["rms_eps"])
        lat1 = f32(bf16(np.concatenate([c1, np_rope(kva[kl:], 1)])))
        lats = np.stack([f32(lat0), lat1])
        W = f32(m.get_tensor(synth.WUKV, 0)).reshape(H, nope + vd, kl)
        o = []
        for h in range(H):
            kn = lats[:, :kl] @ W[h, :nope].T
            vv = lats[:, :kl] @ W[h, nope:].T
            s = (kn @ q[h, :nope] + lats[:, kl:] @ np_rope(q[h, nope:], 1)) / np.sqrt(nope + rd)
            o.append(sp_softmax(s) @ vv)
        x1 = x + f32(m.get_tensor(synth.WO, 0)).reshape(d, -1) @ np.concatenate(o)
        ref = f32(m.get_tensor(synth.LM_HEAD)).reshape(-1, d) @ np_rms(x1, f32(m.get_tensor(synth.FINAL_NORM)),
                                                                       cfg["rms_eps"])
        assert np.allclose(out, ref, rtol=1e-9, atol=1e-11)
        assert np.array_equal(kvx.read(0, 0, 1, 1)[0], bf16(lat1))
