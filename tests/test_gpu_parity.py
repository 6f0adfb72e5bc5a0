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
    print(cfg["name"], cfg["n_layers"], "layers", B, T, rep)
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


@pytest.mark.parametrize("name,T", [("mid", 1), ("deep", 3)])
def test_paged_cache_with_permuted_block_table(name, T):
    # pages in a random order: GQA chunks are copied from their page's
    # address, MLA chunks by tensor-map coordinates (page index, half page)
    cfg = configs.scaled(configs.ALL[name], n_layers=2)
    rng = np.random.default_rng(3)

    def table(pps, B=2):
        return rng.permutation(B * pps).astype(np.int32).reshape(B, pps)

    _run(cfg, 2, T, 2, 700, block_table=table, want_accept=T > 1)


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


@pytest.mark.parametrize("B", [4, 8])
def test_deep_batched(B):
    # the deep model's batched path (MLA with B query rows per head, the
    # router folded into the output projection, shared expert in token groups
    # of 4, routed units over their own tokens) at the full 8192-position context
    cfg = configs.scaled(configs.DEEP, n_layers=2)
    _run(cfg, B, 1, 1, cfg["ctx"])


def test_deep_full_depth_batch1():
    # one decode step of all 92 layers (the configuration the throughput is
    # quoted on) against the fp64 oracle, whose layer weights are generated on
    # first use and released after the layer
    cfg = configs.DEEP
    _, _, rep = _run(cfg, 1, 1, 1, cfg["ctx"], lazy=True)
    print(f"deep 92 layers, batch 1, ctx 8192: logits max-abs {rep['max_abs']:.3e} "
          f"mean-abs {rep['mean_abs']:.3e}, router margin max |gpu - oracle| {rep['margin_maxdiff']:.3e}")


def test_verify_step_with_planted_drafts():
    # drafts are the oracle's own greedy continuation with one error planted
    # at a known draft index per sequence (or none), so the acceptance lengths
    # 1..7 are all exercised and compared with the oracle's
    import oracle
    cfg = configs.scaled(configs.VERIFY, n_layers=2)
    B, T, ctx = 8, 7, 2000
    V = cfg["vocab"]
    first = parity_tokens(cfg, B)
    # greedy continuation of every sequence, one oracle step per token
    om = oracle.Model(cfg)
    okv = oracle.KV(om, B, ctx + T + 1)
    for l in range(cfg["n_layers"]):
        for b in range(B):
            okv.write(l, b, 0, parity._prefill_rows(cfg, l, b, ctx))
    tok = first.copy()
    greedy = np.zeros((B, T - 1), dtype=np.int32)
    for i in range(T - 1):
        lg = oracle.decode(om, okv, tok[:, None], np.full(B, ctx + i, dtype=np.int32))["logits"][:, 0]
        tok = lg.argmax(1).astype(np.int32)
        greedy[:, i] = tok
    okv.close()
    om.close()
    err_at = [0, 1, 2, 3, 4, 5, 6, 0]  # draft index (1..6) made wrong, 0: none
    block = np.concatenate([first[:, None], greedy], axis=1)
    for b, j in enumerate(err_at):
        if j:
            block[b, j] = (block[b, j] + 1) % V
    expect = np.array([j if j else T for j in err_at], dtype=np.int32)
    g, o, rep = _run(cfg, B, T, 1, ctx, want_accept=True, tokens_fn=lambda s: block)
    acc_g, acc_o = g[0]["accept"], o[0]["accept"]
    print("planted accept", expect.tolist(), "gpu", acc_g.tolist(), "oracle", acc_o.tolist())
    assert np.array_equal(acc_o, expect)
    # the GPU's acceptance equals the planted one for every sequence whose
    # argmax decisions are clear: at each row the acceptance reads, the
    # oracle's top-2 logit gap exceeds twice the GPU's largest logit error of
    # that row (parity.compare applies the fixed 4e-2 gap rule on top)
    lg_g, lg_o = g[0]["logits"], o[0]["logits"]
    clear = 0
    for b in range(B):
        rows = range(min(int(expect[b]), T - 1))
        ok = True
        for i in rows:
            srt = np.sort(lg_o[b, i])[::-1]
            if srt[0] - srt[1] <= 2 * np.abs(lg_g[b, i] - lg_o[b, i]).max():
                ok = False
        if ok:
            clear += 1
            assert acc_g[b] == expect[b], (b, acc_g[b], expect[b])
    assert clear >= B - 2, f"only {clear} of {B} sequences had clear argmax decisions"


def parity_tokens(cfg, B):
    from moe_decode_megakernel_02_gb300 import workload
    return workload.tokens(cfg, 0, B, 1)[:, 0].astype(np.int32)


def test_ring_slots_of_the_loaded_build():
    # the suite also runs against the 2-slot ring build (MK_LIB, see below):
    # the library this process loaded reports its own ring depth
    import os
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    model = workload.load_synthetic(configs.TINY, max_batch=1, max_tokens_per_seq=1, max_ctx=80)
    want = 2 if os.environ.get("MK_LIB", "").endswith("libmk_nslot2.so") else 3
    assert model.info().ring_slots == want


def test_two_slot_ring_build_parity():
    # a shrunken ring (2 slots instead of 3) changes every producer/consumer
    # interleaving; the same parity cases must pass with that build
    import os
    import subprocess
    import sys
    import moe_decode_megakernel_02_gb300 as mk
    if os.environ.get("MK_LIB"):
        pytest.skip("already running against another build")
    assert os.path.exists(mk.LIB_NSLOT2), "libmk_nslot2.so is not built"
    env = dict(os.environ, MK_LIB=mk.LIB_NSLOT2)
    sel = ("ring_slots_of_the_loaded_build or tiny_sixteen or mid_batched or deep_reduced_layers or "
           "verify_step_reduced or deep_batched")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-k", sel, __file__],
                       env=env, cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       capture_output=True, text=True, timeout=1200)
    print(r.stdout[-2000:])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name,B,T,steps", [("tiny", 1, 1, 3), ("mid", 4, 1, 1), ("deep", 2, 1, 2),
                                            ("verify", 8, 7, 1), ("dense", 1, 1, 1)])
def test_unfused_one_launch_per_stage(name, B, T, steps):
    # the comparison path: the same stages, each its own launch (a CUDA graph
    # replayed per step), ordered by the stream instead of counters
    cfg = configs.ALL[name]
    if name != "tiny":
        cfg = configs.scaled(cfg, n_layers=2)
    ctx = min(cfg["ctx"], 2000)
    _run(cfg, B, T, steps, ctx, entry="decode_step_unfused", want_accept=T > 1)


@pytest.mark.parametrize("B", [1, 3])
def test_deep_separate_absorbed_query_and_value_stages(monkeypatch, B):
    # the schedule in which the absorbed query (QLAT) and the value
    # up-projection (UV) are stages of their own (used when the tokens' inputs
    # do not fit the staging area at once); by default, for few tokens, the
    # QB CTAs and the combine CTAs compute them
    monkeypatch.setenv("MK_QLAT_STAGE", "1")
    monkeypatch.setenv("MK_UV_STAGE", "1")
    cfg = configs.scaled(configs.DEEP, n_layers=2)
    _run(cfg, B, 1, 2, cfg["ctx"])


# MXFP8 expert weights: the oracle dequantises the
# generator's E4M3 codes and E8M0 scales exactly, the kernel streams the codes
# and scales and takes the same values; the tolerance is the bf16 model's
# (the arithmetic is the same once the weights are read).
# d_model 2048 (deep, mid): 16-row gate/up tiles, 4 chunks of 16 codes per
# lane; 1024 and 512: 32- and 64-row tiles, 2 and 1 chunks (at 512 one down
# tile per unit)
_MX = dict(expert_format=1)
_MX_SMALL = dict(_MX, n_layers=2, vocab=4096, n_q_heads=4, n_kv_heads=2, head_dim=128, n_routed_experts=16,
                 top_k=4, ctx=300)


@pytest.mark.parametrize("name,over", [
    ("deep", dict(_MX, n_layers=3)),
    ("mid", dict(_MX, n_layers=2)),
    ("mid", dict(_MX_SMALL, d_model=1024, ffn_dim=512, shared_ffn_dim=256)),
    ("mid", dict(_MX_SMALL, d_model=512, ffn_dim=256, shared_ffn_dim=128)),
])
def test_mxfp8_experts_batch1(name, over):
    cfg = configs.scaled(configs.ALL[name], **over)
    _run(cfg, 1, 1, 2, cfg["ctx"])


@pytest.mark.parametrize("name,B,T,over", [
    ("deep", 2, 1, dict(_MX, n_layers=2)),
    ("deep", 8, 1, dict(_MX, n_layers=2)),
    ("mid", 4, 1, dict(_MX, n_layers=2)),
    ("mid", 3, 1, dict(_MX_SMALL, d_model=1024, ffn_dim=512, shared_ffn_dim=256)),
    ("verify", 8, 7, dict(_MX, n_layers=2)),
])
def test_mxfp8_experts_several_tokens(name, B, T, over):
    # every token of an expert unit takes the unit's tiles in turn (routed
    # experts: the tokens routed to them, in groups the staging area holds;
    # the shared expert: token groups); verify B 8 x T 7: 56 tokens, gathered
    cfg = configs.scaled(configs.ALL[name], **over)
    ctx = min(cfg["ctx"], 2000)
    _run(cfg, B, T, 1, ctx, want_accept=T > 1)


def test_mxfp8_experts_full_depth_batch1():
    cfg = configs.scaled(configs.DEEP, **_MX)
    _, _, rep = _run(cfg, 1, 1, 1, cfg["ctx"], lazy=True)
    print(f"deep 92 layers, MXFP8 experts, batch 1, ctx 8192: logits max-abs {rep['max_abs']:.3e} "
          f"mean-abs {rep['mean_abs']:.3e}")


@pytest.mark.parametrize("name,B", [("deep", 8), ("mid", 4), ("tiny", 1)])
def test_repeated_steps_reproduce_routing_and_logits(name, B):
    # the same step five times (same tokens, same positions: the KV entries
    # are rewritten with the same values): the experts chosen are the same
    # every time wherever the router margin exceeds 1e-3, and the logits
    # differ only by the order of the floating-point additions the CTAs make
    # with atomics (residual rows, split-K partial sums)
    from moe_decode_megakernel_02_gb300 import workload
    cfg = configs.scaled(configs.ALL[name], n_layers=2)
    ctx = min(cfg["ctx"], 2000)
    tok = workload.tokens(cfg, 0, B, 1)
    g, _ = parity.run_gpu(cfg, B, 1, 5, ctx, positions_fn=lambda s: np.full(B, ctx, dtype=np.int32),
                          tokens_fn=lambda s: tok)
    r0 = g[0]
    for r in g[1:]:
        assert np.abs(r["logits"] - r0["logits"]).max() <= 1e-4
        clear = r0["route_margin"] > 1e-3
        same = (np.sort(r["route_idx"], axis=-1) == np.sort(r0["route_idx"], axis=-1)).all(axis=-1)
        assert same[clear].all()


@pytest.mark.parametrize("name", ["deep", "mid"])
def test_mxfp8_experts_unfused(name):
    # MXFP8 experts through the one-launch-per-stage path
    cfg = configs.scaled(configs.ALL[name], n_layers=2, **_MX)
    _run(cfg, 1, 1, 2, min(cfg["ctx"], 2000), entry="decode_step_unfused")
