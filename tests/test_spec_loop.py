"""Greedy speculative decoding loop (moe_decode_megakernel_02_gb300.spec).

CPU: the loop's bookkeeping against a stand-in model whose greedy token is a
known function of (token, position) and whose acceptance follows the verify
step's rule; the emitted tokens must equal plain greedy decoding whatever the
drafts, and positions advance by the accept lengths.
GPU: the loop over the CUDA verify step must reproduce the oracle's plain
one-token greedy decoding of the same model and cache, with the accept lengths
the planted draft errors imply.
"""
import numpy as np
import pytest
import torch

from moe_decode_megakernel_02_gb300.spec import GreedySpecLoop, PlantedDrafter, RandomDrafter


class FakeModel:
    """Greedy next token f(token, position); acceptance as the verify step defines it."""

    def __init__(self, V):
        self.V = V
        self.amax = None

    def f(self, tok, pos):
        return (int(tok) * 31 + int(pos) * 7 + 3) % self.V

    def decode_step(self, kv, tokens, positions, logits, accept, stream=None):
        t, p = tokens.numpy(), positions.numpy()
        B, T = t.shape
        am = np.array([[self.f(t[b, i], p[b] + i) for i in range(T)] for b in range(B)], dtype=np.int32)
        acc = np.zeros(B, dtype=np.int32)
        for b in range(B):
            a = 0
            while a < T - 1 and am[b, a] == t[b, a + 1]:
                a += 1
            acc[b] = a + 1
        self.amax = am.reshape(-1)
        accept.copy_(torch.from_numpy(acc))

    def check(self, stream=None):
        pass

    def last_argmax(self, out, stream=None):
        out.copy_(torch.from_numpy(self.amax))
        return out


def greedy_streams(model, first, pos0, n):
    out = []
    for b in range(len(first)):
        tok, pos, s = int(first[b]), int(pos0[b]), []
        for _ in range(n):
            tok = model.f(tok, pos)
            pos += 1
            s.append(tok)
        out.append(s)
    return out


def run_loop(model, drafter, first, pos0, T, steps):
    loop = GreedySpecLoop(model, None, first, pos0, T, model.V, drafter, device="cpu")
    for _ in range(steps):
        before = loop.pos.copy()
        acc = loop.step()
        assert np.all((acc >= 1) & (acc <= T))
        assert np.array_equal(loop.pos, before + acc)
    return loop


def test_exact_drafts_accept_whole_blocks():
    m = FakeModel(997)
    first, pos0 = np.array([5, 11]), np.array([64, 130])
    ref = greedy_streams(m, first, pos0, 100)
    loop = run_loop(m, PlantedDrafter(ref, m.V), first, pos0, 7, 5)
    assert all(np.all(a == 7) for a in loop.accepts)
    for b in range(2):
        assert loop.emitted[b] == ref[b][:35]


def test_planted_errors_set_the_accept_lengths():
    m = FakeModel(997)
    first, pos0 = np.array([5]), np.array([64])
    ref = greedy_streams(m, first, pos0, 100)
    wrong = {2, 9, 10, 17}
    loop = run_loop(m, PlantedDrafter(ref, m.V, wrong=lambda b, i: i in wrong), first, pos0, 7, 5)
    # step 1 drafts 0..5, 2 wrong -> 2 accepted + bonus (index 2); step 2 drafts 3..8 -> 6 + bonus 9;
    # step 3 drafts 10..15, 10 wrong -> bonus 10; step 4 drafts 11..16 -> 6 + bonus 17; step 5 drafts 18..23
    assert [int(a[0]) for a in loop.accepts] == [3, 7, 1, 7, 7]
    assert loop.emitted[0] == ref[0][:25]


def test_random_drafts_still_decode_greedily():
    m = FakeModel(50)  # small vocabulary: some random drafts are accepted
    first, pos0 = np.array([1, 2, 3]), np.array([0, 10, 20])
    ref = greedy_streams(m, first, pos0, 200)
    loop = run_loop(m, RandomDrafter(m.V, seed=3), first, pos0, 4, 30)
    for b in range(3):
        n = len(loop.emitted[b])
        assert n == int(sum(a[b] for a in loop.accepts))
        assert loop.emitted[b] == ref[b][:n]


def test_bad_arguments():
    m = FakeModel(10)
    with pytest.raises(ValueError):
        GreedySpecLoop(m, None, [1], [0], 1, 10, RandomDrafter(10), device="cpu")
    loop = GreedySpecLoop(m, None, [1], [0], 4, 10, lambda lp: np.zeros((1, 2), np.int32), device="cpu")
    with pytest.raises(ValueError):
        loop.step()


class OracleVerifyModel:
    """The oracle's verify step behind the loop's model interface (CPU)."""

    def __init__(self, om, okv):
        self.om, self.okv, self.amax = om, okv, None

    def decode_step(self, kv, tokens, positions, logits, accept, stream=None):
        import oracle
        r = oracle.decode(self.om, self.okv, tokens.numpy(), positions.numpy(), precision=64)
        self.amax = r["logits"].argmax(-1).reshape(-1).astype(np.int32)  # first maximum: lower id on ties
        accept.copy_(torch.from_numpy(r["accept"].astype(np.int32)))

    def check(self, stream=None):
        pass

    def last_argmax(self, out, stream=None):
        out.copy_(torch.from_numpy(self.amax))
        return out


def test_loop_over_the_oracle_verify_step_decodes_greedily():
    # the oracle's cache keeps the rows of rejected drafts until the next step
    # overwrites them: the loop must still reproduce one-token greedy decoding
    import oracle
    from synth import configs
    cfg = configs.TINY
    B, T, ctx, N = 2, 5, cfg["ctx"], 24
    om = oracle.Model(cfg)
    first = np.array([3, 700], dtype=np.int32)
    pos0 = np.array([ctx, ctx - 10], dtype=np.int32)

    kv = oracle.KV(om, B, ctx + 64)
    kv.prefill(cfg["seed"], ctx)
    tok, pos, ref, gap = first.copy(), pos0.copy(), [[] for _ in range(B)], [[] for _ in range(B)]
    for _ in range(N):
        lg = oracle.decode(om, kv, tok[:, None], pos, precision=64)["logits"][:, 0]
        srt = np.sort(lg, axis=1)
        nxt = lg.argmax(1).astype(np.int32)
        for b in range(B):
            ref[b].append(int(nxt[b]))
            gap[b].append(float(srt[b, -1] - srt[b, -2]))
        tok, pos = nxt, pos + 1
    kv.close()

    kv = oracle.KV(om, B, ctx + 64)
    kv.prefill(cfg["seed"], ctx)
    wrong = {1, 2, 9}
    loop = GreedySpecLoop(OracleVerifyModel(om, kv), None, first, pos0, T, cfg["vocab"],
                          PlantedDrafter(ref, cfg["vocab"], wrong=lambda b, i: i in wrong), device="cpu")
    while min(len(e) for e in loop.emitted) < N - T:
        loop.step()
    # drafts 0..3 with 1 wrong -> 2; drafts 2..5 with 2 wrong -> 1; drafts 3..6 -> 5; drafts 8..11 with 9 wrong -> 2
    assert [int(a[0]) for a in loop.accepts[:4]] == [2, 1, 5, 2]
    for b in range(B):
        n = min(len(loop.emitted[b]), N)
        i = next((i for i in range(n) if loop.emitted[b][i] != ref[b][i]), n)
        assert i == n or gap[b][i] < 1e-9, (b, i)
    kv.close()
    om.close()


@pytest.mark.gpu
def test_verify_loop_matches_the_oracles_greedy_decoding():
    import time
    import oracle
    import moe_decode_megakernel_02_gb300 as mk
    from moe_decode_megakernel_02_gb300 import workload
    from synth import configs
    import parity

    cfg = configs.scaled(configs.VERIFY, n_layers=2)
    B, T, ctx, N = 2, 7, 300, 30
    V = cfg["vocab"]
    model = workload.load_synthetic(cfg, max_batch=B, max_tokens_per_seq=T, max_ctx=ctx + 64)
    first = workload.tokens(cfg, 0, B, 1)[:, 0].astype(np.int32)
    pos0 = np.full(B, ctx, dtype=np.int32)

    # reference: the oracle's plain greedy decoding, one token per step
    om = oracle.Model(cfg)
    okv = oracle.KV(om, B, ctx + 64)
    for l in range(cfg["n_layers"]):
        for b in range(B):
            okv.write(l, b, 0, parity._prefill_rows(cfg, l, b, ctx))
    tok, pos = first.copy(), pos0.copy()
    ref, gap = [[] for _ in range(B)], [[] for _ in range(B)]
    for _ in range(N):
        lg = oracle.decode(om, okv, tok[:, None], pos)["logits"][:, 0]
        srt = np.sort(lg, axis=1)
        nxt = lg.argmax(1).astype(np.int32)
        for b in range(B):
            ref[b].append(int(nxt[b]))
            gap[b].append(float(srt[b, -1] - srt[b, -2]))
        tok, pos = nxt, pos + 1
    okv.close()
    om.close()

    # the speculative loop over the CUDA verify step, drafts = the oracle's
    # greedy tokens with planted errors
    kv = mk.KVCache(model, B, ctx + 64)
    workload.prefill(kv, cfg, ctx)
    wrong = {3, 4, 12, 20}
    loop = GreedySpecLoop(model, kv, first, pos0, T, V, PlantedDrafter(ref, V, wrong=lambda b, i: i in wrong))
    t0 = time.perf_counter()
    steps = 0
    while min(len(e) for e in loop.emitted) < N - T:
        loop.step()
        steps += 1
    dt = time.perf_counter() - t0
    acc = np.array(loop.accepts)
    print(f"spec loop: {steps} steps, accept per step {acc[:, 0].tolist()}, "
          f"{acc.sum() / dt:.0f} tokens/s with host bookkeeping")
    first_tie = []
    for b in range(B):
        # the GPU loop emits the oracle's greedy tokens; the two may part only
        # at a token whose top-two oracle logits are within the logit
        # tolerance of each other (after that the contexts differ)
        n = min(len(loop.emitted[b]), N)
        i = next((i for i in range(n) if loop.emitted[b][i] != ref[b][i]), n)
        assert i == n or gap[b][i] <= 2 * parity.MAX_ABS, (b, i, gap[b][i])
        first_tie.append(next((j for j in range(N) if gap[b][j] <= 2 * parity.MAX_ABS), N))
    # accept lengths implied by the planted errors: drafts 0..5 with 3 wrong -> 4,
    # then drafts 4..9 with 4 wrong -> 1, then 5..10 -> 7, then 12..17 with 12 wrong -> 1
    # (checked as far as sequence 0's greedy decisions are clear)
    expect = [4, 1, 7, 1]
    done = [0, 4, 5, 12, 13]
    for s_, a in enumerate(expect):
        if done[s_ + 1] + 1 <= first_tie[0]:
            assert acc[s_, 0] == a, (s_, acc[:, 0].tolist())
