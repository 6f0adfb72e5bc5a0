"""Greedy speculative decoding over the verify step.

Speculative decoding as the DSpark paragraphs of "16 块谷歌 TPU v7 跑 Kimi K3"
(section "同样 16 块芯片，TPU 快 57%") describe it: a drafter proposes several
tokens, the model scores them all in one step, and the accepted prefix plus
one model token are kept. Here the drafter is synthetic (the pages' trained
drafter is out of scope) and acceptance is greedy.

Each iteration scores, per sequence, its last committed token followed by
T - 1 drafts in one decode step of T positions (causal within the block).
The step computes its own greedy acceptance (1 + the number of leading
drafts equal to the argmax before them) and the argmax of every row. The
loop keeps the accepted drafts and the model's token after them (the argmax
of row accept - 1), advances the position by `accept`, and feeds that token
first in the next step. Cache rows written for rejected drafts lie past the
new position, so the next step overwrites them: rollback needs no copy. The
tokens produced are those of plain greedy decoding, `accept` per step.

Host work per step is bookkeeping only: the draft block goes to the device,
`accept` and the row argmaxes come back; every step of the model runs in the
CUDA library.
"""
from __future__ import annotations

import numpy as np


class GreedySpecLoop:
    """Speculative greedy decoding of `batch` sequences with blocks of T tokens.

    model, kv: a loaded `Model` and its `KVCache` (or objects with the same
    `decode_step(kv, tokens, positions, logits, accept)`, `check()` and
    `last_argmax(out)` methods). first_tokens[b] is the last token already
    known for sequence b, to be written at position positions[b].
    drafter(loop) returns int32 [batch, T - 1] drafts for the next step.
    """

    def __init__(self, model, kv, first_tokens, positions, T, vocab, drafter, device="cuda"):
        import torch
        self.model, self.kv, self.T, self.V, self.drafter = model, kv, int(T), int(vocab), drafter
        if self.T < 2:
            raise ValueError("speculative steps need T >= 2")
        self.t0 = np.asarray(first_tokens, dtype=np.int32).copy()
        self.pos = np.asarray(positions, dtype=np.int32).copy()
        B = self.B = len(self.t0)
        if self.pos.shape != (B,):
            raise ValueError("one position per sequence")
        self.emitted = [[] for _ in range(B)]
        self.accepts = []
        self.tok = torch.empty((B, self.T), dtype=torch.int32, device=device)
        self.posd = torch.empty((B,), dtype=torch.int32, device=device)
        self.logits = torch.empty((B * self.T, self.V), dtype=torch.float32, device=device)
        self.acc = torch.empty((B,), dtype=torch.int32, device=device)
        self.amax = torch.empty((B * self.T,), dtype=torch.int32)  # host

    def step(self, stream=None):
        """One verify step; returns the accept lengths (int32 [batch])."""
        import torch
        drafts = np.asarray(self.drafter(self), dtype=np.int32)
        if drafts.shape != (self.B, self.T - 1):
            raise ValueError(f"drafter returned shape {drafts.shape}, expected {(self.B, self.T - 1)}")
        block = np.concatenate([self.t0[:, None], drafts], axis=1)
        self.tok.copy_(torch.from_numpy(block))
        self.posd.copy_(torch.from_numpy(self.pos))
        self.model.decode_step(self.kv, self.tok, self.posd, self.logits, self.acc, stream=stream)
        self.model.check(stream)
        acc = self.acc.cpu().numpy().astype(np.int32)
        am = self.model.last_argmax(self.amax, stream=stream).numpy()
        for b in range(self.B):
            a = int(acc[b])
            nxt = int(am[b * self.T + a - 1])
            self.emitted[b].extend(int(x) for x in drafts[b, :a - 1])
            self.emitted[b].append(nxt)
            self.pos[b] += a
            self.t0[b] = nxt
        self.accepts.append(acc)
        return acc


class PlantedDrafter:
    """Drafts read from known continuations, with chosen drafts replaced.

    streams[b] is the token sequence that follows sequence b's first token.
    wrong(b, i) says whether the draft for continuation index i is replaced
    by another token ((true + 1) mod V). With exact continuations every draft
    is accepted (accept = T each step)."""

    def __init__(self, streams, vocab, wrong=lambda b, i: False):
        self.streams = [list(s) for s in streams]
        self.V = vocab
        self.wrong = wrong

    def __call__(self, loop):
        out = np.zeros((loop.B, loop.T - 1), dtype=np.int32)
        for b in range(loop.B):
            n = len(loop.emitted[b])  # continuation index of the first draft
            for j in range(loop.T - 1):
                i = n + j
                tok = self.streams[b][i] if i < len(self.streams[b]) else 0
                out[b, j] = (tok + 1) % self.V if self.wrong(b, i) else tok
        return out


class RandomDrafter:
    """Uniform random drafts from a seeded generator (acceptance near 1)."""

    def __init__(self, vocab, seed=0):
        self.V = vocab
        self.rng = np.random.default_rng(seed)

    def __call__(self, loop):
        return self.rng.integers(0, self.V, size=(loop.B, loop.T - 1), dtype=np.int32)
