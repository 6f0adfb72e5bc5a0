"""Seeded synthetic workloads for the decode megakernel (weights, pre-filled KV, token ids).

Every number comes from the shared input generator (`synth`): weights are
bf16 draws of N(0, 0.02) (RMSNorm gains 1 + N(0, 0.02)), pre-filled KV entries
bf16 N(0, 1), token ids uniform. Weights are generated in device memory by the
library itself (mk_load_synthetic); KV entries by the generator's CUDA
implementation, then handed to mk_kv_write.
"""
from __future__ import annotations

import numpy as np
import torch

import synth

from . import KVCache, Model, make_config


def load_synthetic(cfg, max_batch, max_tokens_per_seq, max_ctx, seed=None):
    """The model of workload `cfg` with the generator's seeded weights (mk_load_synthetic)."""
    seed = cfg["seed"] if seed is None else seed
    return Model.synthetic(make_config(cfg, max_batch, max_tokens_per_seq, max_ctx), seed)


def kv_row(cfg) -> int:
    if cfg["attn_kind"] == 0:
        return 2 * cfg["n_kv_heads"] * cfg["head_dim"]
    return cfg["kv_lora_rank"] + cfg["qk_rope_dim"]


def prefill(kv: KVCache, cfg, ctx: int, seed=None, batch=None, device="cuda"):
    """Fill positions [0, ctx) of every layer and sequence from the generator."""
    seed = cfg["seed"] if seed is None else seed
    batch = kv.batch if batch is None else batch
    if ctx == 0:
        return
    stream = torch.cuda.current_stream().cuda_stream
    if cfg["attn_kind"] == 0:
        half = cfg["n_kv_heads"] * cfg["head_dim"]
        k = torch.empty((ctx, half), dtype=torch.int16, device=device)
        v = torch.empty((ctx, half), dtype=torch.int16, device=device)
        for l in range(cfg["n_layers"]):
            for b in range(batch):
                synth.fill_bf16_cuda(k.data_ptr(), ctx * half, seed, synth.tensor_id(synth.KV_K, l, b), 1.0, 0.0,
                                     0, stream)
                synth.fill_bf16_cuda(v.data_ptr(), ctx * half, seed, synth.tensor_id(synth.KV_V, l, b), 1.0, 0.0,
                                     0, stream)
                rows = torch.cat([k, v], dim=1).contiguous()
                kv.write(l, b, 0, rows)
    else:
        row = kv_row(cfg)
        lat = torch.empty((ctx, row), dtype=torch.int16, device=device)
        for l in range(cfg["n_layers"]):
            for b in range(batch):
                synth.fill_bf16_cuda(lat.data_ptr(), ctx * row, seed, synth.tensor_id(synth.KV_LATENT, l, b), 1.0,
                                     0.0, 0, stream)
                kv.write(l, b, 0, lat)
    torch.cuda.synchronize()


def tokens(cfg, step, batch, T, seed=None) -> np.ndarray:
    seed = cfg["seed"] if seed is None else seed
    return synth.tokens(seed, step, batch, T, cfg["vocab"])
