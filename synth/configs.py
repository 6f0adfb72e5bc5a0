"""The five workload shapes of the MoE decode step (dimensions, seed, context, batches).

Shapes are the ones the workload descriptions state; where they are silent the
value chosen is noted inline. ``ctx`` is the number of pre-filled KV positions
(the first decoded position equals ``ctx``).
"""

_COMMON = dict(rms_eps=1e-6, rope_theta=1e4, kv_page_size=64,
               q_lora_rank=0, kv_lora_rank=0, qk_nope_dim=0, qk_rope_dim=0, v_head_dim=0)

TINY = dict(_COMMON, name="tiny", n_layers=2, d_model=256, vocab=1024, attn_kind=0,
            n_q_heads=4, n_kv_heads=2, head_dim=64,
            n_routed_experts=8, top_k=2, n_shared_experts=1, ffn_dim=512, shared_ffn_dim=512,
            seed=0, ctx=64, batches=(1,), T=1, steps=16)

MID = dict(_COMMON, name="mid", n_layers=8, d_model=2048, vocab=32000, attn_kind=0,
           n_q_heads=16, n_kv_heads=4, head_dim=128,
           n_routed_experts=64, top_k=6, n_shared_experts=1, ffn_dim=1024, shared_ffn_dim=1024,
           seed=1234, ctx=4096, batches=(1, 4, 8), T=1, steps=1)

DEEP = dict(_COMMON, name="deep", n_layers=92, d_model=2048, vocab=64000, attn_kind=1,
            n_q_heads=16, n_kv_heads=1, head_dim=0,
            q_lora_rank=1024, kv_lora_rank=512, qk_nope_dim=128, qk_rope_dim=64, v_head_dim=128,
            n_routed_experts=64, top_k=8, n_shared_experts=1, ffn_dim=768, shared_ffn_dim=768,
            seed=1234, ctx=8192, batches=(1, 2, 4, 8), T=1, steps=1)

DENSE = dict(_COMMON, name="dense", n_layers=64, d_model=5120, vocab=151936, attn_kind=0,
             n_q_heads=40, n_kv_heads=8, head_dim=128,
             n_routed_experts=0, top_k=0, n_shared_experts=1, ffn_dim=0, shared_ffn_dim=17408,
             seed=1234, ctx=4096, batches=(1, 8), T=1, steps=1)

VERIFY = dict(DEEP, name="verify", batches=(8,), T=7)

ALL = {c["name"]: c for c in (TINY, MID, DEEP, DENSE, VERIFY)}

# the deep model with MXFP8 expert weights (E4M3 codes, one E8M0 scale per 32
# codes of a row)
DEEP_MXFP8 = dict(DEEP, name="deep_mxfp8", expert_format=1, batches=(1, 8))


def scaled(cfg, **over):
    """A copy of `cfg` with some fields replaced (for reduced-size test cases)."""
    out = dict(cfg)
    out.update(over)
    return out


def weight_bytes(cfg) -> int:
    """Total bf16 bytes of all weight tensors of the model."""
    d, L, V = cfg["d_model"], cfg["n_layers"], cfg["vocab"]
    per = 2 * d  # two norm gains
    if cfg["attn_kind"] == 0:
        hq, hkv, hd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
        per += d * hq * hd * 2 + d * hkv * hd * 2
    else:
        H = cfg["n_q_heads"]
        ql, kl = cfg["q_lora_rank"], cfg["kv_lora_rank"]
        nope, rope, vd = cfg["qk_nope_dim"], cfg["qk_rope_dim"], cfg["v_head_dim"]
        per += ql * d + ql + H * (nope + rope) * ql + (kl + rope) * d + kl + H * (nope + vd) * kl + d * H * vd
    E = cfg["n_routed_experts"]
    if E:
        per += E * d + E * 3 * d * cfg["ffn_dim"]
    if cfg["n_shared_experts"]:
        per += 3 * d * cfg["shared_ffn_dim"]
    return 2 * (L * per + 2 * V * d + d)
