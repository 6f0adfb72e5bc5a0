"""The bench's algorithmic byte count (CPU only), checked against the
generator's own tensor shapes: a step touches every non-routed weight, the
routed experts it selected, the LM head, its embedding rows and the KV cache.
"""
import numpy as np

import bench
import synth
from synth import configs


def _tensor_bytes(cfg, kind, per_elem):
    r, c, _, _ = synth.weight_spec(cfg, kind)
    return r * c * per_elem


def _expected(cfg, idx, pos, f8):
    L, d, V = cfg["n_layers"], cfg["d_model"], cfg["vocab"]
    layer = sum(_tensor_bytes(cfg, k, 2) for k in synth.LAYER_KINDS
                if k not in (synth.SH_GATE, synth.SH_UP, synth.SH_DOWN) and synth.weight_spec(cfg, k))
    def expert(kinds):
        if not f8:
            return sum(_tensor_bytes(cfg, k, 2) for k in kinds)
        return sum(_tensor_bytes(cfg, k, 1) + _tensor_bytes(cfg, synth.SCALE_OF[k], 1) for k in kinds)
    sh = expert((synth.SH_GATE, synth.SH_UP, synth.SH_DOWN))
    routed = expert((synth.GATE, synth.UP, synth.DOWN))
    row = cfg["kv_lora_rank"] + cfg["qk_rope_dim"]
    total = L * (layer + sh) + _tensor_bytes(cfg, synth.LM_HEAD, 2)
    total += _tensor_bytes(cfg, synth.FINAL_NORM, 2) + 2 * d  # final norm, one embedding row
    total += sum(len(set(np.asarray(idx[l]).ravel().tolist())) for l in range(L)) * routed
    total += 2 * row * L * (pos + 1)  # KV read (pos positions) and written (one)
    return total


def test_algorithmic_bytes_bf16_and_mxfp8():
    rng = np.random.default_rng(0)
    for cfg, f8 in ((configs.scaled(configs.DEEP, n_layers=3), False),
                    (configs.scaled(configs.DEEP_MXFP8, n_layers=3), True)):
        idx = [rng.choice(64, size=(1, 8), replace=False) for _ in range(3)]
        got = bench.algorithmic_bytes(cfg, 1, 1, [8192], idx)
        assert got == _expected(cfg, idx, 8192, f8)
    # the MXFP8 model moves 1 + 1/32 bytes per expert weight instead of 2
    idx = [np.arange(8).reshape(1, 8)] * 3
    a = bench.algorithmic_bytes(configs.scaled(configs.DEEP, n_layers=3), 1, 1, [8192], idx)
    b = bench.algorithmic_bytes(configs.scaled(configs.DEEP_MXFP8, n_layers=3), 1, 1, [8192], idx)
    ex = 3 * (9 * 3 * 2048 * 768)  # 3 layers x 9 experts (8 routed + shared) x 3 matrices
    assert a - b == 2 * ex - ex * 33 // 32
