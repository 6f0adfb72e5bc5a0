"""Seeded synthetic inputs for the MoE decode step (weights, pre-filled KV, token ids).

This package is the only code shared by the CPU oracle and the CUDA-path
harness. It holds no model arithmetic: it maps (seed, tensor id, index) to
numbers as defined in ``synth.h`` and knows each tensor's shape and scale.
``configs`` holds the five workload shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import configs  # noqa: F401  (re-export)

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
HOST_LIB = os.path.join(_BUILD, "libsynth.so")
CUDA_LIB = os.path.join(_BUILD, "libsynth_cuda.so")

# tensor kinds (synth.h enum synth_kind)
EMBED, LM_HEAD, FINAL_NORM, ATTN_NORM, FFN_NORM = 1, 2, 3, 4, 5
WQ, WK, WV, WO = 6, 7, 8, 9
WDQ, Q_NORM, WUQ, WDKV, KV_NORM, WUKV = 10, 11, 12, 13, 14, 15
ROUTER, GATE, UP, DOWN, SH_GATE, SH_UP, SH_DOWN = 16, 17, 18, 19, 20, 21, 22
GATE_SCALE, UP_SCALE, DOWN_SCALE, SH_GATE_SCALE, SH_UP_SCALE, SH_DOWN_SCALE = 23, 24, 25, 26, 27, 28
KV_K, KV_V, KV_LATENT, TOKENS = 40, 41, 42, 43

# MXFP8 expert weights: E4M3 codes of sigma-16 draws, one E8M0 scale per 32
# elements of a row (synth.h); the scale kind of a code kind is kind + 6
F8_SIGMA = 16.0
MX_BLOCK = 32
F8_KINDS = (GATE, UP, DOWN, SH_GATE, SH_UP, SH_DOWN)
SCALE_OF = {k: k + 6 for k in F8_KINDS}

GLOBAL_KINDS = (EMBED, LM_HEAD, FINAL_NORM)
LAYER_KINDS = (ATTN_NORM, FFN_NORM, WQ, WK, WV, WO, WDQ, Q_NORM, WUQ, WDKV, KV_NORM, WUKV,
               ROUTER, SH_GATE, SH_UP, SH_DOWN)
EXPERT_KINDS = (GATE, UP, DOWN)


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "d_model", "vocab", "attn_kind",
        "n_q_heads", "n_kv_heads", "head_dim",
        "q_lora_rank", "kv_lora_rank", "qk_nope_dim", "qk_rope_dim", "v_head_dim",
        "n_routed_experts", "top_k", "n_shared_experts", "ffn_dim", "shared_ffn_dim")]


def build(verbose: bool = False) -> list:
    """Return the compile commands for the host and device generator libraries."""
    os.makedirs(_BUILD, exist_ok=True)
    src_h = os.path.join(_HERE, "synth_host.c")
    src_d = os.path.join(_HERE, "synth_cuda.cu")
    return [
        ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
         src_h, "-o", HOST_LIB],
        ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
         "-Xcompiler", "-fPIC", "-shared", src_d, "-o", CUDA_LIB],
    ]


_host = None
_cuda = None


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            for cmd in build()[:1]:
                subprocess.check_call(cmd)
        lib = ctypes.CDLL(HOST_LIB)
        lib.synth_fill_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_float, ctypes.c_float, ctypes.c_uint64, ctypes.c_int]
        lib.synth_fill_bf16.restype = None
        lib.synth_tensor_id.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        lib.synth_tensor_id.restype = ctypes.c_uint64
        lib.synth_token.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32]
        lib.synth_token.restype = ctypes.c_int32
        lib.synth_weight_spec.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32] + [ctypes.c_void_p] * 4
        lib.synth_weight_spec.restype = ctypes.c_int
        lib.synth_kv_row.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32]
        lib.synth_kv_row.restype = ctypes.c_int32
        lib.synth_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_draw.restype = ctypes.c_uint64
        lib.synth_mix64.argtypes = [ctypes.c_uint64]
        lib.synth_mix64.restype = ctypes.c_uint64
        lib.synth_bf16_rne.argtypes = [ctypes.c_float]
        lib.synth_bf16_rne.restype = ctypes.c_uint16
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float, ctypes.c_float]
        lib.synth_normal_f32.restype = ctypes.c_float
        lib.synth_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_key.restype = ctypes.c_uint64
        lib.synth_scale_const.argtypes = [ctypes.c_float]
        lib.synth_scale_const.restype = ctypes.c_float
        lib.synth_e4m3_rne.argtypes = [ctypes.c_float]
        lib.synth_e4m3_rne.restype = ctypes.c_uint8
        lib.synth_fill_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_int]
        lib.synth_fill_e4m3.restype = None
        lib.synth_fill_e8m0.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint64]
        lib.synth_fill_e8m0.restype = None
        _host = lib
    return _host


def _load_cuda():
    global _cuda
    if _cuda is None:
        if not os.path.exists(CUDA_LIB):
            raise RuntimeError("libsynth_cuda.so is not built (run __graft_entry__.build())")
        lib = ctypes.CDLL(CUDA_LIB)
        lib.synth_fill_bf16_cuda.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                             ctypes.c_float, ctypes.c_float, ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_fill_bf16_cuda.restype = ctypes.c_int
        for fn in (lib.synth_fill_e4m3_cuda, lib.synth_fill_e8m0_cuda):
            fn.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                           ctypes.c_void_p]
            fn.restype = ctypes.c_int
        _cuda = lib
    return _cuda


def host_lib():
    return _load_host()


def dims_of(cfg) -> Dims:
    return Dims(*[int(cfg[f]) for f, _ in Dims._fields_])


def tensor_id(kind: int, layer: int = -1, expert: int = 0) -> int:
    return int(_load_host().synth_tensor_id(kind, layer, expert))


def weight_spec(cfg, kind: int):
    """(rows, cols, sigma, mean) of a weight kind under the recipe, or None if absent."""
    d = dims_of(cfg)
    r, c = ctypes.c_int32(), ctypes.c_int32()
    s, m = ctypes.c_float(), ctypes.c_float()
    rc = _load_host().synth_weight_spec(ctypes.byref(d), kind, ctypes.byref(r), ctypes.byref(c),
                                        ctypes.byref(s), ctypes.byref(m))
    if rc != 0:
        return None
    return r.value, c.value, s.value, m.value


def kv_row(cfg, kind: int) -> int:
    return int(_load_host().synth_kv_row(ctypes.byref(dims_of(cfg)), kind))


def fill_bf16_host(n: int, seed: int, tid: int, sigma: float, mean: float = 0.0, index0: int = 0,
                   threads: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _load_host().synth_fill_bf16(out.ctypes.data, n, seed, tid, sigma, mean, index0, threads)
    return out


def fill_bf16_cuda(dev_ptr: int, n: int, seed: int, tid: int, sigma: float, mean: float = 0.0,
                   index0: int = 0, stream: int = 0) -> None:
    rc = _load_cuda().synth_fill_bf16_cuda(dev_ptr, n, seed, tid, sigma, mean, index0, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_bf16_cuda failed with CUDA error {rc}")


def e4m3_rne(f: float) -> int:
    """The generator's fp32 -> FP8 E4M3 rounding (nearest, ties to even, saturating)."""
    return int(_load_host().synth_e4m3_rne(f))


def fill_e4m3_host(n: int, seed: int, tid: int, index0: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _load_host().synth_fill_e4m3(out.ctypes.data, n, seed, tid, index0, 1)
    return out


def fill_e8m0_host(n: int, seed: int, tid: int, index0: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _load_host().synth_fill_e8m0(out.ctypes.data, n, seed, tid, index0)
    return out


def fill_e4m3_cuda(dev_ptr: int, n: int, seed: int, tid: int, index0: int = 0, stream: int = 0) -> None:
    rc = _load_cuda().synth_fill_e4m3_cuda(dev_ptr, n, seed, tid, index0, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_e4m3_cuda failed with CUDA error {rc}")


def fill_e8m0_cuda(dev_ptr: int, n: int, seed: int, tid: int, index0: int = 0, stream: int = 0) -> None:
    rc = _load_cuda().synth_fill_e8m0_cuda(dev_ptr, n, seed, tid, index0, stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_e8m0_cuda failed with CUDA error {rc}")


def token(seed: int, step: int, b: int, t: int, vocab: int) -> int:
    return int(_load_host().synth_token(seed, step, b, t, vocab))


def tokens(seed: int, step: int, batch: int, T: int, vocab: int) -> np.ndarray:
    """Token ids [batch, T] (int32) of decode step `step`."""
    return np.array([[token(seed, step, b, t, vocab) for t in range(T)] for b in range(batch)], dtype=np.int32)


def weight_tensors(cfg):
    """Yield (kind, layer, expert, rows, cols, sigma, mean) for every weight tensor of the model."""
    for kind in GLOBAL_KINDS:
        r, c, s, m = weight_spec(cfg, kind)
        yield kind, -1, 0, r, c, s, m
    for layer in range(cfg["n_layers"]):
        for kind in LAYER_KINDS:
            spec = weight_spec(cfg, kind)
            if spec is not None:
                yield (kind, layer, 0) + tuple(spec)
        for e in range(cfg["n_routed_experts"]):
            for kind in EXPERT_KINDS:
                yield (kind, layer, e) + tuple(weight_spec(cfg, kind))


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)
