"""CPU oracle of the MoE decode step (ctypes binding of liboracle.so).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package. It shares
no code with the CUDA path (its one shared dependency is the ``synth`` input
generator, which holds no model arithmetic).

Parity status: every function is pinned by CPU tests in tests/test_oracle_*.py
against closed forms, library routines it does not itself use, invariants and
brute force (see the test docstrings for which pin covers what).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_BUILD = os.path.join(_HERE, "_build")
LIB = os.path.join(_BUILD, "liboracle.so")


def build_cmds() -> list:
    os.makedirs(_BUILD, exist_ok=True)
    return [["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
             os.path.join(_HERE, "oracle.cpp"), os.path.join(_ROOT, "synth", "synth_host.c"),
             "-o", LIB]]


class Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "d_model", "vocab", "attn_kind",
        "n_q_heads", "n_kv_heads", "head_dim",
        "q_lora_rank", "kv_lora_rank", "qk_nope_dim", "qk_rope_dim", "v_head_dim",
        "n_routed_experts", "top_k", "n_shared_experts", "ffn_dim", "shared_ffn_dim")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("expert_format", ctypes.c_int32)]

# expert_format values: every weight bf16, or MXFP8 expert weights
BF16, MXFP8 = 0, 1


def cfg_struct(cfg) -> Cfg:
    vals = {f: int(cfg[f]) for f, t in Cfg._fields_ if t is ctypes.c_int32 and f != "expert_format"}
    return Cfg(**vals, rms_eps=float(cfg["rms_eps"]), rope_theta=float(cfg["rope_theta"]),
               expert_format=int(cfg.get("expert_format", BF16)))


_lib = None
P = ctypes.c_void_p
I32 = ctypes.c_int32
DP = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            for cmd in build_cmds():
                subprocess.check_call(cmd)
        L = ctypes.CDLL(LIB)
        L.oracle_create.argtypes = [ctypes.POINTER(Cfg), ctypes.c_uint64, ctypes.c_int, ctypes.c_int]
        L.oracle_create.restype = P
        L.oracle_destroy.argtypes = [P]
        L.oracle_set_tensor.argtypes = [P, I32, I32, I32, P, ctypes.c_int64]
        L.oracle_set_tensor.restype = ctypes.c_int
        L.oracle_get_tensor.argtypes = [P, I32, I32, I32, P, ctypes.c_int64]
        L.oracle_get_tensor.restype = ctypes.c_int64
        L.oracle_kv_create.argtypes = [P, I32, I32]
        L.oracle_kv_create.restype = P
        L.oracle_kv_destroy.argtypes = [P]
        L.oracle_kv_prefill.argtypes = [P, ctypes.c_uint64, I32, ctypes.c_int]
        L.oracle_kv_prefill.restype = ctypes.c_int
        L.oracle_kv_rows.argtypes = [P, I32, I32, I32, I32, P, ctypes.c_int]
        L.oracle_kv_rows.restype = ctypes.c_int
        L.oracle_kv_row_len.argtypes = [P]
        L.oracle_kv_row_len.restype = I32
        L.oracle_decode.argtypes = [P, P, P, P, I32, I32, ctypes.c_int, ctypes.c_int, P, P, P, P, P]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_full_recompute.argtypes = [P, P, I32, I32, ctypes.c_int, P]
        L.oracle_full_recompute.restype = ctypes.c_int
        L.oracle_rmsnorm.argtypes = [P, P, I32, ctypes.c_double, P]
        L.oracle_rope.argtypes = [P, I32, I32, ctypes.c_double]
        L.oracle_softmax.argtypes = [P, I32, P]
        L.oracle_topk.argtypes = [P, I32, I32, P, P, P]
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_mx_dequant.argtypes = [P, P, I32, I32, P]
        L.oracle_mx_dequant.restype = None
        L.oracle_attend.argtypes = [P, P, P, I32, I32, ctypes.c_double, P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class Model:
    """Oracle model over synthetic weights (seeded), optionally with tensors replaced."""

    def __init__(self, cfg, seed=None, lazy=False, gen_threads=0):
        self.cfg = cfg
        self._c = cfg_struct(cfg)
        self.h = lib().oracle_create(ctypes.byref(self._c), int(cfg["seed"] if seed is None else seed),
                                     int(lazy), int(gen_threads))
        if not self.h:
            raise ValueError("oracle_create rejected the configuration")

    def close(self):
        if self.h:
            lib().oracle_destroy(self.h)
            self.h = None

    __del__ = close

    def set_tensor(self, kind, layer, expert, data_u16):
        a = np.ascontiguousarray(data_u16, dtype=np.uint16)
        if lib().oracle_set_tensor(self.h, kind, layer, expert, a.ctypes.data, a.size) != 0:
            raise ValueError("oracle_set_tensor: bad tensor")

    def get_tensor(self, kind, layer=-1, expert=0):
        n = lib().oracle_get_tensor(self.h, kind, layer, expert, None, 0)
        if n < 0:
            raise ValueError("no such tensor")
        out = np.empty(n, dtype=np.uint16)
        lib().oracle_get_tensor(self.h, kind, layer, expert, out.ctypes.data, n)
        return out


class KV:
    def __init__(self, model: Model, batch: int, max_pos: int):
        self.model = model
        self.batch = batch
        self.max_pos = max_pos
        self.h = lib().oracle_kv_create(model.h, batch, max_pos)
        if not self.h:
            raise ValueError("oracle_kv_create failed")
        self.row = lib().oracle_kv_row_len(self.h)

    def close(self):
        if self.h:
            lib().oracle_kv_destroy(self.h)
            self.h = None

    __del__ = close

    def prefill(self, seed: int, ctx: int, gen_threads: int = 0):
        if lib().oracle_kv_prefill(self.h, seed, ctx, gen_threads) != 0:
            raise ValueError("prefill failed")

    def read(self, layer, seq, pos0, n):
        out = np.empty((n, self.row), dtype=np.uint16)
        if lib().oracle_kv_rows(self.h, layer, seq, pos0, n, out.ctypes.data, 0) != 0:
            raise ValueError("bad kv range")
        return out

    def write(self, layer, seq, pos0, rows_u16):
        a = np.ascontiguousarray(rows_u16, dtype=np.uint16)
        if lib().oracle_kv_rows(self.h, layer, seq, pos0, a.shape[0], a.ctypes.data, 1) != 0:
            raise ValueError("bad kv range")


def decode(model: Model, kv: KV, tokens, positions, precision=64, mla_absorbed=True, want_logits=True):
    """One decode/verify step. tokens [B, T] int, positions [B] int.

    Returns dict(logits [B, T, V] float64, route_idx [L, B*T, k], route_w, route_margin [L, B*T],
    accept [B] (T > 1 only)).
    """
    cfg = model.cfg
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    B, T = tok.shape
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    L, k, V = cfg["n_layers"], max(cfg["top_k"], 1), cfg["vocab"]
    logits = np.empty((B, T, V), dtype=np.float64) if (want_logits or T > 1) else None
    ridx = np.full((L, B * T, k), -1, dtype=np.int32)
    rw = np.zeros((L, B * T, k), dtype=np.float64)
    rm = np.zeros((L, B * T), dtype=np.float64)
    acc = np.zeros(B, dtype=np.int32) if T > 1 else None
    rc = lib().oracle_decode(model.h, kv.h, tok.ctypes.data, pos.ctypes.data, B, T, precision, int(mla_absorbed),
                             _ptr(logits), ridx.ctypes.data, rw.ctypes.data, rm.ctypes.data, _ptr(acc))
    if rc != 0:
        raise ValueError(f"oracle_decode failed ({rc})")
    return dict(logits=logits, route_idx=ridx, route_w=rw, route_margin=rm, accept=acc)


def full_recompute(model: Model, tokens, precision=64):
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    B, P_ = tok.shape
    out = np.empty((B, P_, model.cfg["vocab"]), dtype=np.float64)
    if lib().oracle_full_recompute(model.h, tok.ctypes.data, B, P_, precision, out.ctypes.data) != 0:
        raise ValueError("oracle_full_recompute failed")
    return out


# ---- building blocks (fp64) ----

def rmsnorm(x, gain_u16, eps):
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(gain_u16, dtype=np.uint16)
    out = np.empty_like(x)
    lib().oracle_rmsnorm(x.ctypes.data, g.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def rope(x, pos, theta):
    x = np.array(x, dtype=np.float64)
    lib().oracle_rope(x.ctypes.data, x.size, pos, theta)
    return x


def softmax(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().oracle_softmax(x.ctypes.data, x.size, out.ctypes.data)
    return out


def topk(logits, k):
    x = np.ascontiguousarray(logits, dtype=np.float64)
    idx = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    mg = np.empty(1, dtype=np.float64)
    lib().oracle_topk(x.ctypes.data, x.size, k, idx.ctypes.data, w.ctypes.data, mg.ctypes.data)
    return idx, w, float(mg[0])


def silu(z: float) -> float:
    return float(lib().oracle_silu(z))


def attend(q, K_u16, V_u16, scale):
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K_u16, dtype=np.uint16)
    V = np.ascontiguousarray(V_u16, dtype=np.uint16)
    n, hd = K.shape
    out = np.empty(hd, dtype=np.float64)
    lib().oracle_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, n, hd, scale, out.ctypes.data)
    return out


def e4m3_value(code: int) -> float:
    """Value of an FP8 E4M3 code (the oracle's decoder)."""
    return float(lib().oracle_e4m3_value(code))


def mx_dequant(codes_u8, scales_u8, rows: int, cols: int) -> np.ndarray:
    """MX dequantisation of E4M3 codes [rows, cols] with E8M0 scales [rows, cols/32] (fp64)."""
    q = np.ascontiguousarray(codes_u8, dtype=np.uint8).reshape(rows, cols)
    sc = np.ascontiguousarray(scales_u8, dtype=np.uint8).reshape(rows, cols // 32)
    out = np.empty((rows, cols))
    lib().oracle_mx_dequant(q.ctypes.data, sc.ctypes.data, rows, cols, out.ctypes.data)
    return out
