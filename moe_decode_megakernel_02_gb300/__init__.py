"""Python binding of the single-launch MoE decode megakernel (libmk.so, include/mk.h).

Argument marshalling only: every step of the decode path runs in the CUDA
library. PyTorch supplies device memory and streams. There is no CPU or
eager-PyTorch fallback: if the library is missing or CUDA is unavailable the
calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_BUILD = os.path.join(_HERE, "_build")
# the library this process loads: libmk.so, or another build of the same
# sources named by MK_LIB (the 2-slot ring build used by the shrunken-ring
# parity check)
LIB = os.environ.get("MK_LIB") or os.path.join(_BUILD, "libmk.so")
LIB_NSLOT2 = os.path.join(_BUILD, "libmk_nslot2.so")
HEADER = os.path.join(_ROOT, "include", "mk.h")

OK, ERR_INVALID_ARG, ERR_OOM, ERR_CUDA, ERR_UNSUPPORTED, ERR_TIMEOUT, ERR_STATE = 0, -1, -2, -3, -4, -5, -6
ATTN_GQA, ATTN_MLA = 0, 1
EXPERT_BF16, EXPERT_MXFP8 = 0, 1  # mk_config.expert_format
EXPORTS = ("mk_load_weights", "mk_load_synthetic", "mk_alloc_kv", "mk_kv_set_block_table", "mk_kv_pages_per_seq",
           "mk_kv_write", "mk_kv_read", "mk_decode_step", "mk_decode_step_unfused", "mk_decode_step_noalloc",
           "mk_step_status",
           "mk_debug_routing", "mk_debug_scratch_read", "mk_last_argmax", "mk_model_info", "mk_trace_read", "mk_free",
           "mk_last_error")
TRACE_CAP = 8192


def build_cmds() -> list:
    """nvcc commands for the library (the megakernel, its host side and the
    synthetic loader, which links the input generator module) and for a
    second build of the same sources with a 2-slot ring (MK_NSLOT=2)."""
    os.makedirs(_BUILD, exist_ok=True)
    srcs = [os.path.join(_HERE, "csrc", "mk_host.cu"), os.path.join(_HERE, "csrc", "mk_synth.cu"),
            os.path.join(_ROOT, "synth", "synth_cuda.cu"), os.path.join(_ROOT, "synth", "synth_host.c")]
    base = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC", "-shared", "-lpthread"]
    return [base + srcs + ["-o", os.path.join(_BUILD, "libmk.so")],
            base + ["-DMK_NSLOT=2"] + srcs + ["-o", LIB_NSLOT2]]


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "d_model", "vocab", "attn_kind", "n_q_heads", "n_kv_heads", "head_dim",
        "q_lora_rank", "kv_lora_rank", "qk_nope_dim", "qk_rope_dim", "v_head_dim",
        "n_routed_experts", "top_k", "n_shared_experts", "ffn_dim", "shared_ffn_dim",
        "max_batch", "max_tokens_per_seq", "max_ctx", "kv_page_size")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("expert_format", ctypes.c_int32)]


class Weight(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("layer", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("data", ctypes.c_void_p)]


class Info(ctypes.Structure):
    _fields_ = [("weight_bytes", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64)] + [
        (n, ctypes.c_int32) for n in ("grid_ctas", "threads_per_cta", "smem_bytes", "ring_slots", "slot_bytes",
                                      "sm_count")]


class MKError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"mk error {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """Load libmk.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        P, I32 = ctypes.c_void_p, ctypes.c_int32
        L.mk_load_weights.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weight), I32, P, ctypes.POINTER(P)]
        L.mk_load_synthetic.argtypes = [ctypes.POINTER(Config), ctypes.c_uint64, P, ctypes.POINTER(P)]
        L.mk_alloc_kv.argtypes = [P, I32, I32, ctypes.POINTER(P)]
        L.mk_kv_set_block_table.argtypes = [P, P]
        L.mk_kv_pages_per_seq.argtypes = [P]
        L.mk_kv_pages_per_seq.restype = I32
        L.mk_kv_write.argtypes = [P, I32, I32, I32, I32, P, P]
        L.mk_kv_read.argtypes = [P, I32, I32, I32, I32, P, P]
        L.mk_decode_step.argtypes = [P, P, P, P, I32, I32, P, P, P]
        L.mk_decode_step_noalloc.argtypes = [P, P, P, P, I32, I32, P, P, P]
        L.mk_decode_step_unfused.argtypes = [P, P, P, P, I32, I32, P, P, P]
        L.mk_step_status.argtypes = [P, P]
        L.mk_debug_routing.argtypes = [P, P, P, P, P]
        L.mk_debug_scratch_read.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P]
        L.mk_last_argmax.argtypes = [P, P, P]
        L.mk_model_info.argtypes = [P, ctypes.POINTER(Info)]
        L.mk_trace_read.argtypes = [P, P, ctypes.c_int64, P, P]
        L.mk_free.argtypes = [P]
        L.mk_free.restype = None
        L.mk_last_error.restype = ctypes.c_char_p
        for f in ("mk_load_weights", "mk_load_synthetic", "mk_alloc_kv", "mk_kv_set_block_table", "mk_kv_write",
                  "mk_kv_read", "mk_decode_step", "mk_decode_step_unfused", "mk_decode_step_noalloc", "mk_step_status",
                  "mk_debug_routing",
                  "mk_debug_scratch_read", "mk_last_argmax", "mk_model_info", "mk_trace_read"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc):
    if rc != OK:
        raise MKError(rc, lib().mk_last_error().decode())
    return rc


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def make_config(cfg, max_batch, max_tokens_per_seq, max_ctx) -> Config:
    vals = {f: int(cfg.get(f, 0)) for f, t in Config._fields_ if t is ctypes.c_int32}
    vals.update(max_batch=max_batch, max_tokens_per_seq=max_tokens_per_seq, max_ctx=max_ctx,
                kv_page_size=int(cfg.get("kv_page_size", 64)))
    return Config(**vals, rms_eps=float(cfg["rms_eps"]), rope_theta=float(cfg["rope_theta"]))


class Model:
    """A loaded model: mk_load_weights over a list of (kind, layer, expert, data_ptr)."""

    def __init__(self, config: Config, table=None, stream=None, seed=None):
        h = ctypes.c_void_p()
        self.config = config
        if table is None:
            # seeded synthetic weights generated on the device (mk_load_synthetic)
            _check(lib().mk_load_synthetic(ctypes.byref(config), int(seed), _stream(stream), ctypes.byref(h)))
        else:
            arr = (Weight * len(table))(*[Weight(k, l, e, 0, p) for (k, l, e, p) in table])
            _check(lib().mk_load_weights(ctypes.byref(config), arr, len(table), _stream(stream), ctypes.byref(h)))
        self.h = h

    @classmethod
    def synthetic(cls, config: Config, seed: int, stream=None) -> "Model":
        """mk_load_synthetic: the model of `config` with the generator's seeded weights."""
        return cls(config, None, stream, seed)

    def info(self) -> Info:
        out = Info()
        _check(lib().mk_model_info(self.h, ctypes.byref(out)))
        return out

    def decode_step(self, kv, tokens, positions, logits, accept=None, stream=None):
        """tokens int32 [B, T], positions int32 [B], logits float32 [B*T, V] (all CUDA tensors)."""
        B, T = tokens.shape
        _check(lib().mk_decode_step(self.h, kv.h, tokens.data_ptr(), positions.data_ptr(), B, T,
                                    logits.data_ptr(), None if accept is None else accept.data_ptr(),
                                    _stream(stream)))

    def decode_step_unfused(self, kv, tokens, positions, logits, accept=None, stream=None):
        """decode_step as one kernel launch per stage (replayed from a CUDA graph): the comparison path."""
        B, T = tokens.shape
        _check(lib().mk_decode_step_unfused(self.h, kv.h, tokens.data_ptr(), positions.data_ptr(), B, T,
                                            logits.data_ptr(), None if accept is None else accept.data_ptr(),
                                            _stream(stream)))

    def decode_step_noalloc(self, kv, tokens, positions, logits, accept=None, stream=None):
        """decode_step with the step's scratch in the library's static device
        array (nothing is allocated on the call path). For callers that may not
        allocate while they run. Synchronises the stream; raises on a device error."""
        B, T = tokens.shape
        _check(lib().mk_decode_step_noalloc(self.h, kv.h, tokens.data_ptr(), positions.data_ptr(), B, T,
                                            logits.data_ptr(), None if accept is None else accept.data_ptr(),
                                            _stream(stream)))

    def status(self, stream=None):
        return lib().mk_step_status(self.h, _stream(stream))

    def check(self, stream=None):
        _check(self.status(stream))

    def routing(self, M, stream=None):
        """Routing of the last step: idx [L, M, k], w [L, M, k], margin [L, M] (k-th minus (k+1)-th logit)."""
        import numpy as np
        L, k = self.config.n_layers, self.config.top_k
        idx = np.zeros((L, M, k), dtype=np.int32)
        w = np.zeros((L, M, k), dtype=np.float32)
        mg = np.zeros((L, M), dtype=np.float32)
        _check(lib().mk_debug_routing(self.h, idx.ctypes.data, w.ctypes.data, mg.ctypes.data, _stream(stream)))
        return idx, w, mg

    def scratch(self, offset=0, nbytes=None, stream=None):
        """Bytes [offset, offset + nbytes) of the model's own step scratch (numpy uint8)."""
        import numpy as np
        n = self.info().scratch_bytes - offset if nbytes is None else nbytes
        out = np.empty(n, dtype=np.uint8)
        _check(lib().mk_debug_scratch_read(self.h, offset, n, out.ctypes.data, _stream(stream)))
        return out

    def last_argmax(self, out, stream=None):
        """Argmax of every row of the last step that had an accept buffer, into
        `out` (int32 tensor of batch*T entries, host or device)."""
        _check(lib().mk_last_argmax(self.h, out.data_ptr(), _stream(stream)))
        return out

    def trace(self, stream=None):
        """Stage trace of the last step (needs MK_TRACE=1 at load): structured numpy array per record."""
        import numpy as np
        G = self.info().grid_ctas
        dt = np.dtype([("code", "<u4"), ("n", "<u4"), ("t_wait", "<i8"), ("t_ready", "<i8"), ("t_end", "<i8")])
        recs = np.zeros(G * TRACE_CAP, dtype=dt)
        counts = np.zeros(G, dtype=np.int32)
        _check(lib().mk_trace_read(self.h, recs.ctypes.data, recs.nbytes, counts.ctypes.data, _stream(stream)))
        recs = recs.reshape(G, TRACE_CAP)
        return [recs[g, :counts[g]] for g in range(G)]

    def close(self):
        if getattr(self, "h", None):
            lib().mk_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVCache:
    def __init__(self, model: Model, batch: int, max_ctx: int):
        h = ctypes.c_void_p()
        _check(lib().mk_alloc_kv(model.h, batch, max_ctx, ctypes.byref(h)))
        self.h = h
        self.model = model  # keep the model alive
        self.batch = batch
        self.max_ctx = max_ctx

    @property
    def pages_per_seq(self) -> int:
        return int(lib().mk_kv_pages_per_seq(self.h))

    def set_block_table(self, table):
        import numpy as np
        t = np.ascontiguousarray(table, dtype=np.int32)
        _check(lib().mk_kv_set_block_table(self.h, t.ctypes.data))

    def write(self, layer, seq, pos0, rows, stream=None):
        """rows: bf16 bits [n, row] (CUDA tensor or numpy uint16 array)."""
        ptr = rows.data_ptr() if hasattr(rows, "data_ptr") else rows.ctypes.data
        _check(lib().mk_kv_write(self.h, layer, seq, pos0, rows.shape[0], ptr, _stream(stream)))

    def read(self, layer, seq, pos0, n, stream=None):
        import numpy as np
        row = self.model.config.n_kv_heads * self.model.config.head_dim * 2 \
            if self.model.config.attn_kind == ATTN_GQA else \
            self.model.config.kv_lora_rank + self.model.config.qk_rope_dim
        out = np.empty((n, row), dtype=np.uint16)
        _check(lib().mk_kv_read(self.h, layer, seq, pos0, n, out.ctypes.data, _stream(stream)))
        return out

    def close(self):
        if getattr(self, "h", None):
            lib().mk_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
