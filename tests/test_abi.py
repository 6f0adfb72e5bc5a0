"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/mk.h declares, keeps its enums in step with the generator's tensor
kinds, and rejects bad arguments with status codes instead of crashing."""
import ctypes
import re

import pytest

import moe_decode_megakernel_02_gb300 as mk
import synth
from synth import configs
from conftest import have_gpu


def declared_functions():
    src = open(mk.HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in mk.EXPORTS:
        assert n in names
    assert set(names) == set(mk.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = mk.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"{n} not exported"


def test_weight_kinds_match_generator():
    src = open(mk.HEADER).read()
    kinds = dict((k, int(v)) for k, v in re.findall(r"MK_W_([A-Z_]+) = (\d+)", src))
    for name, val in kinds.items():
        assert getattr(synth, name) == val, name


def test_null_arguments_are_rejected():
    L = mk.lib()
    out = ctypes.c_void_p()
    assert L.mk_load_weights(None, None, 0, None, ctypes.byref(out)) == mk.ERR_INVALID_ARG
    assert b"NULL" in L.mk_last_error()
    assert L.mk_alloc_kv(None, 1, 16, ctypes.byref(out)) == mk.ERR_INVALID_ARG
    assert L.mk_decode_step(None, None, None, None, 1, 1, None, None, None) == mk.ERR_INVALID_ARG
    assert L.mk_step_status(None, None) == mk.ERR_INVALID_ARG
    assert L.mk_last_argmax(None, None, None) == mk.ERR_INVALID_ARG
    L.mk_free(None)


def _bad(cfg, **over):
    c = mk.make_config(dict(cfg, **over), 1, 1, 128)
    out = ctypes.c_void_p()
    w = (mk.Weight * 1)(mk.Weight(1, -1, 0, 0, 1))
    return mk.lib().mk_load_weights(ctypes.byref(c), w, 1, None, ctypes.byref(out))


def test_unsupported_shapes_are_reported():
    assert _bad(configs.TINY, kv_page_size=32) == mk.ERR_UNSUPPORTED
    assert _bad(configs.TINY, head_dim=96) == mk.ERR_UNSUPPORTED
    assert _bad(configs.DEEP, n_q_heads=8) == mk.ERR_UNSUPPORTED
    assert _bad(configs.TINY, top_k=9) == mk.ERR_UNSUPPORTED
    assert _bad(configs.TINY, n_q_heads=3) == mk.ERR_INVALID_ARG
    assert _bad(configs.TINY, d_model=0) == mk.ERR_INVALID_ARG


def test_missing_and_duplicate_tensors_are_reported():
    c = mk.make_config(configs.TINY, 1, 1, 128)
    out = ctypes.c_void_p()
    dup = (mk.Weight * 2)(mk.Weight(1, -1, 0, 0, 8), mk.Weight(1, -1, 0, 0, 8))
    assert mk.lib().mk_load_weights(ctypes.byref(c), dup, 2, None, ctypes.byref(out)) == mk.ERR_INVALID_ARG
    assert b"duplicate" in mk.lib().mk_last_error()


@pytest.mark.skipif(have_gpu(), reason="checks the no-GPU error path")
def test_no_device_gives_cuda_error_not_crash():
    assert _bad(configs.TINY) in (mk.ERR_CUDA, mk.ERR_INVALID_ARG)


@pytest.mark.parametrize("fault,code", [("oom", mk.ERR_OOM), ("bad_arg", mk.ERR_INVALID_ARG)])
def test_injected_host_faults_are_reported(monkeypatch, fault, code):
    # MK_FAULT makes the library report the failure before it touches the
    # device, so the caller's error handling can be exercised anywhere
    monkeypatch.setenv("MK_FAULT", fault)
    c = mk.make_config(configs.TINY, 1, 1, 128)
    out = ctypes.c_void_p()
    w = (mk.Weight * 1)(mk.Weight(1, -1, 0, 0, 8))
    assert mk.lib().mk_load_weights(ctypes.byref(c), w, 1, None, ctypes.byref(out)) == code
    assert b"MK_FAULT=" + fault.encode() in mk.lib().mk_last_error()
    assert not out.value
    if fault == "oom":
        assert mk.lib().mk_load_synthetic(ctypes.byref(c), 0, None, ctypes.byref(out)) == mk.ERR_OOM
        assert b"MK_FAULT=oom" in mk.lib().mk_last_error()
    monkeypatch.delenv("MK_FAULT")
    assert mk.lib().mk_load_weights(ctypes.byref(c), w, 1, None, ctypes.byref(out)) != code or code != mk.ERR_OOM


def test_debug_entry_points_reject_bad_handles():
    L = mk.lib()
    assert L.mk_load_synthetic(None, 0, None, None) == mk.ERR_INVALID_ARG
    assert L.mk_debug_routing(None, None, None, None, None) == mk.ERR_INVALID_ARG
    assert L.mk_debug_scratch_read(None, 0, 0, None, None) == mk.ERR_INVALID_ARG
    assert L.mk_decode_step_noalloc(None, None, None, None, 1, 1, None, None, None) == mk.ERR_INVALID_ARG


def test_mxfp8_expert_shapes_are_checked():
    # MXFP8 experts: d_model 512 / 1024 / 2048; an unknown format is an
    # argument error (both found before any device call)
    mx = dict(expert_format=1)
    assert _bad(configs.TINY, **mx) == mk.ERR_UNSUPPORTED  # d_model 256
    assert b"MXFP8" in mk.lib().mk_last_error()
    assert _bad(configs.DENSE, **mx) == mk.ERR_UNSUPPORTED  # d_model 5120
    assert _bad(configs.DEEP, expert_format=2) == mk.ERR_INVALID_ARG
