"""The C ABI library without a GPU: it loads, exports every entry point include/mk.h declares,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from moe_transformer_decode_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:mk_status|void|const char\*)\s+(mk_\w+)\s*\(", src, re.M))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mk_create", "mk_build_schedule", "mk_decode_step", "mk_status_sync", "mk_last_error", "mk_set_mode",
              "mk_enable_trace", "mk_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    for n in declared_functions():
        assert hasattr(lib, n), f"libmk.so does not export {n}"
    assert set(B.EXPORTS) <= declared_functions()


def test_host_side_argument_errors():
    lib = B.lib()
    out = ctypes.c_void_p()
    assert lib.mk_create(None, None, ctypes.byref(out)) == B.MK_ERR_INVALID_ARG
    cfg = B.mk_model_cfg(2, 256, 4, 2, 64, 8, 2, 512, 1024, 16, 1, 8, 1e4, 1e-6)
    w = B.mk_weight_ptrs()
    assert lib.mk_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(out)) == B.MK_ERR_INVALID_ARG
    w = B.mk_weight_ptrs(*([0x1000] * 5 + [None] + [0x1000] * 4))
    bad = B.mk_model_cfg(2, 300, 4, 2, 64, 8, 2, 512, 1024, 16, 1, 8, 1e4, 1e-6)  # hidden 300
    assert lib.mk_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(out)) == B.MK_ERR_UNSUPPORTED
    bad = B.mk_model_cfg(2, 256, 4, 2, 64, 8, 9, 512, 1024, 16, 1, 8, 1e4, 1e-6)  # top_k > experts
    assert lib.mk_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(out)) == B.MK_ERR_INVALID_ARG
    bad = B.mk_model_cfg(2, 256, 4, 2, 64, 8, 2, 512, 1024, 32, 1, 8, 1e4, 1e-6)  # page size 32
    assert lib.mk_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(out)) == B.MK_ERR_UNSUPPORTED
    # each shape limit the header states is rejected before any device work
    for fields, why in (((2, 256, 4, 2, 64, 264, 2, 512, 1024, 16, 1, 8), "n_experts > 256"),
                        ((2, 256, 4, 2, 64, 12, 2, 512, 1024, 16, 1, 8), "n_experts not a multiple of 8"),
                        ((2, 256, 4, 2, 64, 8, 2, 512, 1000, 16, 1, 8), "vocab not a multiple of 64"),
                        ((2, 256, 4, 2, 96, 8, 2, 512, 1024, 16, 1, 8), "head_dim 96"),
                        ((2, 256, 18, 2, 64, 8, 2, 512, 1024, 16, 1, 8), "9 query heads per KV head"),
                        ((2, 256, 4, 2, 64, 8, 2, 320, 1024, 16, 1, 8), "expert_inter not a multiple of 256"),
                        ((2, 256, 4, 2, 64, 8, 2, 2048, 1024, 16, 8, 8), "activations of batch 8 at 2048 > a stage"),
                        ((2, 256, 4, 2, 64, 8, 2, 512, 1024, 16, 9, 8), "max_batch 9")):
        bad = B.mk_model_cfg(*fields, 1e4, 1e-6)
        assert lib.mk_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(out)) == B.MK_ERR_UNSUPPORTED, why
    w2 = B.mk_weight_ptrs(*([0x1008] * 5 + [None] + [0x1000] * 4))  # misaligned
    assert lib.mk_create(ctypes.byref(cfg), ctypes.byref(w2), ctypes.byref(out)) == B.MK_ERR_INVALID_ARG
    assert lib.mk_build_schedule(None, 1, None, None) == B.MK_ERR_INVALID_ARG
    kv = B.mk_kv_pages()
    assert lib.mk_decode_step(None, None, None, ctypes.byref(kv), None, None, None) == B.MK_ERR_INVALID_ARG
    assert lib.mk_decode_greedy(None, 1, None, None, ctypes.byref(kv), None, None, None) == B.MK_ERR_INVALID_ARG
    assert lib.mk_status_sync(None) == B.MK_ERR_INVALID_ARG
    assert lib.mk_set_mode(None, 0) == B.MK_ERR_INVALID_ARG
    assert lib.mk_enable_trace(None, None, 0) == B.MK_ERR_INVALID_ARG
    assert lib.mk_last_error(None) == b"null context"
    lib.mk_destroy(None)


def test_binding_raises_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()
