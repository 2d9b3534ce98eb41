"""ctypes binding for libmk (include/mk.h): the same names, argument marshalling only.

Every step of the decode path runs in libmk's CUDA kernels; this module converts torch
tensors to device pointers and status codes to exceptions. It raises at import-time use if
the library is missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import platform

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", platform.machine(), "libmk.so")

MK_OK, MK_ERR_INVALID_ARG, MK_ERR_UNSUPPORTED, MK_ERR_CUDA, MK_ERR_OOM = 0, 1, 2, 3, 4
MK_ERR_NO_SCHEDULE, MK_ERR_BAD_PAGE, MK_ERR_DEVICE_TIMEOUT, MK_ERR_BAD_TOKEN = 5, 6, 7, 8
STATUS_NAMES = {0: "MK_OK", 1: "MK_ERR_INVALID_ARG", 2: "MK_ERR_UNSUPPORTED", 3: "MK_ERR_CUDA", 4: "MK_ERR_OOM",
                5: "MK_ERR_NO_SCHEDULE", 6: "MK_ERR_BAD_PAGE", 7: "MK_ERR_DEVICE_TIMEOUT", 8: "MK_ERR_BAD_TOKEN"}
MK_MODE_MEGAKERNEL, MK_MODE_PER_OP = 0, 1

EXPORTS = ["mk_create", "mk_plan_schedule", "mk_build_schedule", "mk_decode_step", "mk_decode_greedy", "mk_status_sync", "mk_last_error",
           "mk_set_mode", "mk_set_wait_limit", "mk_enable_trace", "mk_get_activations", "mk_get_launch_info", "mk_decode_step_noalloc", "mk_destroy"]


class mk_model_cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "n_experts",
                                                "top_k", "expert_inter", "vocab", "page_size", "max_batch",
                                                "max_pages_per_seq")] + [("rope_theta", ctypes.c_float),
                                                                         ("rms_eps", ctypes.c_float)]


class mk_weight_ptrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("embed", "norm_gain", "w_qkv", "w_o", "w_router", "router_bias",
                                                "w_gate_up", "w_down", "final_gain", "lm_head")]


class mk_kv_pages(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int32)]


class mk_activations(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "q", "attn", "attn_out", "moe_out", "router", "topk_ids",
                                                "topk_w")]


class mk_plan_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_tasks", "n_counters", "max_chunks", "n_lm_sm", "n_op_launches",
                                                       "n_attn_sm")]


class mk_trace_entry(ctypes.Structure):
    _fields_ = [("t_start_ns", ctypes.c_uint64), ("wait_ns", ctypes.c_uint32), ("run_ns", ctypes.c_uint32),
                ("sm", ctypes.c_uint16), ("op", ctypes.c_uint16), ("layer", ctypes.c_uint16), ("pad", ctypes.c_uint16),
                ("a", ctypes.c_int32), ("b", ctypes.c_int32)]


class MkError(RuntimeError):
    def __init__(self, status, msg=""):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")


_lib = None


def lib():
    """The loaded libmk. Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmk.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        L.mk_create.restype = ctypes.c_int
        L.mk_create.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.POINTER(mk_weight_ptrs), ctypes.POINTER(vp)]
        L.mk_plan_schedule.restype = ctypes.c_int
        L.mk_plan_schedule.argtypes = [ctypes.POINTER(mk_model_cfg), i32, i32, vp, ctypes.POINTER(mk_plan_info), vp,
                                       i32, vp, vp]
        L.mk_build_schedule.restype = ctypes.c_int
        L.mk_build_schedule.argtypes = [vp, i32, vp, vp]
        L.mk_decode_step.restype = ctypes.c_int
        L.mk_decode_step.argtypes = [vp, vp, vp, ctypes.POINTER(mk_kv_pages), vp, vp, vp]
        L.mk_decode_greedy.restype = ctypes.c_int
        L.mk_decode_greedy.argtypes = [vp, i32, vp, vp, ctypes.POINTER(mk_kv_pages), vp, vp, vp]
        L.mk_status_sync.restype = ctypes.c_int
        L.mk_status_sync.argtypes = [vp]
        L.mk_last_error.restype = ctypes.c_char_p
        L.mk_last_error.argtypes = [vp]
        L.mk_set_mode.restype = ctypes.c_int
        L.mk_set_mode.argtypes = [vp, ctypes.c_int]
        L.mk_set_wait_limit.restype = ctypes.c_int
        L.mk_set_wait_limit.argtypes = [vp, ctypes.c_int64]
        L.mk_enable_trace.restype = ctypes.c_int
        L.mk_enable_trace.argtypes = [vp, vp, ctypes.c_size_t]
        L.mk_get_activations.restype = ctypes.c_int
        L.mk_get_activations.argtypes = [vp, ctypes.POINTER(mk_activations)]
        L.mk_get_launch_info.restype = ctypes.c_int
        L.mk_get_launch_info.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.mk_decode_step_noalloc.restype = ctypes.c_int
        L.mk_decode_step_noalloc.argtypes = [ctypes.POINTER(mk_model_cfg), ctypes.POINTER(mk_weight_ptrs), i32, vp, vp,
                                             vp, vp, ctypes.POINTER(mk_kv_pages), vp, vp, vp, ctypes.c_char_p, i32]
        L.mk_destroy.restype = None
        L.mk_destroy.argtypes = [vp]
        _lib = L
    return _lib


def _check(ctx, status):
    if status != MK_OK:
        msg = lib().mk_last_error(ctx).decode() if ctx else ""
        raise MkError(status, msg)


def _ptr(t):
    return None if t is None else t.data_ptr()


def mk_create(cfg: mk_model_cfg, weights: mk_weight_ptrs):
    out = ctypes.c_void_p()
    _check(None, lib().mk_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(out)))
    return out


TASK_DTYPE = [("op", "u1"), ("flags", "u1"), ("layer", "<u2"), ("a", "<i4"), ("b", "<i4"), ("c", "<i4")]


def mk_plan_schedule(cfg: mk_model_cfg, n_sm: int, seq_lens):
    """Host-only plan: returns (info, tasks as a structured numpy array grouped by SM, sm_begin, sm_bytes)."""
    import numpy as np

    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    info = mk_plan_info()
    _check(None, lib().mk_plan_schedule(ctypes.byref(cfg), n_sm, len(sl), sl.ctypes.data, ctypes.byref(info), None, 0,
                                        None, None))
    tasks = np.zeros(info.n_tasks, dtype=np.dtype(TASK_DTYPE))
    begin = np.zeros(n_sm + 1, dtype=np.int32)
    load = np.zeros(n_sm, dtype=np.int64)
    _check(None, lib().mk_plan_schedule(ctypes.byref(cfg), n_sm, len(sl), sl.ctypes.data, ctypes.byref(info),
                                        tasks.ctypes.data, info.n_tasks, begin.ctypes.data, load.ctypes.data))
    return info, tasks, begin, load


def mk_build_schedule(ctx, batch: int, seq_lens, block_tables) -> None:
    """seq_lens: host int32 numpy array [batch]; block_tables: device int32 tensor [batch][max_pages]."""
    import numpy as np

    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    _check(ctx, lib().mk_build_schedule(ctx, batch, sl.ctypes.data, _ptr(block_tables)))


def mk_decode_step(ctx, token_ids, positions, kv: mk_kv_pages, logits_out=None, argmax_out=None, stream=None) -> None:
    _check(ctx, lib().mk_decode_step(ctx, _ptr(token_ids), _ptr(positions), ctypes.byref(kv), _ptr(logits_out),
                                     _ptr(argmax_out), stream))


def mk_decode_greedy(ctx, n_steps: int, token_ids, positions, kv: mk_kv_pages, logits_out, tokens_out,
                     stream=None) -> None:
    _check(ctx, lib().mk_decode_greedy(ctx, n_steps, _ptr(token_ids), _ptr(positions), ctypes.byref(kv),
                                       _ptr(logits_out), _ptr(tokens_out), stream))


def mk_status_sync(ctx) -> int:
    return lib().mk_status_sync(ctx)


def mk_last_error(ctx) -> str:
    return lib().mk_last_error(ctx).decode()


def mk_set_mode(ctx, mode: int) -> None:
    _check(ctx, lib().mk_set_mode(ctx, mode))


def mk_set_wait_limit(ctx, ns: int) -> None:
    _check(ctx, lib().mk_set_wait_limit(ctx, ns))


def mk_enable_trace(ctx, buf) -> None:
    _check(ctx, lib().mk_enable_trace(ctx, _ptr(buf), 0 if buf is None else buf.numel() * buf.element_size()))


def mk_get_activations(ctx) -> mk_activations:
    a = mk_activations()
    _check(ctx, lib().mk_get_activations(ctx, ctypes.byref(a)))
    return a


def mk_get_launch_info(ctx):
    n, t, l = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(ctx, lib().mk_get_launch_info(ctx, ctypes.byref(n), ctypes.byref(t), ctypes.byref(l)))
    return n.value, t.value, l.value


def mk_decode_step_noalloc(cfg: mk_model_cfg, weights: mk_weight_ptrs, seq_lens, block_tables, token_ids,
                           positions, kv: mk_kv_pages, logits_out=None, argmax_out=None, stream=None) -> None:
    """The decode step with its workspace in the library's static device array (no allocation)."""
    import numpy as np

    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    msg = ctypes.create_string_buffer(256)
    st = lib().mk_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(weights), len(sl), sl.ctypes.data,
                                      _ptr(block_tables), _ptr(token_ids), _ptr(positions), ctypes.byref(kv),
                                      _ptr(logits_out), _ptr(argmax_out), stream, msg, len(msg))
    if st != MK_OK:
        raise MkError(st, msg.value.decode())


def mk_destroy(ctx) -> None:
    lib().mk_destroy(ctx)
