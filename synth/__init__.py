"""Seeded synthetic inputs shared by the checker and the benchmark (see synth.h).

Only numbers are made here: SplitMix64 streams, Irwin-Hall(12) normals rounded to bf16,
uniform integers and permutations. The decode step's arithmetic lives elsewhere.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

SYNTH_EMBED, SYNTH_GAIN, SYNTH_FINAL_GAIN, SYNTH_QKV, SYNTH_O, SYNTH_ROUTER = 1, 2, 3, 4, 5, 6
SYNTH_GATE_UP, SYNTH_DOWN, SYNTH_LM, SYNTH_K, SYNTH_V = 7, 8, 9, 10, 11
SYNTH_TOKENS, SYNTH_CTX, SYNTH_PAGES, SYNTH_ZIPF = 12, 13, 14, 15

WEIGHT_SIGMA = 0.02
GAIN_SIGMA = 0.05

_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(_build.build_host())
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        lib.synth_tid.restype = u64
        lib.synth_tid.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.synth_key.restype = u64
        lib.synth_key.argtypes = [u64, u64]
        lib.synth_draw.restype = u64
        lib.synth_draw.argtypes = [u64, u64]
        lib.synth_normal.restype = ctypes.c_float
        lib.synth_normal.argtypes = [u64, u64]
        lib.synth_bf16.restype = ctypes.c_uint16
        lib.synth_bf16.argtypes = [ctypes.c_float]
        lib.synth_fill_bf16.restype = None
        lib.synth_fill_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
        lib.synth_fill_uniform_int.restype = None
        lib.synth_fill_uniform_int.argtypes = [u64, u64, u64, u64, i64, i64, ctypes.c_void_p]
        lib.synth_permutation.restype = None
        lib.synth_permutation.argtypes = [u64, u64, i64, ctypes.c_void_p]
        _host = lib
    return _host


def dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(_build.build_device())
        lib.synth_dev_fill_stack.restype = ctypes.c_int
        lib.synth_dev_fill_stack.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_uint64, ctypes.c_float, ctypes.c_float, ctypes.c_void_p,
                                             ctypes.c_void_p]
        lib.synth_dev_fill_kv.restype = ctypes.c_int
        lib.synth_dev_fill_kv.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        _dev = lib
    return _dev


def tid(kind: int, layer: int, sub: int) -> int:
    return host_lib().synth_tid(kind, layer, sub)


def fill_bf16(seed: int, kind: int, layer: int, sub: int, count: int, sigma: float, offset: float = 0.0,
              start: int = 0) -> np.ndarray:
    """bf16 bits (uint16) of `count` elements of stream tid(kind, layer, sub) from `start`."""
    out = np.empty(count, dtype=np.uint16)
    host_lib().synth_fill_bf16(seed, tid(kind, layer, sub), start, count, sigma, offset, out.ctypes.data)
    return out


def uniform_int(seed: int, t: int, start: int, count: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(count, dtype=np.int64)
    host_lib().synth_fill_uniform_int(seed, t, start, count, lo, hi, out.ctypes.data)
    return out


def permutation(seed: int, t: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    host_lib().synth_permutation(seed, t, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- host model (small configs)

def host_model(w) -> dict:
    """Whole model as numpy bf16 bits in the decode library's layouts (small configs only)."""
    s = w.seed
    qkv_rows, od = w.qkv_rows, w.nq * w.d
    stack = lambda kind, rows, cols: np.stack([fill_bf16(s, kind, l, 0, rows * cols, WEIGHT_SIGMA)
                                               for l in range(w.L)]).reshape(w.L, rows, cols)
    experts = lambda kind, rows, cols: np.stack([
        np.stack([fill_bf16(s, kind, l, e, rows * cols, WEIGHT_SIGMA) for e in range(w.E)])
        for l in range(w.L)]).reshape(w.L, w.E, rows, cols)
    return {
        "embed": fill_bf16(s, SYNTH_EMBED, 0, 0, w.V * w.H, WEIGHT_SIGMA).reshape(w.V, w.H),
        "norm_gain": np.stack([fill_bf16(s, SYNTH_GAIN, l, 0, w.H, GAIN_SIGMA, 1.0) for l in range(w.L)]),
        "w_qkv": stack(SYNTH_QKV, qkv_rows, w.H),
        "w_o": stack(SYNTH_O, w.H, od),
        "w_router": stack(SYNTH_ROUTER, w.E, w.H),
        "w_gate_up": experts(SYNTH_GATE_UP, 2 * w.I, w.H),
        "w_down": experts(SYNTH_DOWN, w.H, w.I),
        "final_gain": fill_bf16(s, SYNTH_FINAL_GAIN, 0, 0, w.H, GAIN_SIGMA, 1.0),
        "lm_head": fill_bf16(s, SYNTH_LM, 0, 0, w.V * w.H, WEIGHT_SIGMA).reshape(w.V, w.H),
    }


def host_kv(w, ctx, block_table, num_pages):
    """Paged K and V pools [L][num_pages][nkv][page][d] (bf16 bits) prefilled to ctx[b]."""
    K = np.zeros((w.L, num_pages, w.nkv, w.page, w.d), dtype=np.uint16)
    V = np.zeros_like(K)
    for pool, kind in ((K, SYNTH_K), (V, SYNTH_V)):
        for l in range(w.L):
            for b in range(w.B):
                for g in range(w.nkv):
                    vals = fill_bf16(w.seed, kind, l, b * w.nkv + g, int(ctx[b]) * w.d, 1.0).reshape(-1, w.d)
                    for pos in range(int(ctx[b])):
                        pool[l, block_table[b, pos // w.page], g, pos % w.page] = vals[pos]
    return K, V


# ---------------------------------------------------------------- device model

def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def device_model(w, device="cuda") -> dict:
    """Whole model as torch bf16 tensors on `device`, generated there (same values as host_model)."""
    import torch

    s, lib = w.seed, dev_lib()
    stream = torch.cuda.current_stream(device).cuda_stream
    qkv_rows, od = w.qkv_rows, w.nq * w.d

    def make(shape, kind, n_layer, n_sub, sigma, offset=0.0):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        inner = t.numel() // (n_layer * n_sub)
        _check(lib.synth_dev_fill_stack(s, kind, 0, n_layer, n_sub, inner, sigma, offset, t.data_ptr(), stream),
               "synth_dev_fill_stack")
        return t

    m = {
        "embed": make((w.V, w.H), SYNTH_EMBED, 1, 1, WEIGHT_SIGMA),
        "norm_gain": make((w.L, w.H), SYNTH_GAIN, w.L, 1, GAIN_SIGMA, 1.0),
        "w_qkv": make((w.L, qkv_rows, w.H), SYNTH_QKV, w.L, 1, WEIGHT_SIGMA),
        "w_o": make((w.L, w.H, od), SYNTH_O, w.L, 1, WEIGHT_SIGMA),
        "w_router": make((w.L, w.E, w.H), SYNTH_ROUTER, w.L, 1, WEIGHT_SIGMA),
        "w_gate_up": make((w.L, w.E, 2 * w.I, w.H), SYNTH_GATE_UP, w.L, w.E, WEIGHT_SIGMA),
        "w_down": make((w.L, w.E, w.H, w.I), SYNTH_DOWN, w.L, w.E, WEIGHT_SIGMA),
        "final_gain": make((w.H,), SYNTH_FINAL_GAIN, 1, 1, GAIN_SIGMA, 1.0),
        "lm_head": make((w.V, w.H), SYNTH_LM, 1, 1, WEIGHT_SIGMA),
    }
    torch.cuda.synchronize(device)
    return m


def device_kv(w, ctx, block_table, num_pages, device="cuda"):
    """Paged K and V pools on `device` [L][num_pages][nkv][page][d] bf16, prefilled to ctx[b]."""
    import torch

    if int(np.max(ctx)) > block_table.shape[1] * w.page:
        raise ValueError("context longer than the block table")
    lib = dev_lib()
    stream = torch.cuda.current_stream(device).cuda_stream
    ctx_d = torch.as_tensor(np.asarray(ctx, dtype=np.int32), device=device)
    bt_d = torch.as_tensor(np.ascontiguousarray(block_table, dtype=np.int32), device=device)
    pools = []
    for kind in (SYNTH_K, SYNTH_V):
        pool = torch.zeros((w.L, num_pages, w.nkv, w.page, w.d), dtype=torch.bfloat16, device=device)
        _check(lib.synth_dev_fill_kv(w.seed, kind, w.L, w.B, w.nkv, w.d, w.page, ctx_d.data_ptr(), int(np.max(ctx)),
                                     bt_d.data_ptr(), block_table.shape[1], num_pages, pool.data_ptr(), stream),
               "synth_dev_fill_kv")
        pools.append(pool)
    torch.cuda.synchronize(device)
    return pools[0], pools[1]
