"""CPU oracle for the parallel-layer MoE decode step (ctypes over oracle/_lib/liboracle.so).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline
leg use it. The decode library never imports it and shares no code with it.
What each function computes, and which passage of the Cohere megakernel news pages
it follows, is documented in oracle.h / oracle.c.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

ORC_EMBED, ORC_GAIN, ORC_FINAL_GAIN, ORC_QKV, ORC_O, ORC_ROUTER, ORC_GATE_UP, ORC_DOWN, ORC_LM = range(1, 10)


class OrcCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("L", "H", "nq", "nkv", "d", "E", "topk", "I", "V")] + [
        ("rope_theta", ctypes.c_double), ("eps", ctypes.c_double)]


WEIGHT_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int)
BIAS_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int)
KV_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                         ctypes.c_int, ctypes.c_void_p)
FETCH_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int)


class OrcSource(ctypes.Structure):
    _fields_ = [("ctx", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("kv_read", ctypes.c_void_p), ("kv_write", ctypes.c_void_p)]


class OrcTrace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "q", "k_new", "v_new", "attn", "attn_out", "router",
                                                "topk_ids", "topk_w", "moe_out")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build.build())
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_double
        L.orc_threads.restype = ctypes.c_int
        L.orc_threads.argtypes = []
        L.orc_decode_step.restype = ctypes.c_int
        L.orc_decode_step.argtypes = [ctypes.POINTER(OrcCfg), ctypes.POINTER(OrcSource), ctypes.c_int, vp, vp, vp, vp,
                                      ctypes.POINTER(OrcTrace)]
        L.orc_bf16_to_double.restype = dbl
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_double_to_bf16.restype = ctypes.c_uint16
        L.orc_double_to_bf16.argtypes = [dbl]
        L.orc_matvec.restype = None
        L.orc_matvec.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_rmsnorm.restype = None
        L.orc_rmsnorm.argtypes = [vp, vp, ctypes.c_int, dbl, vp]
        L.orc_rope.restype = None
        L.orc_rope.argtypes = [vp, ctypes.c_int, ctypes.c_int, dbl]
        L.orc_attention_head.restype = None
        L.orc_attention_head.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, vp]
        L.orc_route.restype = None
        L.orc_route.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_expert.restype = None
        L.orc_expert.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_moe.restype = None
        L.orc_moe.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, FETCH_FN, vp, vp, vp,
                              vp, vp]
        L.orc_dense_source_create.restype = vp
        L.orc_dense_source_create.argtypes = [ctypes.POINTER(OrcCfg)] + [vp] * 13 + [i32] * 5 + [ctypes.POINTER(OrcSource)]
        L.orc_dense_source_destroy.restype = None
        L.orc_dense_source_destroy.argtypes = [vp]
        L.orc_synth_source_create.restype = vp
        L.orc_synth_source_create.argtypes = [ctypes.POINTER(OrcCfg), ctypes.c_uint64, i32, vp, i32, vp, i32,
                                              ctypes.POINTER(OrcSource)]
        L.orc_synth_source_destroy.restype = None
        L.orc_synth_source_destroy.argtypes = [vp]
        _lib = L
    return _lib


def cfg_of(w) -> OrcCfg:
    return OrcCfg(w.L, w.H, w.nq, w.nkv, w.d, w.E, w.topk, w.I, w.V, w.rope_theta, w.eps)


def _p(a):
    return None if a is None else a.ctypes.data


def _u16(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint16)


class DenseSource:
    """Host arrays in the decode library's layouts. With block_table=None the KV arrays are
    contiguous [L][B][nkv][max_len][d]. KV arrays are written in place by decode steps."""

    def __init__(self, w, model: dict, K: np.ndarray, V: np.ndarray, block_table=None, bias=None):
        self.cfg = cfg_of(w)
        self.keep = {k: _u16(v) for k, v in model.items()}
        assert K.dtype == np.uint16 and K.flags.c_contiguous and V.flags.c_contiguous
        self.K, self.V = K, V
        self.bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self.bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
        self.src = OrcSource()
        m = self.keep
        if self.bt is not None:
            B, max_pages = self.bt.shape
            num_pages, page, max_len = K.shape[1], K.shape[3], 0
        else:
            B, max_len = K.shape[1], K.shape[3]
            max_pages, num_pages, page = 0, 0, 0
        self.h = lib().orc_dense_source_create(
            ctypes.byref(self.cfg), _p(m["embed"]), _p(m["norm_gain"]), _p(m["final_gain"]), _p(m["w_qkv"]),
            _p(m["w_o"]), _p(m["w_router"]), _p(self.bias), _p(m["w_gate_up"]), _p(m["w_down"]), _p(m["lm_head"]),
            _p(K), _p(V), _p(self.bt), B, max_pages, page, num_pages, max_len, ctypes.byref(self.src))

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_dense_source_destroy(self.h)
            self.h = None


class SynthSource:
    """The seeded model and prefilled cache, generated on demand (any size)."""

    def __init__(self, w, ctx, max_new: int, bias=None, keep_all_experts: bool = False):
        self.cfg = cfg_of(w)
        self.ctx = np.ascontiguousarray(ctx, dtype=np.int32)
        self.bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self.src = OrcSource()
        self.h = lib().orc_synth_source_create(ctypes.byref(self.cfg), w.seed, w.B, _p(self.ctx), max_new,
                                               _p(self.bias), int(keep_all_experts), ctypes.byref(self.src))

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_synth_source_destroy(self.h)
            self.h = None


def threads() -> int:
    """Host threads the oracle's parallel loops use."""
    return int(lib().orc_threads())


def decode_step(w, source, tokens, positions, trace: bool = False):
    """One oracle decode step. Returns (logits [B][V] fp32, next [B] int32, trace dict or None)."""
    B = len(tokens)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    logits = np.empty((B, w.V), dtype=np.float32)
    nxt = np.empty(B, dtype=np.int32)
    tr = None
    trs = None
    if trace:
        tr = {
            "x": np.zeros((w.L + 1, B, w.H), np.float32), "q": np.zeros((w.L, B, w.nq, w.d), np.float32),
            "k_new": np.zeros((w.L, B, w.nkv, w.d), np.uint16), "v_new": np.zeros((w.L, B, w.nkv, w.d), np.uint16),
            "attn": np.zeros((w.L, B, w.nq, w.d), np.float32), "attn_out": np.zeros((w.L, B, w.H), np.float32),
            "router": np.zeros((w.L, B, w.E), np.float32), "topk_ids": np.zeros((w.L, B, w.topk), np.int32),
            "topk_w": np.zeros((w.L, B, w.topk), np.float32), "moe_out": np.zeros((w.L, B, w.H), np.float32),
        }
        trs = OrcTrace(*[tr[n].ctypes.data for n, _ in OrcTrace._fields_])
    rc = lib().orc_decode_step(ctypes.byref(source.cfg), ctypes.byref(source.src), B, tok.ctypes.data,
                               pos.ctypes.data, logits.ctypes.data, nxt.ctypes.data,
                               ctypes.byref(trs) if trs is not None else None)
    if rc != 0:
        raise RuntimeError(f"orc_decode_step failed with status {rc}")
    return logits, nxt, tr


# ---------------------------------------------------------------- the step's parts

def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def rmsnorm(x, gain_bits, eps):
    x = _f64(x)
    g = _u16(gain_bits)
    out = np.empty_like(x)
    lib().orc_rmsnorm(x.ctypes.data, g.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def rope(v, pos, theta):
    v = _f64(v).copy()
    lib().orc_rope(v.ctypes.data, v.size, pos, theta)
    return v


def attention_head(q, K_bits, V_bits):
    q = _f64(q)
    K, V = _u16(K_bits), _u16(V_bits)
    out = np.empty(q.size, dtype=np.float64)
    lib().orc_attention_head(q.ctypes.data, K.ctypes.data, V.ctypes.data, K.shape[0], q.size, out.ctypes.data)
    return out


def route(logits, k):
    lg = _f64(logits)
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    lib().orc_route(lg.ctypes.data, lg.size, k, ids.ctypes.data, w.ctypes.data)
    return ids, w


def expert(Wgu_bits, Wd_bits, x):
    Wgu, Wd, x = _u16(Wgu_bits), _u16(Wd_bits), _f64(x)
    H, I = Wd.shape
    y = np.empty(H, dtype=np.float64)
    lib().orc_expert(Wgu.ctypes.data, Wd.ctypes.data, H, I, x.ctypes.data, y.ctypes.data)
    return y


def moe(x, Wr_bits, bias, Wgu_bits, Wd_bits, k):
    """Wgu_bits [E][2I][H], Wd_bits [E][H][I]; returns (y, logits, ids, w)."""
    x, Wr = _f64(x), _u16(Wr_bits)
    Wgu, Wd = _u16(Wgu_bits), _u16(Wd_bits)
    E, H, I = Wd.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)

    @FETCH_FN
    def fetch(_ctx, e, which):
        return (Wd if which else Wgu)[e].ctypes.data

    y = np.empty(H, dtype=np.float64)
    lg = np.empty(E, dtype=np.float64)
    ids = np.empty(k, dtype=np.int32)
    w = np.empty(k, dtype=np.float64)
    lib().orc_moe(x.ctypes.data, Wr.ctypes.data, _p(b), H, I, E, k, fetch, None, y.ctypes.data, lg.ctypes.data,
                  ids.ctypes.data, w.ctypes.data)
    return y, lg, ids, w


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v):
    v = np.asarray(v, dtype=np.float64)
    return np.array([lib().orc_double_to_bf16(float(x)) for x in v.ravel()], dtype=np.uint16).reshape(v.shape)
