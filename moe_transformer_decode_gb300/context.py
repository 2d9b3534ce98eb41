"""Convenience wrapper around the C ABI for callers holding torch tensors.

Argument marshalling only: shapes are checked, pointers passed to libmk, and the
library-owned activations exposed as zero-copy torch views. No arithmetic of the decode
step happens here.
"""
from __future__ import annotations

import numpy as np

from . import binding as B


class _CudaArray:
    """Minimal __cuda_array_interface__ exporter for a raw device pointer."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 3, "strides": None}


def _view(ptr, shape, typestr, device):
    import torch

    return torch.as_tensor(_CudaArray(ptr, shape, typestr), device=device)


class DecodeContext:
    """Holds an mk_ctx for one model. `shape` needs attributes L, H, nq, nkv, d, E, topk, I, V,
    rope_theta, eps; `weights` maps the mk_weight_ptrs field names to CUDA tensors (bf16, router
    bias fp32 or absent)."""

    def __init__(self, shape, weights: dict, max_batch: int, max_pages_per_seq: int):
        import torch

        self.shape = shape
        self.weights = weights  # keep alive
        self.device = weights["embed"].device
        cfg = B.mk_model_cfg(shape.L, shape.H, shape.nq, shape.nkv, shape.d, shape.E, shape.topk, shape.I, shape.V,
                             16, max_batch, max_pages_per_seq, float(shape.rope_theta), float(shape.eps))
        for k, t in weights.items():
            if t is None:
                continue
            want = torch.float32 if k == "router_bias" else torch.bfloat16
            if t.dtype != want or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"weight {k}: expected contiguous CUDA {want}")
        ptrs = B.mk_weight_ptrs(**{k: (None if weights.get(k) is None else weights[k].data_ptr())
                                   for k, _ in B.mk_weight_ptrs._fields_})
        self.ctx = B.mk_create(cfg, ptrs)
        self.max_pages_per_seq = max_pages_per_seq
        self.batch = 0

    def close(self):
        if getattr(self, "ctx", None):
            B.mk_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        self.close()

    def schedule(self, seq_lens, block_tables):
        seq_lens = np.asarray(seq_lens, dtype=np.int32)
        if block_tables.dtype.__str__() != "torch.int32" or block_tables.shape[1] != self.max_pages_per_seq:
            raise ValueError("block_tables must be int32 [batch][max_pages_per_seq]")
        self.block_tables = block_tables
        B.mk_build_schedule(self.ctx, len(seq_lens), seq_lens, block_tables)
        self.batch = len(seq_lens)

    @staticmethod
    def kv_pages(K, V):
        return B.mk_kv_pages(K.data_ptr(), V.data_ptr(), K.shape[1])

    def step(self, tokens, positions, K, V, logits=None, argmax=None, stream=None):
        kv = self.kv_pages(K, V)
        B.mk_decode_step(self.ctx, tokens, positions, kv, logits, argmax, stream)

    def greedy(self, n_steps, tokens, positions, K, V, logits, tokens_out, stream=None):
        B.mk_decode_greedy(self.ctx, n_steps, tokens, positions, self.kv_pages(K, V), logits, tokens_out, stream)

    def sync(self):
        st = B.mk_status_sync(self.ctx)
        if st != B.MK_OK:
            raise B.MkError(st, B.mk_last_error(self.ctx))

    def set_mode(self, mode):
        B.mk_set_mode(self.ctx, mode)

    def set_wait_limit(self, ns: int):
        B.mk_set_wait_limit(self.ctx, int(ns))

    def launch_info(self):
        return B.mk_get_launch_info(self.ctx)

    def activations(self) -> dict:
        """Zero-copy views of the library-owned per-layer activations of the last step."""
        s, b = self.shape, self.batch
        a = B.mk_get_activations(self.ctx)
        f4, i4 = "<f4", "<i4"
        return {
            "x": _view(a.x, (s.L + 1, b, s.H), f4, self.device),
            "q": _view(a.q, (s.L, b, s.nq, s.d), f4, self.device),
            "attn": _view(a.attn, (s.L, b, s.nq, s.d), f4, self.device),
            "attn_out": _view(a.attn_out, (s.L, b, s.H), f4, self.device),
            "moe_out": _view(a.moe_out, (s.L, b, s.H), f4, self.device),
            "router": _view(a.router, (s.L, b, s.E), f4, self.device),
            "topk_ids": _view(a.topk_ids, (s.L, b, s.topk), i4, self.device),
            "topk_w": _view(a.topk_w, (s.L, b, s.topk), f4, self.device),
        }
