"""Synthetic workloads: model shapes, seeds and input recipes.

Shapes and recipes follow the five decode workloads this library is measured on: a tiny
and a small parallel-layer MoE decoder, and a 30B-total / 3.3B-active-shaped model
(48 layers, hidden 2048, 32/4 heads of 128, 128 experts top-8 with intermediate 768,
vocab 151552) at batch 1 with 8K context, batch 8 with 1K-8K contexts (uniform or
Zipf(1.2)-skewed routing) and batch 1 with 256K context. The pages describing the
original system give only "30B total, 3.3B active", BF16, 8K context and 1K output
tokens; every dimension here is a chosen stand-in, and all values are seeded draws.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import SYNTH_CTX, SYNTH_PAGES, SYNTH_TOKENS, SYNTH_ZIPF, permutation, tid, uniform_int


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    H: int
    nq: int
    nkv: int
    d: int
    E: int
    topk: int
    I: int
    V: int
    B: int
    ctx_lo: int
    ctx_hi: int
    steps: int
    seed: int
    routing: str = "uniform"  # or "zipf"
    rope_theta: float = 1e4
    eps: float = 1e-6
    page: int = 16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def qkv_rows(self) -> int:
        return (self.nq + 2 * self.nkv) * self.d

    def weight_bytes(self) -> int:
        per_layer = (self.qkv_rows * self.H + self.H * self.nq * self.d + self.E * self.H
                     + self.E * 3 * self.I * self.H + self.H)
        return 2 * (self.L * per_layer + 2 * self.V * self.H + self.H)

    def kv_bytes(self, total_positions: int) -> int:
        return 2 * 2 * self.L * self.nkv * self.d * total_positions


TINY = Workload("tiny", L=2, H=256, nq=4, nkv=2, d=64, E=8, topk=2, I=512, V=1024, B=1, ctx_lo=32,
                ctx_hi=32, steps=1, seed=0)
SMALL = Workload("small_bs8_ragged", L=4, H=1024, nq=16, nkv=4, d=64, E=32, topk=4, I=512, V=8192, B=8,
                 ctx_lo=64, ctx_hi=2048, steps=128, seed=1)
M30B_BS1 = Workload("moe30b_a3b_bs1_ctx8k", L=48, H=2048, nq=32, nkv=4, d=128, E=128, topk=8, I=768,
                    V=151552, B=1, ctx_lo=8192, ctx_hi=8192, steps=1024, seed=2)
M30B_BS8 = M30B_BS1.with_(name="moe30b_a3b_bs8_ctx1k8k", B=8, ctx_lo=1024, ctx_hi=8192, seed=3)
M30B_BS8_ZIPF = M30B_BS8.with_(name="moe30b_a3b_bs8_ctx1k8k_zipf", routing="zipf")
M30B_256K = M30B_BS1.with_(name="moe30b_a3b_bs1_ctx256k", ctx_lo=262144, ctx_hi=262144, steps=256, seed=4)
# the 30B-shaped layer and LM head with 4 layers: small enough (~1.8 GB) for profiler captures
M30B_L4 = M30B_BS1.with_(name="moe30b_shape_l4_bs1_ctx8k", L=4)

ALL = {w.name: w for w in (TINY, SMALL, M30B_BS1, M30B_BS8, M30B_BS8_ZIPF, M30B_256K, M30B_L4)}


def context_lengths(w: Workload) -> np.ndarray:
    """Prefilled positions per sequence: uniform integers in [ctx_lo, ctx_hi]."""
    if w.ctx_lo == w.ctx_hi:
        return np.full(w.B, w.ctx_lo, dtype=np.int32)
    return uniform_int(w.seed, tid(SYNTH_CTX, 0, 0), 0, w.B, w.ctx_lo, w.ctx_hi).astype(np.int32)


def first_tokens(w: Workload) -> np.ndarray:
    return uniform_int(w.seed, tid(SYNTH_TOKENS, 0, 0), 0, w.B, 0, w.V - 1).astype(np.int32)


def page_tables(w: Workload, ctx: np.ndarray, new_tokens: int):
    """Random page tables: each sequence gets ceil((ctx_b + new_tokens) / page) pages, drawn
    in order from a seeded permutation of the whole pool. Unused entries are -1.
    Returns (block_table [B][max_pages] int32, num_pages)."""
    need = [(int(c) + new_tokens + w.page - 1) // w.page for c in ctx]
    num_pages = int(sum(need))
    perm = permutation(w.seed, tid(SYNTH_PAGES, 0, 0), num_pages)
    max_pages = max(need)
    bt = np.full((w.B, max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


def router_bias(w: Workload):
    """None for uniform routing. For "zipf": per layer a seeded expert permutation pi and
    bias_e = ln(p(rank_pi(e))) - mean, p(r) = r^-1.2 / sum_r' r'^-1.2, so that expert
    popularity under the bias follows Zipf(1.2) over a random expert order."""
    if w.routing == "uniform":
        return None
    s = 1.2
    ranks = np.arange(1, w.E + 1, dtype=np.float64)
    logp = -s * np.log(ranks) - math.log(np.sum(ranks ** -s))
    bias = np.zeros((w.L, w.E), dtype=np.float64)
    for l in range(w.L):
        perm = permutation(w.seed, tid(SYNTH_ZIPF, l, 0), w.E)  # perm[r] = expert with rank r+1
        bias[l, perm] = logp
        bias[l] -= bias[l].mean()
    return bias.astype(np.float32)
