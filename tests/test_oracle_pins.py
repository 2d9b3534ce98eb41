"""Pins for the CPU oracle: closed forms, invariants and library routines, each chosen so
that a plausible mistake (a dropped term, a wrong sign or index, a transposed operand)
fails at least one. None of these re-types the oracle's own code."""
import cmath
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from synth import workloads as W

RNG = np.random.default_rng(1234)


def rand_bf16(shape, scale=1.0):
    t = torch.from_numpy(RNG.standard_normal(shape).astype(np.float32) * scale).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_t(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)


# ------------------------------------------------------------------ bf16 rounding

def test_bf16_round_trip_and_ties():
    lib = oracle.lib()
    assert lib.orc_double_to_bf16(1.0) == 0x3F80
    assert lib.orc_double_to_bf16(-2.0) == 0xC000
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert lib.orc_double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert lib.orc_double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert lib.orc_double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    # agrees with torch's fp32 -> bf16 rounding on fp32-representable values
    x = RNG.standard_normal(4096).astype(np.float32) * np.float32(3.0)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)
    bits = ref
    assert np.array_equal(np.array([lib.orc_bf16_to_double(int(b)) for b in bits]),
                          torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy())


# ------------------------------------------------------------------ GEMV

def test_matvec_matches_numpy():
    W_ = rand_bf16((37, 53))
    x = RNG.standard_normal(53)
    y = np.empty(37)
    oracle.lib().orc_matvec(W_.ctypes.data, 37, 53, np.ascontiguousarray(x).ctypes.data, y.ctypes.data)
    np.testing.assert_allclose(y, bits_to_t(W_).numpy() @ x, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    n, eps = 64, 1e-6
    g = rand_bf16(n, 0.1)
    gd = bits_to_t(g).numpy()
    for c in (0.5, -3.0, 1e-4):
        out = oracle.rmsnorm(np.full(n, c), g, eps)
        np.testing.assert_allclose(out, math.copysign(1, c) * abs(c) / math.sqrt(c * c + eps) * gd, rtol=1e-13)


def test_rmsnorm_scale_invariance_and_library():
    n = 256
    x = RNG.standard_normal(n)
    g = rand_bf16(n, 0.5)
    a = oracle.rmsnorm(x, g, 0.0)
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, g, 0.0), a, rtol=1e-13)
    ref = F.rms_norm(torch.from_numpy(x), (n,), weight=bits_to_t(g), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, g, 1e-6), ref, rtol=1e-12)


# ------------------------------------------------------------------ RoPE

def test_rope_d2_is_complex_rotation():
    # with d = 2 there is one pair with frequency theta^0 = 1: (a + ib) e^{i pos}
    for pos in (0, 1, 5, 1000):
        a, b = 0.3, -1.7
        z = complex(a, b) * cmath.exp(1j * pos)
        np.testing.assert_allclose(oracle.rope([a, b], pos, 1e4), [z.real, z.imag], rtol=1e-12, atol=1e-12)


def test_rope_pair_frequencies_and_layout():
    # d = 4: element i pairs with i + 2 and turns by pos * theta^(-2i/4)
    theta, pos = 1e4, 3
    v = np.array([1.0, 2.0, 3.0, 4.0])
    out = oracle.rope(v, pos, theta)
    for i in range(2):
        z = complex(v[i], v[i + 2]) * cmath.exp(1j * pos * theta ** (-2 * i / 4))
        assert out[i] == pytest.approx(z.real, abs=1e-12)
        assert out[i + 2] == pytest.approx(z.imag, abs=1e-12)


def test_rope_identity_norm_and_relative_position():
    d = 64
    q, k = RNG.standard_normal(d), RNG.standard_normal(d)
    np.testing.assert_array_equal(oracle.rope(q, 0, 1e4), q)
    r = oracle.rope(q, 777, 1e4)
    for i in range(d // 2):
        assert math.hypot(r[i], r[i + d // 2]) == pytest.approx(math.hypot(q[i], q[i + d // 2]), rel=1e-12)
    dots = [oracle.rope(q, p + s, 1e4) @ oracle.rope(k, s, 1e4) for p, s in ((5, 0), (5, 11), (5, 300))]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ------------------------------------------------------------------ attention

def test_attention_single_key_returns_value():
    d = 64
    K, V = rand_bf16((1, d)), rand_bf16((1, d))
    out = oracle.attention_head(RNG.standard_normal(d) * 10, K, V)
    np.testing.assert_array_equal(out, bits_to_t(V).numpy()[0])


def test_attention_equal_keys_give_mean_value():
    d, n = 32, 9
    K = np.repeat(rand_bf16((1, d)), n, axis=0)
    V = rand_bf16((n, d))
    out = oracle.attention_head(RNG.standard_normal(d), K, V)
    np.testing.assert_allclose(out, bits_to_t(V).numpy().mean(0), rtol=1e-12, atol=1e-14)


def test_attention_matches_library_sdpa():
    d, n = 64, 300
    q = RNG.standard_normal(d)
    K, V = rand_bf16((n, d)), rand_bf16((n, d))
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None, None, None], bits_to_t(K)[None, None],
                                         bits_to_t(V)[None, None])[0, 0, 0].numpy()
    np.testing.assert_allclose(oracle.attention_head(q, K, V), ref, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ router and experts

def test_route_topk_and_softmax():
    E, k = 128, 8
    lg = RNG.standard_normal(E)
    ids, w = oracle.route(lg, k)
    ref_ids = np.argsort(-lg.astype(np.float32), kind="stable")[:k]
    assert np.array_equal(ids, ref_ids)
    ref_w = torch.softmax(torch.from_numpy(lg[ref_ids]), 0).numpy()
    np.testing.assert_allclose(w, ref_w, rtol=1e-13)
    assert w.sum() == pytest.approx(1.0, abs=1e-14)


def test_route_ties_go_to_lower_expert_id():
    lg = np.array([0.0, 2.0, 5.0, 2.0, 5.0, 1.0])
    ids, w = oracle.route(lg, 3)
    assert list(ids) == [2, 4, 1]
    np.testing.assert_allclose(w[:2], w[0])
    # values equal in fp32 but not in fp64 still tie (the decision is taken in fp32)
    lg2 = np.array([1.0, 1.0 + 1e-12, 0.5])
    assert list(oracle.route(lg2, 1)[0]) == [0]
    # +0 and -0 are equal logits: the lower id goes first whatever the sign bit
    lg3 = np.array([-1.0, 0.0, -0.0, -2.0])
    assert list(oracle.route(lg3, 2)[0]) == [1, 2]
    lg4 = np.array([-1.0, -0.0, 0.0, -2.0])
    assert list(oracle.route(lg4, 2)[0]) == [1, 2]
    # -inf logits still yield k distinct, valid experts (lowest free ids first)
    lg5 = np.array([-np.inf, 3.0, -np.inf, -np.inf])
    assert list(oracle.route(lg5, 3)[0]) == [1, 0, 2]


def test_expert_matches_library_swiglu():
    H, I = 64, 96
    Wgu, Wd = rand_bf16((2 * I, H), 0.1), rand_bf16((H, I), 0.1)
    x = RNG.standard_normal(H)
    Wg, Wu = bits_to_t(Wgu)[:I], bits_to_t(Wgu)[I:]
    xt = torch.from_numpy(x)
    ref = (bits_to_t(Wd) @ (F.silu(Wg @ xt) * (Wu @ xt))).numpy()
    np.testing.assert_allclose(oracle.expert(Wgu, Wd, x), ref, rtol=1e-11, atol=1e-13)


def test_moe_one_expert_top1_is_dense_swiglu():
    H, I = 48, 80
    Wr = rand_bf16((1, H))
    Wgu, Wd = rand_bf16((1, 2 * I, H), 0.1), rand_bf16((1, H, I), 0.1)
    x = RNG.standard_normal(H)
    y, _, ids, w = oracle.moe(x, Wr, None, Wgu, Wd, 1)
    assert list(ids) == [0] and w[0] == 1.0
    xt = torch.from_numpy(x)
    g, u = bits_to_t(Wgu[0])[:I] @ xt, bits_to_t(Wgu[0])[I:] @ xt
    np.testing.assert_allclose(y, (bits_to_t(Wd[0]) @ (F.silu(g) * u)).numpy(), rtol=1e-11, atol=1e-13)


def test_moe_all_experts_is_softmax_weighted_sum_with_bias():
    H, I, E = 32, 40, 6
    Wr = rand_bf16((E, H))
    Wgu, Wd = rand_bf16((E, 2 * I, H), 0.1), rand_bf16((E, H, I), 0.1)
    bias = RNG.standard_normal(E).astype(np.float32)
    x = RNG.standard_normal(H)
    y, lg, ids, w = oracle.moe(x, Wr, bias, Wgu, Wd, E)
    xt = torch.from_numpy(x)
    logits = bits_to_t(Wr) @ xt + torch.from_numpy(bias).double()
    np.testing.assert_allclose(lg, logits.numpy(), rtol=1e-12)
    p = torch.softmax(logits, 0)
    ref = sum(p[e] * (bits_to_t(Wd[e]) @ (F.silu(bits_to_t(Wgu[e])[:I] @ xt) * (bits_to_t(Wgu[e])[I:] @ xt)))
              for e in range(E))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-10, atol=1e-13)
    assert sorted(ids) == list(range(E))


# ------------------------------------------------------------------ whole step

MINI = W.Workload("pin_mini", L=2, H=64, nq=4, nkv=2, d=16, E=4, topk=2, I=32, V=50, B=1, ctx_lo=4, ctx_hi=4,
                  steps=1, seed=7)


def _torch_full_forward(w, m, tokens):
    """Textbook full-sequence causal forward in fp64 with library ops (F.rms_norm, SDPA with a
    causal mask, F.silu, torch.topk). K and V are rounded to bf16 as a bf16 cache holds them.
    Returns (logits at every position [T][V], per-layer bf16 K and V [L][T][nkv][d])."""
    T = len(tokens)
    x = bits_to_t(m["embed"])[torch.as_tensor(tokens, dtype=torch.long)]
    pos = torch.arange(T, dtype=torch.float64)
    inv = w.rope_theta ** (-2.0 * torch.arange(w.d // 2, dtype=torch.float64) / w.d)
    ang = pos[:, None] * inv[None]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(t):  # [T][heads][d], rotate-half
        a, b = t[..., : w.d // 2], t[..., w.d // 2:]
        c, s = cos[:, None], sin[:, None]
        return torch.cat([a * c - b * s, a * s + b * c], -1)

    Ks, Vs = [], []
    for l in range(w.L):
        n = F.rms_norm(x, (w.H,), weight=bits_to_t(m["norm_gain"][l]), eps=w.eps)
        qkv = n @ bits_to_t(m["w_qkv"][l]).T
        q = qkv[:, : w.nq * w.d].view(T, w.nq, w.d)
        k = qkv[:, w.nq * w.d:(w.nq + w.nkv) * w.d].view(T, w.nkv, w.d)
        v = qkv[:, (w.nq + w.nkv) * w.d:].view(T, w.nkv, w.d)
        q, k = rot(q), rot(k)
        k = k.to(torch.bfloat16).double()
        v = v.to(torch.bfloat16).double()
        Ks.append(k), Vs.append(v)
        rep = w.nq // w.nkv
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.repeat_interleave(rep, 1).transpose(0, 1),
                                           v.repeat_interleave(rep, 1).transpose(0, 1), is_causal=True)
        attn = o.transpose(0, 1).reshape(T, -1) @ bits_to_t(m["w_o"][l]).T
        r = n @ bits_to_t(m["w_router"][l]).T
        top = torch.topk(r.float(), w.topk, dim=-1).indices
        moe = torch.zeros_like(x)
        for t in range(T):
            wts = torch.softmax(r[t, top[t]], 0)
            for j, e in enumerate(top[t].tolist()):
                gu = bits_to_t(m["w_gate_up"][l, e]) @ n[t]
                h = F.silu(gu[: w.I]) * gu[w.I:]
                moe[t] += wts[j] * (bits_to_t(m["w_down"][l, e]) @ h)
        x = x + attn + moe
    n = F.rms_norm(x, (w.H,), weight=bits_to_t(m["final_gain"]), eps=w.eps)
    return (n @ bits_to_t(m["lm_head"]).T).numpy(), Ks, Vs


def test_decode_step_equals_full_causal_forward():
    w = MINI
    m = synth.host_model(w)
    tokens = [3, 17, 42, 8, 29]
    T = len(tokens)
    ref_logits, Ks, Vs = _torch_full_forward(w, m, tokens)
    to_bits = lambda t: t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # contiguous cache [L][B][nkv][max_len][d] holding positions 0..T-2 from the full forward
    K = np.zeros((w.L, 1, w.nkv, T, w.d), np.uint16)
    V = np.zeros_like(K)
    for l in range(w.L):
        K[l, 0, :, : T - 1] = to_bits(Ks[l][: T - 1].transpose(0, 1))
        V[l, 0, :, : T - 1] = to_bits(Vs[l][: T - 1].transpose(0, 1))
    src = oracle.DenseSource(w, m, K, V, block_table=None)
    logits, nxt, _ = oracle.decode_step(w, src, [tokens[-1]], [T - 1])
    np.testing.assert_allclose(logits[0], ref_logits[-1].astype(np.float32), rtol=1e-6, atol=1e-7)
    assert nxt[0] == int(np.argmax(ref_logits[-1].astype(np.float32)))
    # the appended slot holds the full forward's bf16 k and v for the last position
    for l in range(w.L):
        assert np.array_equal(K[l, 0, :, T - 1], to_bits(Ks[l][T - 1]))
        assert np.array_equal(V[l, 0, :, T - 1], to_bits(Vs[l][T - 1]))


def _paged(w, K_c, V_c, ctx, perm_seed):
    """Scatter a contiguous cache into a randomly permuted page pool."""
    rng = np.random.default_rng(perm_seed)
    need = [(c + w.page) // w.page + 1 for c in ctx]
    num_pages = sum(need) + 3
    perm = rng.permutation(num_pages)
    bt = np.full((w.B, max(need)), -1, np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += n
    Kp = np.zeros((w.L, num_pages, w.nkv, w.page, w.d), np.uint16)
    Vp = np.zeros_like(Kp)
    for l in range(w.L):
        for b in range(w.B):
            for pos in range(ctx[b]):
                pg = bt[b, pos // w.page]
                Kp[l, pg, :, pos % w.page] = K_c[l, b, :, pos]
                Vp[l, pg, :, pos % w.page] = V_c[l, b, :, pos]
    return Kp, Vp, bt


def test_paged_equals_contiguous_and_append_touches_one_slot():
    w = MINI.with_(B=3)
    m = synth.host_model(w)
    ctx = [5, 21, 0]
    max_len = 40
    K_c = np.zeros((w.L, w.B, w.nkv, max_len, w.d), np.uint16)
    V_c = np.zeros_like(K_c)
    for b, c in enumerate(ctx):
        K_c[:, b, :, :c] = rand_bf16((w.L, w.nkv, c, w.d))
        V_c[:, b, :, :c] = rand_bf16((w.L, w.nkv, c, w.d))
    tokens = [1, 2, 3]
    Kp, Vp, bt = _paged(w, K_c, V_c, ctx, 5)
    Kp2, Vp2, bt2 = _paged(w, K_c, V_c, ctx, 6)
    before = (Kp.copy(), Vp.copy())
    a = oracle.decode_step(w, oracle.DenseSource(w, m, K_c, V_c), tokens, ctx)
    b = oracle.decode_step(w, oracle.DenseSource(w, m, Kp, Vp, bt), tokens, ctx)
    c = oracle.decode_step(w, oracle.DenseSource(w, m, Kp2, Vp2, bt2), tokens, ctx)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[0], c[0])
    # only slot (bt[b][pos / page], pos % page) changed, in every layer and group
    mask = np.zeros(Kp.shape, bool)
    for bb, p in enumerate(ctx):
        mask[:, bt[bb, p // w.page], :, p % w.page] = True
    for pool, old in zip((Kp, Vp), before):
        assert np.array_equal(pool[~mask], old[~mask])
        assert not np.array_equal(pool[mask], old[mask])


def test_batch_invariance_and_residual_trace():
    w = W.TINY.with_(B=3)
    ctx = np.array([32, 7, 19], np.int32)
    tokens = np.array([5, 900, 77], np.int32)
    full = oracle.decode_step(w, oracle.SynthSource(w, ctx, 2), tokens, ctx, trace=True)
    for b in range(w.B):
        w1 = w.with_(B=1)
        # the synth source keys KV streams by b, so feed row b's cache through a dense source
        bt, npg = W.page_tables(w, ctx, 2)
        K, V = synth.host_kv(w, ctx, bt, npg)
        src = oracle.DenseSource(w1, synth.host_model(w), K, V, bt[b:b + 1])
        one = oracle.decode_step(w1, src, tokens[b:b + 1], ctx[b:b + 1])
        assert np.array_equal(one[0][0], full[0][b])
    tr = full[2]
    np.testing.assert_allclose(tr["x"][1:], tr["x"][:-1] + tr["attn_out"] + tr["moe_out"], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(tr["topk_w"].sum(-1), 1.0, rtol=1e-6)


def test_sol_arithmetic_reproduces_pages():
    import json
    import os

    from moe_transformer_decode_gb300 import metrics

    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_sol.json")))
    sol = metrics.sol_tok_s((g["weight_gb_per_step"] + g["kv_gb_per_step_at_8k"]) * 1e9, 1, g["hbm_tb_per_s"] * 1e12)
    assert abs(sol - g["sol_tok_s_about"]) < 5  # "about 470"
    assert round(100 * g["megakernel_tok_s"] / sol) == g["megakernel_pct_of_sol"]
    assert round(100 * g["vllm_tok_s"] / sol) == g["vllm_pct_of_sol"]
    assert round(g["megakernel_tok_s"] / g["vllm_tok_s"], 2) == g["speedup_bs1"]
    assert 100 - g["vllm_pct_of_sol"] == g["idle_bandwidth_pct"]
