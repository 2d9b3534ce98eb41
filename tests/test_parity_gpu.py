"""GPU parity: the single-kernel decode step (through the C ABI) against the CPU oracle on the
same seeded model and KV cache, teacher-forced with the oracle's greedy tokens.

Acceptance: per row and step max|dlogit| <= 3e-2 * std(oracle logits); router top-k ids
identical except where the oracle's router logits tie within 1e-3; >= 99% greedy-argmax
agreement; KV append slot and page lookups bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from harness import Setup, check_step
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch

    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _run(w, steps, per_layer=False, mode=0):
    s = Setup(w, steps, mode=mode)
    tokens = W.first_tokens(w)
    agree = total = waived = 0
    try:
        for i in range(steps):
            pos = s.ctx + i
            rng = np.random.default_rng(i)
            touched = {int(s.bt[b, pos[b] // w.page]) for b in range(w.B)}
            sample_pages = sorted(touched | set(rng.integers(0, s.num_pages, 16).tolist()))
            K_before = {pg: _bits(s.K[:, pg]) for pg in sample_pages}
            V_before = {pg: _bits(s.V[:, pg]) for pg in sample_pages}
            got_logits, got_next = s.gpu_step(tokens, pos)
            ref_logits, ref_next, tr = s.oracle_step(tokens, pos)
            # host copies at once: no device view of the library's workspace outlives the step
            acts = {k: v.cpu().numpy() for k, v in s.dc.activations().items()}
            a, rep = check_step(w, got_logits, got_next, ref_logits, ref_next, acts, tr)
            agree += a
            total += rep["compared"]
            waived += len(rep["waived"])
            if rep["waived"]:
                # a router tie changed those tokens' residual streams after the flipped layer, hence
                # the K/V they appended there: continue from the oracle's appended values
                _resync_new_slots(s, w, pos, tr, rep["waived"])
            elif per_layer:
                _check_layers(w, acts, tr, pos)
            # the appended K/V sit at (block_table[b][pos / 16], pos % 16): the rest of those
            # pages, and a sample of other pages, are unchanged (bit-exact indexing); the values
            # match the oracle's within bf16 rounding
            for pool, before in ((s.K, K_before), (s.V, V_before)):
                for pg in sample_pages:
                    after = _bits(pool[:, pg])
                    keep = np.ones(after.shape, dtype=bool)
                    for b in range(w.B):
                        if s.bt[b, pos[b] // w.page] == pg:
                            keep[:, :, pos[b] % w.page] = False
                    assert np.array_equal(after[keep], before[pg][keep]), "KV bytes outside the new slots changed"
            # values: one bf16 rounding apart, plus the error the step's input carries at depth.
            # The new k and v are outputs of the same QKV GEMV as q, from the same normalized
            # input, so they get q's absolute tolerance (2e-4 of the largest magnitude in the
            # head, as in _check_layers) on top of one bf16 rounding of the value itself.
            kv_abs = 2e-4
            for b in range(w.B):
                if b in rep["waived"]:
                    continue
                pg, sl = s.bt[b, pos[b] // w.page], pos[b] % w.page
                for kv, got, ref in (("K", _bits(s.K[:, pg, :, sl]), tr["k_new"][:, b]),
                                     ("V", _bits(s.V[:, pg, :, sl]), tr["v_new"][:, b])):
                    g32 = synth.bf16_bits_to_f32(got).astype(np.float64)
                    r32 = synth.bf16_bits_to_f32(ref).astype(np.float64)
                    scale = np.abs(r32).max(axis=-1, keepdims=True)
                    bound = 2.0 ** -7 * np.abs(r32) + kv_abs * scale
                    bad = np.abs(g32 - r32) > bound
                    if bad.any():
                        l_, g_, e_ = np.argwhere(bad)[0]
                        raise AssertionError(
                            f"step {i} row {b} pos {pos[b]}: appended {kv} differs from the oracle beyond bf16 "
                            f"rounding and the input's error at {bad.sum()} elements; first at layer {l_} group {g_} "
                            f"dim {e_}: gpu {g32[l_, g_, e_]:.6g} oracle {r32[l_, g_, e_]:.6g} bound {bound[l_, g_, e_]:.3g}"
                            f" (scale {scale[l_, g_, 0]:.3g})")
            tokens = ref_next  # teacher forcing
    finally:
        s.close()
    # a router tie within 1e-3 may pick a different expert on the two sides (allowed); the rows
    # where that happened are not compared on logits, and they must stay a minority
    assert waived <= max(1, (steps * w.B) // 4), f"{waived} of {steps * w.B} rows changed expert on a router tie"
    assert total > 0 and agree >= 0.99 * total, f"greedy agreement {agree}/{total}"


def _resync_new_slots(s, w, pos, tr, rows):
    """Writes the oracle's appended K/V of this step (bf16 bits) for the given rows into the
    GPU's pools."""
    import torch

    for b in rows:
        pg, sl = int(s.bt[b, pos[b] // w.page]), int(pos[b] % w.page)
        for pool, key in ((s.K, "k_new"), (s.V, "v_new")):
            vals = torch.as_tensor(tr[key][:, b].astype(np.int16), device=pool.device).view(torch.bfloat16)
            pool[:, pg, :, sl] = vals


def _check_layers(w, acts, tr, pos):
    for name, tol in (("x", 2e-4), ("attn_out", 2e-3), ("moe_out", 2e-3)):
        got = acts[name]
        ref = tr[name]
        scale = np.abs(ref).max()
        err = np.abs(got - ref).max()
        assert err <= tol * max(scale, 1e-6), f"{name}: max err {err:.3e} vs scale {scale:.3e}"
    q = acts["q"].astype(np.float64)  # before RoPE: rotate with the oracle's RoPE
    for l in range(w.L):
        for b in range(w.B):
            for h in range(w.nq):
                q[l, b, h] = oracle.rope(q[l, b, h], int(pos[b]), w.rope_theta)
    np.testing.assert_allclose(q, tr["q"], rtol=0, atol=2e-4 * np.abs(tr["q"]).max())
    np.testing.assert_allclose(acts["attn"], tr["attn"], rtol=0, atol=2e-3 * np.abs(tr["attn"]).max())


def test_tiny_one_step_all_layers():
    _run(W.TINY, 1, per_layer=True)


def test_tiny_batch3_ragged():
    _run(W.TINY.with_(B=3, ctx_lo=0, ctx_hi=70, steps=4), 4, per_layer=True)


def test_small_bs8_ragged_teacher_forced():
    """All 128 greedy steps of the small batch-8 workload, so the >= 99 % greedy-agreement bar
    is taken over 1,024 tokens."""
    _run(W.SMALL, 128, per_layer=True)


def test_per_op_mode_matches_megakernel_bitwise():
    import torch

    from moe_transformer_decode_gb300 import binding as B

    w = W.SMALL.with_(steps=2)
    outs = []
    for mode in (B.MK_MODE_MEGAKERNEL, B.MK_MODE_PER_OP, B.MK_MODE_MEGAKERNEL):
        s = Setup(w, 2, mode=mode)
        tok = W.first_tokens(w)
        lg, nx = s.gpu_step(tok, s.ctx)
        outs.append((lg, nx, _bits(s.K).copy()))
        s.close()
        torch.cuda.empty_cache()
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])
        assert np.array_equal(o[2], outs[0][2])


def test_greedy_loop_matches_single_steps():
    import torch

    w = W.SMALL
    n = 5
    a = Setup(w, n)
    tok = torch.as_tensor(W.first_tokens(w), device="cuda")
    pos = torch.as_tensor(a.ctx, device="cuda")
    toks = torch.empty((n, w.B), dtype=torch.int32, device="cuda")
    a.dc.greedy(n, tok, pos, a.K, a.V, a.logits, toks)
    a.dc.sync()
    greedy_tokens = toks.cpu().numpy()
    greedy_logits = a.logits.cpu().numpy()
    a.close()
    b = Setup(w, n)
    t = W.first_tokens(w)
    for i in range(n):
        lg, nx = b.gpu_step(t, b.ctx + i)
        assert np.array_equal(nx, greedy_tokens[i])
        t = nx
    assert np.array_equal(lg, greedy_logits)
    b.close()


def test_30b_shape_4_layers_bs1_ctx8k_per_layer():
    """The production layer shape at batch 1 (4 of 48 layers): the attention/expert SM partition,
    attention chunks sized to the partition, and expert-down tasks of 8-row blocks in passes of
    one stage's rows (more row blocks than expert SMs), checked layer by layer."""
    _run(W.M30B_L4, 2, per_layer=True)


@pytest.mark.slow
def test_30b_bs1_ctx8k_full_size():
    """The headline workload at full size (61 GB of weights), 32 teacher-forced steps."""
    _run(W.M30B_BS1, 32)


@pytest.mark.slow
def test_30b_bs8_uniform_full_size():
    _run(W.M30B_BS8, 8)


@pytest.mark.slow
def test_30b_bs8_zipf_full_size():
    _run(W.M30B_BS8_ZIPF, 8)


@pytest.mark.slow
def test_30b_bs1_ctx256k_full_size():
    """The long-context workload: 262,144 cached positions (26 GB of paged KV), 2 steps. The
    oracle synthesises the cache on read, so no host copy of it is made."""
    _run(W.M30B_256K, 2)
