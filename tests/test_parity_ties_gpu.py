"""GPU parity where several answers are plausible and one is canonical: exact ties in the router
logits and in the LM-head logits, and cache slots past the context that hold garbage bits.

The model is the tiny config with rows of its weights duplicated on the host, so that the tie is
exact in both the oracle (fp64 over the same bf16 rows) and the kernel (the same products in the
same order); the oracle reads the modified host arrays (dense source), the kernel copies of them.
Canonical answers: router top-k ids lowest id first among equal logits; greedy argmax the lowest
id among equal logits."""
import numpy as np
import pytest

import oracle
import synth
from harness import router_ties_ok
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _device(model):
    import torch

    out = {}
    for k, v in model.items():
        if v is None:
            continue
        if k == "router_bias":
            out[k] = torch.as_tensor(np.ascontiguousarray(v, np.float32), device="cuda")
        else:
            out[k] = torch.as_tensor(np.ascontiguousarray(v).view(np.int16), device="cuda").view(torch.bfloat16)
    return out


def _run_dense(w, model, ctx, bt, num_pages, K, V, tokens):
    """One step on both sides; returns (gpu logits, gpu next, gpu activations, oracle logits,
    oracle next, oracle trace)."""
    import torch

    from moe_transformer_decode_gb300.context import DecodeContext

    dev = _device(model)
    Kd = torch.as_tensor(K.view(np.int16), device="cuda").view(torch.bfloat16)
    Vd = torch.as_tensor(V.view(np.int16), device="cuda").view(torch.bfloat16)
    dc = DecodeContext(w, dev, max_batch=w.B, max_pages_per_seq=bt.shape[1])
    dc.schedule(ctx, torch.as_tensor(bt, device="cuda"))
    logits = torch.empty((w.B, w.V), device="cuda")
    nxt = torch.empty(w.B, dtype=torch.int32, device="cuda")
    dc.step(torch.as_tensor(tokens, device="cuda"), torch.as_tensor(ctx, device="cuda"), Kd, Vd, logits, nxt)
    dc.sync()
    acts = {k: v.cpu().numpy() for k, v in dc.activations().items()}
    got = logits.cpu().numpy(), nxt.cpu().numpy()
    dc.close()
    src = oracle.DenseSource(w, model, K.copy(), V.copy(), block_table=bt, bias=model.get("router_bias"))
    ref_logits, ref_next, tr = oracle.decode_step(w, src, tokens, ctx, trace=True)
    return got[0], got[1], acts, ref_logits, ref_next, tr


def _tiny_inputs(w):
    ctx = W.context_lengths(w)
    bt, num_pages = W.page_tables(w, ctx, 2)
    K, V = synth.host_kv(w, ctx, bt, num_pages)
    return ctx, bt, num_pages, K, V


def test_router_exact_ties_pick_the_lowest_ids():
    w = W.TINY
    model = synth.host_model(w)
    # layer 0: every router row identical -> all logits tie -> top-2 is experts (0, 1) with
    # weight 1/2 each; layer 1: rows in identical pairs (2j, 2j + 1) -> the winning pair in
    # id order
    model["w_router"][0, :] = model["w_router"][0, 3]
    model["w_router"][1, 1::2] = model["w_router"][1, 0::2]
    ctx, bt, num_pages, K, V = _tiny_inputs(w)
    tokens = W.first_tokens(w)
    lg, nx, acts, ref_lg, ref_nx, tr = _run_dense(w, model, ctx, bt, num_pages, K, V, tokens)
    r0 = acts["router"][0, 0]
    assert np.all(r0.view(np.uint32) == r0[0].view(np.uint32)), "identical router rows gave different logits"
    assert list(acts["topk_ids"][0, 0]) == [0, 1] and list(tr["topk_ids"][0, 0]) == [0, 1]
    np.testing.assert_allclose(acts["topk_w"][0, 0], [0.5, 0.5], rtol=0, atol=1e-7)
    r1 = acts["router"][1, 0]
    assert np.array_equal(r1[0::2].view(np.uint32), r1[1::2].view(np.uint32))
    ids = list(acts["topk_ids"][1, 0])
    assert ids[1] == ids[0] + 1 and ids[0] % 2 == 0, f"pair ties must come out lower id first: {ids}"
    assert router_ties_ok(tr["router"][1, 0], ids, tr["topk_ids"][1, 0])
    assert np.abs(lg[0] - ref_lg[0]).max() <= 3e-2 * ref_lg[0].std()


def test_lm_head_exact_tie_picks_the_lowest_id():
    w = W.TINY
    model = synth.host_model(w)
    ctx, bt, num_pages, K, V = _tiny_inputs(w)
    tokens = W.first_tokens(w)
    src = oracle.DenseSource(w, model, K.copy(), V.copy(), block_table=bt)
    _, first, _ = oracle.decode_step(w, src, tokens, ctx)
    top = int(first[0])
    low = 0 if top > 0 else 7
    if top == 0:  # make row 0 the maximum's twin by copying it upward, the lower id stays 0
        model["lm_head"][low] = model["lm_head"][0]
        want = 0
    else:
        model["lm_head"][low] = model["lm_head"][top]
        want = low
    lg, nx, acts, ref_lg, ref_nx, tr = _run_dense(w, model, ctx, bt, num_pages, K, V, tokens)
    tied = (top, low)
    assert lg[0, tied[0]].view(np.uint32) == lg[0, tied[1]].view(np.uint32), "identical LM rows, different logits"
    assert int(ref_nx[0]) == want and int(nx[0]) == want, f"argmax tie: gpu {nx[0]}, oracle {ref_nx[0]}, want {want}"


def test_garbage_past_the_context_does_not_leak_into_attention():
    """Slots past each sequence's context (the tail of its last page, and pages it has not yet
    reached) hold NaN and huge values; attention masks them, and its P V must not turn 0 * NaN
    into NaN."""
    w = W.TINY.with_(B=3, ctx_lo=1, ctx_hi=70, steps=2)
    model = synth.host_model(w)
    ctx = W.context_lengths(w)
    bt, num_pages = W.page_tables(w, ctx, 2)
    K, V = synth.host_kv(w, ctx, bt, num_pages)
    live = np.zeros(K.shape[:4], dtype=bool)  # [L][page][g][slot]
    for b in range(w.B):
        for pos in range(int(ctx[b])):
            live[:, bt[b, pos // w.page], :, pos % w.page] = True
    rng = np.random.default_rng(7)
    junk = np.where(rng.random(K.shape) < 0.5, 0x7FC0, 0x7F7F).astype(np.uint16)  # NaN, bf16 max
    K = np.where(live[..., None], K, junk)
    V = np.where(live[..., None], V, junk)
    tokens = W.first_tokens(w)
    lg, nx, acts, ref_lg, ref_nx, tr = _run_dense(w, model, ctx, bt, num_pages, K, V, tokens)
    assert np.all(np.isfinite(lg)), "garbage past the context reached the logits"
    assert np.all(np.isfinite(acts["attn"]))
    for b in range(w.B):
        assert np.abs(lg[b] - ref_lg[b]).max() <= 3e-2 * ref_lg[b].std()
    assert np.array_equal(nx, ref_nx)
