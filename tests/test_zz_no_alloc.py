"""mk_decode_step_noalloc: the decode step for callers that cannot allocate device memory
(an arena or pool owns all device memory, or allocation is forbidden after start-up). It keeps
its workspace in the library's static device array; the GPU tests check it against
mk_decode_step on the same model and KV cache, over two calls in a row with the greedy token
fed back. The CPU tests show that it makes the same checks of its arguments as mk_create, and
returns before any device work when one fails (fake pointers, never dereferenced)."""
import ctypes

import numpy as np
import pytest

from synth import workloads as W


def _cfg(w, max_pages):
    from moe_transformer_decode_gb300 import binding as B

    return B.mk_model_cfg(w.L, w.H, w.nq, w.nkv, w.d, w.E, w.topk, w.I, w.V, 16, w.B, max_pages, w.rope_theta, w.eps)


@pytest.mark.gpu
@pytest.mark.parametrize("w", [W.TINY, W.SMALL], ids=["tiny", "small_bs8"])
def test_noalloc_step_matches_decode_step(w):
    import torch

    import synth
    from moe_transformer_decode_gb300 import binding as B
    from moe_transformer_decode_gb300.context import DecodeContext

    ctx = W.context_lengths(w)
    bt, num_pages = W.page_tables(w, ctx, 4)
    model = synth.device_model(w)
    K1, V1 = synth.device_kv(w, ctx, bt, num_pages)
    K2, V2 = K1.clone(), V1.clone()
    bt_d = torch.as_tensor(bt, device="cuda")
    dc = DecodeContext(w, model, max_batch=w.B, max_pages_per_seq=bt.shape[1])
    dc.schedule(ctx, bt_d)
    cfg = _cfg(w, bt.shape[1])
    ptrs = B.mk_weight_ptrs(**{k: (model[k].data_ptr() if k in model else None) for k, _ in B.mk_weight_ptrs._fields_})
    tok_a = torch.as_tensor(W.first_tokens(w), device="cuda")
    tok_b = tok_a.clone()
    for step in range(2):
        pos = torch.as_tensor(ctx + step, device="cuda")
        lg_a = torch.empty((w.B, w.V), device="cuda")
        nx_a = torch.empty(w.B, dtype=torch.int32, device="cuda")
        dc.step(tok_a, pos, K1, V1, lg_a, nx_a)
        dc.sync()
        lg_b = torch.full((w.B, w.V), float("nan"), device="cuda")
        nx_b = torch.full((w.B,), -1, dtype=torch.int32, device="cuda")
        B.mk_decode_step_noalloc(cfg, ptrs, ctx + step, bt_d, tok_b, pos, B.mk_kv_pages(K2.data_ptr(), V2.data_ptr(),
                                 num_pages), lg_b, nx_b)
        a, b = lg_a.cpu().numpy(), lg_b.cpu().numpy()
        for r in range(w.B):
            assert np.abs(a[r] - b[r]).max() <= 3e-2 * a[r].std(), f"step {step} row {r}: logits differ"
        assert np.array_equal(nx_a.cpu().numpy(), nx_b.cpu().numpy())
        for b_ in range(w.B):  # the appended K/V land in the same slot with the same values
            pg, sl = bt[b_, (ctx[b_] + step) // 16], (ctx[b_] + step) % 16
            assert torch.equal(K1[:, pg, :, sl], K2[:, pg, :, sl]) and torch.equal(V1[:, pg, :, sl], V2[:, pg, :, sl])
        tok_a, tok_b = nx_a.clone(), nx_b.clone()
    dc.close()


@pytest.mark.gpu
def test_noalloc_rejects_workspace_beyond_the_static_array():
    from moe_transformer_decode_gb300 import binding as B

    w = W.M30B_BS1
    cfg = _cfg(w, 600)
    fake = 1 << 20  # never dereferenced: the size check comes first
    ptrs = B.mk_weight_ptrs(*([fake] * 5 + [None] + [fake] * 4))
    kv = B.mk_kv_pages(fake, fake, 600)
    msg = ctypes.create_string_buffer(256)
    lens = np.array([8192], np.int32)
    st = B.lib().mk_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(ptrs), 1, lens.ctypes.data, fake, fake, fake,
                                        ctypes.byref(kv), None, None, None, msg, len(msg))
    assert st == B.MK_ERR_UNSUPPORTED
    assert b"static scratch" in msg.value


FAKE = 1 << 20  # a 16-byte-aligned address that is never dereferenced


def _call(cfg, ptrs, kv, lens):
    from moe_transformer_decode_gb300 import binding as B

    msg = ctypes.create_string_buffer(256)
    lens = np.asarray(lens, np.int32)
    st = B.lib().mk_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(ptrs), len(lens), lens.ctypes.data, FAKE,
                                        FAKE, FAKE, ctypes.byref(kv), None, None, None, msg, len(msg))
    return st, msg.value.decode()


def _good():
    from moe_transformer_decode_gb300 import binding as B

    cfg = B.mk_model_cfg(2, 256, 4, 2, 64, 8, 2, 512, 1024, 16, 1, 8, 1e4, 1e-6)
    ptrs = B.mk_weight_ptrs(*([FAKE] * 5 + [None] + [FAKE] * 4))
    kv = B.mk_kv_pages(FAKE, FAKE, 8)
    return cfg, ptrs, kv


def test_noalloc_rejects_what_mk_create_rejects_before_device_work():
    """Every bad config, pointer or KV pool is refused on the host, before the call looks for a
    device: these run (and must pass) on a machine without a GPU."""
    from moe_transformer_decode_gb300 import binding as B

    lib = B.lib()
    out = ctypes.c_void_p()
    cases = []
    # (fields of mk_model_cfg without theta/eps, theta, eps, expected status, why)
    base = [2, 256, 4, 2, 64, 8, 2, 512, 1024, 16, 1, 8]

    def with_(**kw):
        f = list(base)
        names = ["n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "n_experts", "top_k", "expert_inter",
                 "vocab", "page_size", "max_batch", "max_pages_per_seq"]
        for k, v in kw.items():
            f[names.index(k)] = v
        return f

    # the ring-stage bound: one expert's hi/lo activations for the batch exceed a 32 KB stage
    cases.append((with_(max_batch=8, expert_inter=2048), 1e4, 1e-6, B.MK_ERR_UNSUPPORTED, "batch 8 at inter 2048"))
    cases.append((with_(max_batch=8, expert_inter=1280), 1e4, 1e-6, B.MK_ERR_UNSUPPORTED, "batch 8 at inter 1280"))
    # sizes <= 0 (a negative expert_inter must not reach any offset arithmetic)
    cases.append((with_(expert_inter=-256), 1e4, 1e-6, B.MK_ERR_INVALID_ARG, "negative expert_inter"))
    cases.append((with_(n_q_heads=0), 1e4, 1e-6, B.MK_ERR_INVALID_ARG, "no query heads"))
    cases.append((with_(n_kv_heads=0), 1e4, 1e-6, B.MK_ERR_INVALID_ARG, "no kv heads"))
    cases.append((with_(n_layers=-1), 1e4, 1e-6, B.MK_ERR_INVALID_ARG, "negative layers"))
    cases.append((with_(top_k=9), 1e4, 1e-6, B.MK_ERR_INVALID_ARG, "top_k > experts"))
    cases.append((base, 1e4, -1e-6, B.MK_ERR_INVALID_ARG, "negative rms_eps"))
    cases.append((base, 0.0, 1e-6, B.MK_ERR_INVALID_ARG, "rope_theta 0"))
    cases.append((base, -1e4, 1e-6, B.MK_ERR_INVALID_ARG, "negative rope_theta"))
    cases.append((base, float("nan"), 1e-6, B.MK_ERR_INVALID_ARG, "NaN rope_theta"))
    cases.append((with_(hidden=300), 1e4, 1e-6, B.MK_ERR_UNSUPPORTED, "hidden 300"))
    cases.append((with_(page_size=32), 1e4, 1e-6, B.MK_ERR_UNSUPPORTED, "page size 32"))
    _, ptrs, kv = _good()
    for fields, theta, eps, want, why in cases:
        cfg = B.mk_model_cfg(*fields, theta, eps)
        st, msg = _call(cfg, ptrs, kv, [32])
        assert st == want, f"{why}: got {st} ({msg})"
        assert msg, why
        # mk_create makes the same decision (shared validator)
        assert lib.mk_create(ctypes.byref(cfg), ctypes.byref(ptrs), ctypes.byref(out)) == want, why

    cfg, ptrs, kv = _good()
    for i, name in enumerate(["embed", "norm_gain", "w_qkv", "w_o", "w_router", "w_gate_up", "w_down", "final_gain",
                              "lm_head"]):
        bad = B.mk_weight_ptrs(*([FAKE] * 5 + [None] + [FAKE] * 4))
        setattr(bad, name, FAKE + 8)  # misaligned
        st, msg = _call(cfg, bad, kv, [32])
        assert st == B.MK_ERR_INVALID_ARG and "aligned" in msg, name
        setattr(bad, name, None)  # missing
        st, msg = _call(cfg, bad, kv, [32])
        assert st == B.MK_ERR_INVALID_ARG, name
    bad = B.mk_weight_ptrs(*([FAKE] * 5 + [FAKE + 4] + [FAKE] * 4))  # misaligned router bias
    assert _call(cfg, bad, kv, [32])[0] == B.MK_ERR_INVALID_ARG
    for k, v, n in ((FAKE + 8, FAKE, 8), (FAKE, FAKE + 2, 8), (None, FAKE, 8), (FAKE, FAKE, 0)):
        st, msg = _call(cfg, ptrs, B.mk_kv_pages(k, v, n), [32])
        assert st == B.MK_ERR_INVALID_ARG and "KV" in msg
