"""mk_decode_step_noalloc: the decode step for callers that cannot allocate device memory
(an arena or pool owns all device memory, or allocation is forbidden after start-up). It keeps
its workspace in the library's static device array; this checks it against mk_decode_step on
the same model and KV cache, over two calls in a row with the greedy token fed back."""
import ctypes

import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu


def _cfg(w, max_pages):
    from moe_transformer_decode_gb300 import binding as B

    return B.mk_model_cfg(w.L, w.H, w.nq, w.nkv, w.d, w.E, w.topk, w.I, w.V, 16, w.B, max_pages, w.rope_theta, w.eps)


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
