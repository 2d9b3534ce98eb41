"""Failure detection on the GPU without a fault: every device-side wait has a time limit, and
bad inputs the kernel checks before using them are reported, not acted on.

- A 1 us wait limit makes the step's first dependency wait run out: the step ends early with
  MK_ERR_DEVICE_TIMEOUT (nothing hangs, nothing traps), and after the status is read the same
  context, back at the default limit, produces a step that matches the oracle.
- An out-of-range page id in the block table (a cached page, and the page of the new token's
  slot) is reported as MK_ERR_BAD_PAGE; no KV byte of any valid page changes except the new
  slot of the sequence whose page is valid."""
import numpy as np
import pytest

from harness import Setup, check_step
from moe_transformer_decode_gb300 import binding as B
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(__import__("torch").int16).cpu().numpy().view(np.uint16)


def test_wait_limit_runs_out_then_context_recovers():
    w = W.TINY
    s = Setup(w, 2)
    try:
        tokens = W.first_tokens(w)
        s.dc.set_wait_limit(1000)
        import torch
        tok = torch.as_tensor(tokens, device="cuda")
        pos = torch.as_tensor(s.ctx, device="cuda")
        s.dc.step(tok, pos, s.K, s.V, s.logits, s.next)
        assert B.mk_status_sync(s.dc.ctx) == B.MK_ERR_DEVICE_TIMEOUT
        assert "time" in B.mk_last_error(s.dc.ctx).lower()
        with pytest.raises(B.MkError):
            B.mk_set_wait_limit(s.dc.ctx, 10)  # below the accepted range
        s.dc.set_wait_limit(2_000_000_000)
        got_logits, got_next = s.gpu_step(tokens, s.ctx)
        ref_logits, ref_next, tr = s.oracle_step(tokens, s.ctx)
        acts = {k: v.cpu().numpy() for k, v in s.dc.activations().items()}
        agree, _ = check_step(w, got_logits, got_next, ref_logits, ref_next, acts, tr)
        assert agree == w.B
    finally:
        s.close()


@pytest.mark.parametrize("where", ["cached_page", "new_slot_page"])
def test_bad_page_id_is_reported_without_stray_writes(where):
    import torch

    w = W.TINY.with_(B=2, ctx_lo=40, ctx_hi=40)
    s = Setup(w, 1)
    try:
        bt = s.bt.copy()
        b_bad = 1
        col = 0 if where == "cached_page" else int(s.ctx[b_bad]) // w.page
        bt[b_bad, col] = s.num_pages + 7  # out of range
        s.dc.schedule(s.ctx, torch.as_tensor(bt, device="cuda"))
        before_k, before_v = _bits(s.K), _bits(s.V)
        tok = torch.as_tensor(W.first_tokens(w), device="cuda")
        pos = torch.as_tensor(s.ctx, device="cuda")
        s.dc.step(tok, pos, s.K, s.V, s.logits, s.next)
        assert B.mk_status_sync(s.dc.ctx) == B.MK_ERR_BAD_PAGE
        after_k, after_v = _bits(s.K), _bits(s.V)
        keep = np.ones(after_k.shape, dtype=bool)
        good_b = 0  # the other sequence appends normally
        keep[:, s.bt[good_b, int(s.ctx[good_b]) // w.page], :, int(s.ctx[good_b]) % w.page] = False
        if where == "cached_page":  # sequence 1's own new slot sits on a valid page
            keep[:, s.bt[b_bad, int(s.ctx[b_bad]) // w.page], :, int(s.ctx[b_bad]) % w.page] = False
        assert np.array_equal(after_k[keep], before_k[keep])
        assert np.array_equal(after_v[keep], before_v[keep])
    finally:
        s.close()
