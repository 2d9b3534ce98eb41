"""Run-to-run determinism of the decode step on the GPU.

Every partial sum of the step is combined in a fixed order (the GEMV k-slices, the expert-down
partials in rank order, the attention chunks by log-sum-exp in chunk order), and the gate/up
units are split over the blocks by a rule every block computes alike from the step's routing,
so two runs of the same steps give the same bits. The batch-8 Zipf workload is the case where
the routing concentrates on few experts and the split over the routed units matters most."""
import numpy as np
import pytest

from harness import Setup
from synth import workloads as W


def _run_steps(w, n):
    import torch

    s = Setup(w, n)
    tok = torch.as_tensor(W.first_tokens(w), device="cuda")
    pos = torch.as_tensor(s.ctx, device="cuda")
    toks = torch.empty((n, w.B), dtype=torch.int32, device="cuda")
    s.dc.greedy(n, tok, pos, s.K, s.V, s.logits, toks)
    s.dc.sync()
    # the appended K/V slots of every sequence and step (the only cache bytes a step writes)
    kv = []
    for b in range(w.B):
        for i in range(n):
            pg, sl = s.bt[b, (s.ctx[b] + i) // w.page], (s.ctx[b] + i) % w.page
            kv.append(s.K[:, pg, :, sl].view(torch.int16).cpu().numpy())
            kv.append(s.V[:, pg, :, sl].view(torch.int16).cpu().numpy())
    out = toks.cpu().numpy(), s.logits.cpu().numpy(), np.stack(kv)
    s.close()
    del s
    torch.cuda.empty_cache()
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["moe30b_a3b_bs8_ctx1k8k_zipf", "small_bs8_ragged"])
def test_decode_steps_are_bitwise_deterministic(name):
    w = W.ALL[name]
    n = 4
    t1, l1, k1 = _run_steps(w, n)
    t2, l2, k2 = _run_steps(w, n)
    assert np.array_equal(t1, t2), "greedy tokens differ between two runs"
    assert l1.tobytes() == l2.tobytes(), "last step's logits differ between two runs"
    assert k1.tobytes() == k2.tobytes(), "the appended K/V differ between two runs"
