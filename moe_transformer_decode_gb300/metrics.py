"""Speed-of-light accounting for one decode step.

Bytes a step must move at minimum (the roofline numerator): every weight the step
touches once (QKV, O, router, norm gains, the experts actually routed this step, counted
once per layer however many tokens share them, the LM head and the embedding rows read)
plus the KV cache read (positions 0..c_b of every sequence, the new one included) and
the new K/V written. Activations and logits are ignored (<0.1%). This follows the
aimodeling.com page "cohere-megakernel-north-mini-code-h100", section "Decode is a
bandwidth game": step time at speed of light = (weight bytes + KV bytes) / HBM bandwidth.
"""
from __future__ import annotations

import numpy as np

BF16 = 2


def sol_tok_s(bytes_per_step: float, tokens_per_step: int, bw_bytes_per_s: float) -> float:
    return tokens_per_step * bw_bytes_per_s / bytes_per_step


def step_bytes(w, positions, distinct_experts_per_layer) -> dict:
    """w: workload shape; positions[b]: the new token's position (= cached length);
    distinct_experts_per_layer: number of distinct experts routed in each layer."""
    positions = np.asarray(positions, dtype=np.int64)
    de = np.asarray(distinct_experts_per_layer, dtype=np.float64)  # may be a mean over steps
    assert de.shape == (w.L,)
    dense = w.L * (w.qkv_rows * w.H + w.H * w.nq * w.d + w.E * w.H + w.H) * BF16
    experts = int(round(float(de.sum()) * 3 * w.I * w.H * BF16))
    head = (w.V * w.H + w.H + len(positions) * w.H) * BF16
    kv_row = w.L * 2 * w.nkv * w.d * BF16
    kv_read = int((positions + 1).sum()) * kv_row
    kv_write = len(positions) * kv_row
    total = dense + experts + head + kv_read + kv_write
    return {"dense_weights": dense, "experts": experts, "lm_head_embed": head, "kv_read": kv_read,
            "kv_write": kv_write, "total": total}
