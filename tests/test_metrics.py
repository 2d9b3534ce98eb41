"""The roofline numerator: bytes a decode step must move, against the per-row figures of the
hot-path table (computed there from the model dimensions, independently of this code) and
against invariants of the accounting."""
import numpy as np
import pytest

from moe_transformer_decode_gb300 import metrics
from synth import workloads as W


def test_30b_batch1_8k_step_bytes_match_the_per_row_figures():
    w = W.M30B_BS1
    b = metrics.step_bytes(w, [8192], [8] * w.L)
    assert b["total"] == pytest.approx(6.887e9, rel=1e-3)
    # per layer: QKV 21.0 MB, O-proj 16.8 MB, router 0.52 MB; experts 6.29 + 3.15 MB each
    qkv = (w.nq + 2 * w.nkv) * w.d * w.H * 2
    assert qkv / 1e6 == pytest.approx(21.0, abs=0.05)
    assert w.H * w.nq * w.d * 2 / 1e6 == pytest.approx(16.8, abs=0.05)
    assert w.E * w.H * 2 / 1e6 == pytest.approx(0.52, abs=0.005)
    assert b["experts"] / (w.L * 8) / 1e6 == pytest.approx(6.29 + 3.15, abs=0.01)
    # KV read at 8K: 16.8 MB per layer; LM head 621 MB
    assert b["kv_read"] / w.L / 1e6 == pytest.approx(16.8, abs=0.05)
    assert w.V * w.H * 2 / 1e6 == pytest.approx(621, abs=0.5)
    # expert bytes are 52.6 % of the step, QKV 14.6 %, KV 11.7 %, LM head 9.0 %
    assert b["experts"] / b["total"] == pytest.approx(0.526, abs=0.002)
    assert w.L * qkv / b["total"] == pytest.approx(0.146, abs=0.002)
    assert b["kv_read"] / b["total"] == pytest.approx(0.117, abs=0.002)
    assert w.V * w.H * 2 / b["total"] == pytest.approx(0.090, abs=0.002)


def test_256k_context_is_dominated_by_the_kv_read():
    w = W.M30B_256K
    b = metrics.step_bytes(w, W.context_lengths(w), [8] * w.L)
    assert b["kv_read"] / b["total"] == pytest.approx(0.81, abs=0.01)


def test_accounting_invariants():
    w = W.M30B_BS8
    pos = np.array([1000, 2000, 3000, 4000, 5000, 6000, 7000, 8000])
    one = metrics.step_bytes(w, pos, [20] * w.L)
    more = metrics.step_bytes(w, pos, [21] * w.L)
    # one more distinct expert in every layer adds exactly one expert's three matrices per layer
    assert more["total"] - one["total"] == w.L * 3 * w.I * w.H * 2
    # each cached position adds one K and one V row per layer; each new token writes one of each
    longer = metrics.step_bytes(w, pos + 1, [20] * w.L)
    kv_row = w.L * 2 * w.nkv * w.d * 2
    assert longer["kv_read"] - one["kv_read"] == len(pos) * kv_row
    assert one["kv_write"] == len(pos) * kv_row
    # weights are counted once per step, not once per token
    single = metrics.step_bytes(w, pos[:1], [20] * w.L)
    assert one["dense_weights"] == single["dense_weights"]
    assert metrics.sol_tok_s(one["total"], 8, 8e12) == pytest.approx(8 * 8e12 / one["total"])
