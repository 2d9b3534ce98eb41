"""The seeded input generator: its published definitions and its host/device agreement."""
import numpy as np
import pytest

import synth
from synth import workloads as W


def _splitmix_ref(x):
    # SplitMix64 (Steele, Lea & Flood 2014): state += golden; mix the state
    M = (1 << 64) - 1
    z = (x + 0x9E3779B97F4A7C15) & M
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
    return z ^ (z >> 31)


def test_splitmix_matches_published_definition():
    lib = synth.host_lib()
    seed, t = 12345, synth.tid(synth.SYNTH_QKV, 3, 0)
    key = _splitmix_ref(_splitmix_ref(seed) ^ t)
    assert lib.synth_key(seed, t) == key
    for n in (0, 1, 77, 10 ** 9):
        assert lib.synth_draw(key, n) == _splitmix_ref((key + n * 0x9E3779B97F4A7C15) & ((1 << 64) - 1))
    # Irwin-Hall(12) from the 16-bit quarters of draws 3i..3i+2
    i = 5
    parts = [lib.synth_draw(key, 3 * i + j) for j in range(3)]
    s = sum((p >> (16 * q)) & 0xFFFF for p in parts for q in range(4))
    assert lib.synth_normal(key, i) == np.float32((s - 6 * 65536) / 65536.0)


def test_normal_moments_and_bf16_values():
    z = synth.fill_bf16(3, synth.SYNTH_K, 0, 0, 200000, 1.0)
    f = synth.bf16_bits_to_f32(z).astype(np.float64)
    assert abs(f.mean()) < 0.01 and abs(f.std() - 1.0) < 0.01 and np.abs(f).max() <= 6.0
    w = synth.bf16_bits_to_f32(synth.fill_bf16(3, synth.SYNTH_QKV, 0, 0, 200000, 0.02)).astype(np.float64)
    assert abs(w.std() - 0.02) < 3e-4
    g = synth.bf16_bits_to_f32(synth.fill_bf16(3, synth.SYNTH_GAIN, 1, 0, 100000, 0.05, 1.0)).astype(np.float64)
    assert abs(g.mean() - 1.0) < 2e-3 and abs(g.std() - 0.05) < 2e-3


def test_streams_are_deterministic_and_distinct():
    a = synth.fill_bf16(9, synth.SYNTH_O, 2, 0, 1000, 0.02)
    assert np.array_equal(a, synth.fill_bf16(9, synth.SYNTH_O, 2, 0, 1000, 0.02))
    assert np.array_equal(a[300:], synth.fill_bf16(9, synth.SYNTH_O, 2, 0, 700, 0.02, start=300))
    assert not np.array_equal(a, synth.fill_bf16(9, synth.SYNTH_O, 3, 0, 1000, 0.02))
    assert not np.array_equal(a, synth.fill_bf16(10, synth.SYNTH_O, 2, 0, 1000, 0.02))


def test_workload_recipes():
    w = W.SMALL
    ctx = W.context_lengths(w)
    assert ctx.shape == (8,) and ctx.min() >= 64 and ctx.max() <= 2048
    bt, npg = W.page_tables(w, ctx, w.steps)
    used = bt[bt >= 0]
    assert sorted(used.tolist()) == list(range(npg))  # every page of the pool used exactly once
    for b in range(w.B):
        assert (bt[b] >= 0).sum() == -(-(int(ctx[b]) + w.steps) // w.page)
    bias = W.router_bias(W.M30B_BS8_ZIPF)
    assert bias.shape == (48, 128) and np.allclose(bias.mean(1), 0, atol=1e-5)
    p = np.exp(bias[0].astype(np.float64))
    p /= p.sum()
    top = np.sort(p)[::-1]
    assert top[0] / top[1] == pytest.approx(2 ** 1.2, rel=1e-4)  # Zipf(1.2): p(1) / p(2) = 2^1.2
    assert W.router_bias(W.M30B_BS1) is None


@pytest.mark.gpu
def test_device_generator_matches_host():
    import torch

    w = W.TINY
    m_dev = synth.device_model(w)
    m_host = synth.host_model(w)
    for k, v in m_host.items():
        got = m_dev[k].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, v), k
    ctx = np.array([32], np.int32)
    bt, npg = W.page_tables(w, ctx, 4)
    Kd, Vd = synth.device_kv(w, ctx, bt, npg)
    Kh, Vh = synth.host_kv(w, ctx, bt, npg)
    assert np.array_equal(Kd.view(torch.int16).cpu().numpy().view(np.uint16), Kh)
    assert np.array_equal(Vd.view(torch.int16).cpu().numpy().view(np.uint16), Vh)
