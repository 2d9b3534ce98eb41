"""The trace decoder (moe_transformer_decode_gb300/timeline.py) on hand-built records whose
phase times and idle shares are known exactly."""
import numpy as np

from moe_transformer_decode_gb300 import timeline as T


def _rec(rows):
    e = np.zeros(len(rows), T.TRACE_DTYPE)
    for i, (sm, op, layer, t_us, wait_us, run_us) in enumerate(rows):
        e[i] = (int(t_us * 1000), int(wait_us * 1000), int(run_us * 1000), sm, op, layer, 0, 0, 0)
    return e


def test_decode_reads_the_count_and_the_entries():
    e = _rec([(0, 2, 0, 0, 1, 2), (1, 5, 0, 1, 0, 3)])
    raw = np.zeros(16 + 32 * 4, np.uint8)
    raw[:8] = np.frombuffer(np.uint64(2).tobytes(), np.uint8)
    raw[16:16 + 64] = e.view(np.uint8)
    d = T.decode(raw)
    assert d.size == 2 and np.array_equal(d, e)
    raw[:8] = np.frombuffer(np.uint64(9).tobytes(), np.uint8)  # more than the buffer holds
    assert T.decode(raw).size == 4


def test_idle_share_and_phases():
    # 2 SMs, 4 layers of O-proj (op 5) and down (op 6) tasks; layer l ends at 10 (l + 1) us.
    rows = []
    for l in range(4):
        t = 10.0 * l
        rows.append((0, 2, l, t, 2.0, 3.0))       # QKV: ready at t + 2, runs until t + 5
        rows.append((0, 5, l, t + 5, 1.0, 4.0))   # O-proj: ready t + 6, ends t + 10
        rows.append((1, 6, l, t, 4.0, 6.0))       # down: ready t + 4, ends t + 10
    s = T.summarize(_rec(rows), 4)
    assert s["step_us"] == 40.0 and s["layer_us"] == 10.0
    # SM 0 runs [t + 2, t + 5] and [t + 6, t + 10] of every layer: idle 3 of 10 us;
    # SM 1 runs [t + 4, t + 10]: idle 4 of 10 us
    assert s["sm_idle_share"] == {"mean": 0.35, "min": 0.3, "max": 0.4}
    # middle layers (1 and 2): phases relative to the previous layer's end
    assert s["phases"]["qkv"] == {"first_ready_us": 2.0, "last_ready_us": 2.0, "last_end_us": 5.0}
    assert s["phases"]["o"]["last_end_us"] == 10.0 and s["phases"]["down"]["first_ready_us"] == 4.0
