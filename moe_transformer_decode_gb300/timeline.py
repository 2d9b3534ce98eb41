"""Per-task timeline of one decode step, from the kernel's own trace (mk_enable_trace).

Each task records when its block took it, how long it waited for the tasks it depends on, and
how long it ran from the end of that wait to its release. From those records this module builds
the phase times of a layer (when each op kind's tasks became ready and when the last one ended)
and the share of SM time in which an SM was running no task at all: the cost of the dependent
hand-offs between SMs that a persistent kernel pays instead of launch gaps.
"""
from __future__ import annotations

import numpy as np

from . import binding as B

OP_NAMES = {1: "router", 2: "qkv", 3: "attn", 4: "gu", 5: "o", 6: "down", 7: "lm", 8: "combine"}

TRACE_DTYPE = np.dtype([("t", "<u8"), ("wait", "<u4"), ("run", "<u4"), ("sm", "<u2"), ("op", "<u2"),
                        ("layer", "<u2"), ("pad", "<u2"), ("a", "<i4"), ("b", "<i4")])
assert TRACE_DTYPE.itemsize == 32


def trace_buffer(max_tasks: int, device="cuda"):
    """A device buffer for mk_enable_trace: 16 header bytes (the entry count) + 32 bytes a task."""
    import torch

    return torch.zeros(16 + 32 * max_tasks, dtype=torch.uint8, device=device)


def decode(raw: np.ndarray) -> np.ndarray:
    """The trace entries of the last traced step from the buffer's bytes (uint8 array)."""
    n = int(raw[:8].view(np.uint64)[0])
    cap = (raw.size - 16) // 32
    return raw[16:16 + 32 * min(n, cap)].view(TRACE_DTYPE)


def summarize(e: np.ndarray, n_layers: int) -> dict:
    """Phase times of the middle layers (µs from the end of the previous layer, which is the
    last O-proj or expert-down release of that layer), and SM idle shares over the step."""
    t0 = e["t"].min()
    start = (e["t"] - t0) / 1e3
    ready = start + e["wait"] / 1e3
    end = ready + e["run"] / 1e3
    step_us = float(end.max())
    layer_end = np.array([end[(e["layer"] == l) & np.isin(e["op"], (5, 6))].max() for l in range(n_layers)])
    mid = range(max(1, n_layers // 4), max(2, n_layers - n_layers // 4))
    phases = {}
    for op, name in OP_NAMES.items():
        if op == 7:
            continue
        rows = []
        for l in mid:
            m = (e["layer"] == l) & (e["op"] == op)
            if m.any():
                base = layer_end[l - 1]
                rows.append((ready[m].min() - base, ready[m].max() - base, end[m].max() - base))
        if rows:
            r = np.mean(np.array(rows), axis=0)
            phases[name] = {"first_ready_us": round(float(r[0]), 2), "last_ready_us": round(float(r[1]), 2),
                            "last_end_us": round(float(r[2]), 2)}
    # an SM is busy while one of its tasks runs (between the end of its wait and its release)
    n_sm = int(e["sm"].max()) + 1
    busy = np.zeros(n_sm)
    for s in range(n_sm):
        m = e["sm"] == s
        iv = sorted(zip(ready[m], end[m]))
        tot, cur0, cur1 = 0.0, None, None
        for a, b in iv:
            if cur1 is None or a > cur1:
                if cur1 is not None:
                    tot += cur1 - cur0
                cur0, cur1 = a, b
            else:
                cur1 = max(cur1, b)
        if cur1 is not None:
            tot += cur1 - cur0
        busy[s] = tot
    idle = 1.0 - busy / step_us
    layer_us = float(np.mean(np.diff(layer_end)[mid.start:mid.stop - 1])) if n_layers > 2 else float("nan")
    return {"step_us": round(step_us, 1), "layer_us": round(layer_us, 2), "phases": phases,
            "sm_idle_share": {"mean": round(float(idle.mean()), 3), "min": round(float(idle.min()), 3),
                              "max": round(float(idle.max()), 3)},
            "tasks": int(e.size)}


def trace_step(dc, w, tokens, positions, K, V, logits, next_tokens, max_tasks: int = 200000) -> np.ndarray:
    """Runs one traced step through the context and returns its trace entries (tracing is off
    again afterwards)."""
    buf = trace_buffer(max_tasks)
    B.mk_enable_trace(dc.ctx, buf)
    try:
        dc.step(tokens, positions, K, V, logits, next_tokens)
        dc.sync()
    finally:
        B.mk_enable_trace(dc.ctx, None)
    return decode(buf.cpu().numpy())
