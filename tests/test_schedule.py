"""Host scheduler (no GPU): every unit of work of the step is planned exactly once, each
SM's list follows the global dependency order (so no counter wait can deadlock), and the
bytes are spread evenly over the SMs."""
import numpy as np
import pytest

from moe_transformer_decode_gb300 import binding as B
from synth import workloads as W

OP_ROUTER, OP_QKV, OP_ATTN, OP_GU, OP_O, OP_DOWN, OP_LM, OP_COMBINE = range(1, 9)
RANK = {OP_COMBINE: -1, OP_ROUTER: 0, OP_QKV: 1, OP_GU: 2, OP_ATTN: 3, OP_DOWN: 4, OP_O: 5, OP_LM: 6}


def cfg_of(w, max_pages):
    return B.mk_model_cfg(w.L, w.H, w.nq, w.nkv, w.d, w.E, w.topk, w.I, w.V, 16, w.B, max_pages, w.rope_theta, w.eps)


def rows_per_stage(K):
    kw = min(K, 2048) // 256
    return 8 * (8 // kw)


def _ranges(t):
    return np.concatenate([np.arange(a, a + b) for a, b in zip(t["a"], t["b"])])


@pytest.mark.parametrize("w,n_sm", [(W.TINY, 148), (W.SMALL, 152), (W.M30B_BS1, 148), (W.M30B_BS8, 152),
                                    (W.TINY.with_(B=3, ctx_lo=0, ctx_hi=70), 7)])
def test_plan_covers_everything_once_in_dependency_order(w, n_sm):
    ctx = W.context_lengths(w)
    max_pages = int(np.max(ctx)) // 16 + 64
    info, tasks, begin, load = B.mk_plan_schedule(cfg_of(w, max_pages), n_sm, ctx)
    assert begin[0] == 0 and begin[-1] == info.n_tasks and np.all(np.diff(begin) >= 0)
    # global order inside every SM list: (layer, opcode rank) never decreases
    for s in range(n_sm):
        t = tasks[begin[s]:begin[s + 1]]
        key = t["layer"].astype(np.int64) * 10 + np.array([RANK[o] for o in t["op"]], dtype=np.int64)
        assert np.all(np.diff(key) >= 0), f"SM {s} list out of order"
    maxa = min(w.B * w.topk, w.E)
    upg = (w.nq // w.nkv + 2) * (w.d // 8)
    # batch 5-8: the input of every layer past the first, and the final norm's, is combined by
    # slices of 16 columns, each exactly once
    cb = tasks[tasks["op"] == OP_COMBINE]
    if w.B > 4:
        for l in range(1, w.L + 1):
            c = cb[cb["layer"] == l]
            assert sorted(c["a"].tolist()) == list(range(w.H // 16)) and np.all(c["b"] == w.H // 16)
        assert np.all(cb["layer"] >= 1)
    else:
        assert cb.size == 0
    for l in range(w.L):
        t = tasks[tasks["layer"] == l]
        r = t[t["op"] == OP_ROUTER]
        assert sorted(_ranges(r).tolist()) == list(range(w.E))
        assert (r["flags"] & 1).sum() == 1  # exactly one task stores x of the layer
        q = t[t["op"] == OP_QKV]
        assert sorted(_ranges(q).tolist()) == list(range(w.nkv * upg))
        assert np.all(q["a"] // upg == q["c"]) and np.all((q["a"] + q["b"] - 1) // upg == q["c"])
        at = t[t["op"] == OP_ATTN]
        keys = list(zip(at["a"].tolist(), at["b"].tolist(), at["c"].tolist()))
        assert len(set(keys)) == len(keys)
        for b in range(w.B):
            n = None
            for g in range(w.nkv):
                ch = sorted(c for (bb, gg, c) in keys if bb == b and gg == g)
                assert ch == list(range(len(ch))) and len(ch) >= 1
                assert n is None or n == len(ch)
                n = len(ch)
        # gate/up: task k of n takes an equal share of the routed experts' units (64 gate rows
        # and their up rows each), so the tasks are k = 0 .. n - 1 of n, at most one per SM and
        # no more than there are units
        g = t[t["op"] == OP_GU]
        assert sorted(g["a"].tolist()) == list(range(len(g))) and np.all(g["b"] == len(g))
        assert 1 <= len(g) <= min(n_sm, maxa * (w.I // 64))
        o = t[t["op"] == OP_O]
        rs_o = rows_per_stage(w.nq * w.d)  # O tasks: whole row blocks (the last may be short)
        assert sorted(_ranges(o).tolist()) == list(range(w.H))
        assert np.all((o["b"] % rs_o == 0) | (o["a"] + o["b"] == w.H))
        # down: one task per (128-row block, partial) unit; a partial takes the experts of rank
        # j, j + parts, ..., so every unit of a layer has the same share of the routed experts
        dn = t[t["op"] == OP_DOWN]
        parts = min(4 if w.B <= 4 else 9, maxa)  # expert-down partials: 4 at batch <= 4, 9 at batch 8
        assert sorted(_ranges(dn).tolist()) == list(range((w.H // 128) * parts)) and np.all(dn["b"] == 1)
    lm = tasks[tasks["op"] == OP_LM]
    assert sorted(_ranges(lm).tolist()) == list(range(w.V))
    assert np.all(lm["flags"] & 2) and len(lm) == info.n_lm_sm and sorted(lm["c"].tolist()) == list(range(len(lm)))
    owners = np.searchsorted(begin, np.nonzero(tasks["op"] == OP_LM)[0], side="right")
    assert len(set(owners.tolist())) == len(lm), "two LM tasks on one SM"


@pytest.mark.parametrize("w,n_sm", [(W.M30B_BS1, 148), (W.M30B_BS1, 152), (W.M30B_BS8, 152)])
def test_plan_balances_bytes_over_sms(w, n_sm):
    """Planned bytes are even over the SMs of each partition (the partitions themselves are
    sized by the branches' critical paths, not their bytes)."""
    info, tasks, begin, load = B.mk_plan_schedule(cfg_of(w, 600), n_sm, W.context_lengths(w))
    na = info.n_attn_sm
    for part in ((load[:na], load[na:]) if na < n_sm else (load,)):
        assert part.max() / part.mean() < 1.03


def test_plan_rejects_bad_arguments():
    cfg = cfg_of(W.TINY, 4)
    for n_sm, lens in ((148, [64]), (148, [-1]), (0, [3])):
        with pytest.raises(B.MkError):
            B.mk_plan_schedule(cfg, n_sm, np.array(lens, np.int32))


@pytest.mark.parametrize("w,n_sm", [(W.M30B_BS1, 152), (W.M30B_BS8, 152), (W.SMALL, 152), (W.TINY, 152),
                                    (W.TINY, 7)])
def test_plan_splits_branches_over_disjoint_sms(w, n_sm):
    """At batch 1, attention tasks (attention, O-proj) and expert-branch tasks (router, gate/up,
    down) sit on disjoint SM partitions, and QKV (which needs only the layer's input) spreads
    over every SM, at most one task each; larger batches and very small grids do not split."""
    ctx = W.context_lengths(w)
    info, tasks, begin, load = B.mk_plan_schedule(cfg_of(w, int(np.max(ctx)) // 16 + 64), n_sm, ctx)
    na = info.n_attn_sm
    owner = np.searchsorted(begin, np.arange(info.n_tasks), side="right") - 1
    attn = np.isin(tasks["op"], [OP_ATTN, OP_O])
    moe = np.isin(tasks["op"], [OP_ROUTER, OP_GU, OP_DOWN])
    if n_sm < 8 or w.B > 1:
        assert na == n_sm
        return
    assert 0 < na < n_sm
    assert np.all(owner[attn] < na) and np.all(owner[moe] >= na)
    for l in (0, w.L - 1):
        q = owner[(tasks["op"] == OP_QKV) & (tasks["layer"] == l)]
        assert np.bincount(q, minlength=n_sm).max() <= 1
    if w.H < 2048:  # the small models have fewer tasks than SMs
        return
    # every SM of a partition gets work of its branch in every layer, no SM takes two attention
    # chunks or two O-proj tasks of one layer (a second one would double that phase on its SM),
    # and the down units spread evenly over the expert SMs
    for l in (0, w.L - 1):
        lay = tasks["layer"] == l
        assert set(owner[attn & lay].tolist()) == set(range(na))
        assert set(owner[moe & lay].tolist()) == set(range(na, n_sm))
        for op in (OP_ATTN, OP_O):
            assert np.bincount(owner[(tasks["op"] == op) & lay], minlength=n_sm).max() == 1, op
        dn = owner[(tasks["op"] == OP_DOWN) & lay]
        assert np.bincount(dn, minlength=n_sm).max() == -(-len(dn) // (n_sm - na))


@pytest.mark.parametrize("ctx_len", [100, 1000, 4096, 8192, 16384, 30000])
def test_attention_chunks_fit_the_attention_partition(ctx_len):
    """At batch 1 with the branches partitioned, the attention chunks of a layer are whole ring
    stages (4 pages at d = 128), no more than one per attention SM, and their pages tile the
    context exactly; every page of every chunk but the last is a full chunk's worth."""
    w = W.M30B_BS1.with_(ctx_lo=ctx_len, ctx_hi=ctx_len, L=2)
    ctx = W.context_lengths(w)
    info, tasks, begin, load = B.mk_plan_schedule(cfg_of(w, ctx_len // 16 + 64), 152, ctx)
    if info.n_attn_sm == 152:  # the attention bytes dominate: no partition at this length
        return
    att = tasks[(tasks["op"] == OP_ATTN) & (tasks["layer"] == 0)]
    owner = np.searchsorted(begin, np.nonzero((tasks["op"] == OP_ATTN) & (tasks["layer"] == 0))[0], side="right") - 1
    assert len(att) <= info.n_attn_sm and len(set(owner.tolist())) == len(att)
    npg = -(-ctx_len // 16)
    for g in range(w.nkv):
        ch = sorted(att[att["b"] == g]["c"].tolist())
        assert ch == list(range(len(ch))) and len(ch) == info.max_chunks
    # chunk size: a whole number of 4-page stages, and the chunks cover the pages exactly
    cp = -(-npg // info.max_chunks)
    cp = -(-cp // 4) * 4
    assert (info.max_chunks - 1) * cp < npg <= info.max_chunks * cp


def test_unpartitioned_o_proj_stays_balanced_per_phase():
    """Without an SM partition, O-proj stays balanced per phase (one or two tasks per SM), and
    the SMs that hold no expert-down unit of the layer (144 units on 152 SMs at batch 8) are
    among those taking the phase's extra tasks. (The tie-break by bytes in the layer, which
    decides the rest, is measured in the timings, not pinned here.)"""
    w, n_sm = W.M30B_BS8, 152
    ctx = W.context_lengths(w)
    info, tasks, begin, load = B.mk_plan_schedule(cfg_of(w, int(np.max(ctx)) // 16 + 64), n_sm, ctx)
    assert info.n_attn_sm == n_sm
    owner = np.searchsorted(begin, np.arange(info.n_tasks), side="right") - 1
    for l in (1, w.L // 2, w.L - 1):
        lay = tasks["layer"] == l
        n_o = np.bincount(owner[lay & (tasks["op"] == OP_O)], minlength=n_sm)
        n_dn = np.bincount(owner[lay & (tasks["op"] == OP_DOWN)], minlength=n_sm)
        assert n_o.min() >= 1 and n_o.max() - n_o.min() <= 1
        no_down = np.nonzero(n_dn == 0)[0]
        assert len(no_down) == n_sm - (w.H // 128) * 9
        assert np.all(n_o[no_down] == n_o.max())


def test_batch1_long_context_takes_one_qkv_task_per_sm():
    """At batch 1 without a partition (the KV of a long context dominates), a layer's QKV units
    go out as at most one task per SM."""
    w = W.M30B_256K.with_(L=2)
    ctx = W.context_lengths(w)
    info, tasks, begin, load = B.mk_plan_schedule(cfg_of(w, int(np.max(ctx)) // 16 + 64), 152, ctx)
    assert info.n_attn_sm == 152
    owner = np.searchsorted(begin, np.arange(info.n_tasks), side="right") - 1
    for l in range(w.L):
        q = owner[(tasks["op"] == OP_QKV) & (tasks["layer"] == l)]
        assert np.bincount(q, minlength=152).max() == 1
