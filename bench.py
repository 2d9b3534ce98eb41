"""Decode throughput of the single-kernel MoE decode step on one GB300 (or N replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one decode step of the whole batch: embedding, 48 parallel layers (QKV + RoPE +
paged KV append, GQA paged attention, O-proj, router top-k, SwiGLU experts with weighted
combine, residual + RMSNorm) and LM head + argmax, one persistent kernel launch. The
default workload is the 30B-total / 3.3B-active-shaped model at batch 1 with 8K context;
weights, KV pages and tokens are seeded synthetic values generated on the device.

The JSON line reports tok/s (device-timed, greedy tokens fed back on the device), the
same metric end to end through the C ABI from pinned host buffers, the fraction of HBM
speed-of-light, the CPU oracle's throughput on a bounded sample, and the clocks seen.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "moe30b_a3b_bs1_ctx8k"
METRIC = "decode tok/s (BS=1, BS=8 @8K ctx) and % of GB300 HBM speed-of-light"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() in ("active", "1"):
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the decode kernel from the committed ncu capture,
    if it was taken on this workload and on the kernel source as it stands; else None."""
    here = os.path.dirname(os.path.abspath(__file__))
    try:
        rec = json.load(open(os.path.join(here, "profiles", "mk_decode_kernel_traffic.json")))
        h = hashlib.sha256()
        for f in ("mk_kernel.cu", "mk_internal.h"):
            h.update(open(os.path.join(here, "moe_transformer_decode_gb300", "csrc", f), "rb").read())
    except (OSError, ValueError):
        return None
    if rec.get("workload") != workload or rec.get("source_sha256") != h.hexdigest():
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def setup_gpu(w, capacity, device):
    import torch

    import synth
    from moe_transformer_decode_gb300.context import DecodeContext
    from synth import workloads as W

    ctx = W.context_lengths(w)
    bt, num_pages = W.page_tables(w, ctx, capacity)
    model = synth.device_model(w, device)
    bias = W.router_bias(w)
    if bias is not None:
        model["router_bias"] = torch.as_tensor(bias, device=device)
    K, V = synth.device_kv(w, ctx, bt, num_pages, device)
    dc = DecodeContext(w, model, max_batch=w.B, max_pages_per_seq=bt.shape[1])
    bt_d = torch.as_tensor(bt, device=device)
    dc.schedule(ctx, bt_d)
    return dc, model, K, V, ctx, bt_d


def distinct_experts(dc, w):
    ids = dc.activations()["topk_ids"].cpu().numpy()  # [L][B][k]
    return np.array([len(np.unique(ids[l])) for l in range(w.L)])


ORACLE_BUDGET_S = 30.0  # CPU work the oracle timing may take, per arm


def oracle_protocol(w, max_steps: int, budget_s: float = ORACLE_BUDGET_S):
    """The one timing protocol of the CPU oracle (both the main line's cpu_baseline and the
    reference arm): one warm-up step (it synthesises and caches the weights it touches), one
    step to size the sample, then as many steps as fit the budget (at most max_steps, at least
    one), all at the workload's first position. Returns (seconds per step, steps timed, threads,
    sample description)."""
    import oracle
    from synth import workloads as W

    ctx = np.asarray(W.context_lengths(w), np.int32)
    tokens = W.first_tokens(w)
    src = oracle.SynthSource(w, ctx, 4, W.router_bias(w), keep_all_experts=True)
    oracle.decode_step(w, src, tokens, ctx)
    t0 = time.perf_counter()
    oracle.decode_step(w, src, tokens, ctx)
    first = time.perf_counter() - t0
    timed = max(1, min(max_steps, int(budget_s / max(first, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(timed):
        oracle.decode_step(w, src, tokens, ctx)
    per_step = (time.perf_counter() - t0) / timed
    sample = (f"{timed} oracle decode step(s) of {w.name} (batch {w.B}, all {w.L} layers and the LM head) at the "
              f"workload's first position, after one warm-up step that synthesises and caches the weights it "
              f"touches and one sizing step; KV values synthesised on read; at most {budget_s:.0f} s of CPU work")
    return per_step, timed, oracle.threads(), sample


def bench_config(w, mode: str, world: int) -> dict:
    """The `config` object of both arms' lines (identical keys and values for one workload)."""
    from synth import workloads as W

    ctx = W.context_lengths(w)
    return {"workload": w.name, "batch": w.B, "ctx_start": int(np.max(ctx)), "ctx_min": int(np.min(ctx)),
            "layers": w.L, "experts": f"{w.E} top-{w.topk}", "routing": w.routing, "mode": mode,
            "parallelism": "replicas" if world > 1 else "single_gpu",
            "l2": "inputs larger than L2: each step streams its weights and KV once (GBs vs 129 MB of L2)"}


def ranks_max(x: float, device: str) -> float:
    """The maximum of x over all ranks (a job takes as long as its slowest rank); x itself when
    no process group is up or it has one rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tok_s(batch: int, steps: int, seconds: float, world: int) -> float:
    """Decode tokens per second of the whole job: every rank decodes `batch` tokens per step
    (independent replicas, weak scaling), timed by the slowest rank."""
    return batch * steps * world / seconds


def run_reference(args, w, rank):
    """Reference arm: the CPU oracle as it stands, on this workload, rank 0 only."""
    if rank != 0:
        return
    t0 = time.perf_counter()
    per_step, timed, cores, sample = oracle_protocol(w, args.steps)
    value = w.B / per_step
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "steps_timed": timed, "warmup": args.warmup, "ms_per_step": 1e3 * per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded SplitMix64/Irwin-Hall bf16 weights and KV)",
            "config": bench_config(w, args.mode, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0}
    print(json.dumps(line), flush=True)


def measure(w, args, device, world):
    """Timed greedy decode (device-side token feedback) and the end-to-end loop through the C ABI
    for workload w; returns the per-workload record (the headline line's fields, or one entry of
    by_config)."""
    import torch

    from moe_transformer_decode_gb300 import binding as B
    from moe_transformer_decode_gb300 import metrics
    from synth import workloads as W

    import torch.distributed as dist

    capacity = args.warmup + args.steps + args.e2e_steps + 16
    if capacity > w.steps:
        w = w.with_(steps=capacity)
    dc, model, K, V, ctx, bt_d = setup_gpu(w, capacity, device)
    if args.mode == "per_op":
        dc.set_mode(B.MK_MODE_PER_OP)
    launches_per_step = dc.launch_info()[2]
    tokens0 = torch.as_tensor(W.first_tokens(w), device=device)
    pos = torch.as_tensor(ctx, device=device)
    logits = torch.empty((w.B, w.V), dtype=torch.float32, device=device)
    toks = torch.empty((max(args.steps, args.warmup), w.B), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    # warm-up (greedy, token fed back on the device)
    dc.greedy(args.warmup, tokens0, pos, K, V, logits, toks, stream.cuda_stream)
    dc.sync()
    done = args.warmup
    last_tok = toks[args.warmup - 1].clone()
    pos_t = pos + done

    # timed region: K steps, one launch each; weights streamed per step (6+ GB) exceed L2
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(int(str(device).split(":")[-1])) as clk:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        dc.greedy(args.steps, last_tok, pos_t, K, V, logits, toks, stream.cuda_stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    dc.sync()
    ms = ranks_max(ev0.elapsed_time(ev1), device)
    if world > 1:
        dist.barrier()
    positions_timed = np.asarray(ctx, np.int64)[None, :] + done + np.arange(args.steps)[:, None]
    done += args.steps
    last_tok = toks[args.steps - 1].clone()

    # distinct experts per layer, from this run's own routing (a few single steps)
    de = []
    nxt = torch.empty_like(last_tok)
    for i in range(4):
        dc.step(last_tok, pos + done, K, V, logits, nxt, stream.cuda_stream)
        dc.sync()
        de.append(distinct_experts(dc, w))
        last_tok.copy_(nxt)
        done += 1
    de = np.mean(de, axis=0)

    # end to end through the C ABI: pinned host tokens/positions -> device, one step, the
    # greedy token back to pinned host memory, every step
    h_tok = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h_pos = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h_out = torch.empty(w.B, dtype=torch.int32).pin_memory()
    d_tok = torch.empty(w.B, dtype=torch.int32, device=device)
    d_pos = torch.empty(w.B, dtype=torch.int32, device=device)
    d_out = torch.empty(w.B, dtype=torch.int32, device=device)
    h_tok.copy_(last_tok.cpu())
    ctx_np = np.asarray(ctx, np.int32)
    n_e2e = args.e2e_steps
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        h_pos.numpy()[:] = ctx_np + done + i
        d_tok.copy_(h_tok, non_blocking=True)
        d_pos.copy_(h_pos, non_blocking=True)
        dc.step(d_tok, d_pos, K, V, None, d_out, stream.cuda_stream)
        h_out.copy_(d_out, non_blocking=True)
        stream.synchronize()
        h_tok.copy_(h_out)
    e2e_s = time.perf_counter() - t0
    dc.sync()
    e2e_s = ranks_max(e2e_s, device)
    timeline_summary = None
    if getattr(args, "timeline", False):
        # after every timed region: two traced steps (the first warms the trace path), per-op phase
        # times and SM idle shares from the kernel's own per-task records
        from moe_transformer_decode_gb300 import timeline

        for i in range(2):
            h_pos.numpy()[:] = ctx_np + done + n_e2e + i
            d_pos.copy_(h_pos)
            ent = timeline.trace_step(dc, w, d_tok, d_pos, K, V, None, d_out)
        timeline_summary = timeline.summarize(ent, w.L)
    dc.close()
    del dc, model, K, V
    torch.cuda.empty_cache()

    hbm_gbs, peak_kind = measured_peaks()
    sol = [metrics.step_bytes(w, positions_timed[i], de) for i in range(args.steps)]
    bytes_per_step = float(np.mean([x["total"] for x in sol]))
    kv_share = float(np.mean([(x["kv_read"] + x["kv_write"]) / x["total"] for x in sol]))
    ms_step = ms / args.steps
    achieved = bytes_per_step / (ms_step * 1e-3) / 1e9
    return {
        "workload": w.name, "value": whole_job_tok_s(w.B, args.steps, ms * 1e-3, world), "unit": "tok/s",
        "ms_per_step": ms_step, "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": measured_traffic(w.name), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": bytes_per_step / launches_per_step,
                     "distinct_experts_per_layer": float(np.mean(de))},
        "sol": {"bytes_per_step": bytes_per_step, "frac_of_nominal_8tbs": bytes_per_step / (ms_step * 1e-3) / 8.0e12,
                "frac_of_measured": achieved / hbm_gbs, "kv_share_of_bytes": kv_share,
                "sol_tok_s_measured_bw": metrics.sol_tok_s(bytes_per_step, w.B, hbm_gbs * 1e9)},
        "e2e": {"value": whole_job_tok_s(w.B, n_e2e, e2e_s, world), "unit": "tok/s", "h2d_bytes_per_step": 2 * 4 * w.B,
                "d2h_bytes_per_step": 4 * w.B},
        "clocks": clk.summary(),
        "config": bench_config(w, args.mode, world),
        **({"timeline": timeline_summary} if timeline_summary is not None else {}),
    }


# the metric's other half (batch 8 at 1K-8K contexts, both routing modes) and the long context,
# measured in the same process after the headline workload
EXTRA_WORKLOADS = ("moe30b_a3b_bs8_ctx1k8k", "moe30b_a3b_bs8_ctx1k8k_zipf", "moe30b_a3b_bs1_ctx256k")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only (no by_config lines)")
    ap.add_argument("--mode", default="megakernel", choices=["megakernel", "per_op"])
    ap.add_argument("--timeline", action="store_true",
                    help="after the timed region, trace two steps and print per-op phase times and SM idle "
                         "shares (stderr)")
    args = ap.parse_args()

    from synth import workloads as W

    w = W.ALL[args.workload]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(device))
    assert args.warmup >= 3, "at least 3 warm-up steps"
    head = measure(w, args, device, world)
    if rank == 0 and "timeline" in head:
        print("timeline " + json.dumps({"workload": w.name, **head["timeline"]}), file=sys.stderr, flush=True)
    line = {"metric": METRIC, "value": head["value"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64/Irwin-Hall bf16 weights and KV, generated on the device)",
            "config": head["config"], "gpu_launches": head["gpu_launches"], "roofline": head["roofline"],
            "sol": head["sol"], "e2e": head["e2e"], "clocks": head["clocks"]}
    if not args.no_extra and args.workload == DEFAULT_WORKLOAD:
        line["by_config"] = {}
        for name in EXTRA_WORKLOADS:
            r = measure(W.ALL[name], args, device, world)
            line["by_config"][name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "gpu_launches", "roofline",
                                                         "sol", "e2e", "clocks", "config")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per_step, timed, cores, sample = oracle_protocol(w, args.steps)
        line["cpu_baseline"] = {"value": w.B / per_step, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
