#!/usr/bin/env python
"""Benchmark of the greedy, lossless speculative-decoding verify step on GB300.

Metric: committed tokens/s of speculative decoding (excluding prefill), the
verify-step latency, and the fraction of the HBM roofline reached.

Default workload: the DeepSeek-3B-MoE-shaped bf16 decoder at batch 1 (12
layers, hidden 1280, 10x128 MHA, 64 routed experts top-6 + 2 shared of width
896, vocab 129,280), a prompt of 256 N(0,1) visual rows + 16 token ids, K = 3
drafts from a seeded synthetic drafter whose per-position match probability
is 0.576, 1,085-token pages. Weights are random (N(0, 0.02), seed 0).

One process per GPU; with torchrun each rank runs an independent replica (the
step does not shard) and rank 0 prints one JSON line.

  python bench.py [--steps K] [--warmup W] [--impl reference] [--workload NAME]
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

os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as syn  # noqa: E402

DEFAULT_WORKLOAD = "moe3b_bf16_b1"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--profile-steps", type=int, default=64)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small same-shape cases for ncu captures)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(ms: float, committed: int, device=None):
    """Replica aggregation across ranks: the slowest rank's time and the sum of
    committed tokens (the step has no collective; ranks are independent)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, committed
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    c = torch.tensor([int(committed)], dtype=torch.int64, device=device)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return float(t.item()), int(c.item())


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# --------------------------------------------------------------------------- #
# algorithmic bytes per kernel class (weights actually read + KV + activations)
# --------------------------------------------------------------------------- #
def welt(cfg) -> int:
    return {syn.F32: 4, syn.BF16: 2, syn.FP8: 1}[cfg.wdtype]


def side_elt(cfg) -> int:
    return 4 if cfg.wdtype == syn.F32 else 2


def class_bytes(cfg, stats: dict, T: int, ctx_sum: float, n_steps: int) -> dict:
    """Algorithmic bytes (summed over the profiled launches) per kernel class.
    ctx_sum = sum over profiled steps of the keys a layer's attention reads."""
    h, d, L = cfg.hidden, cfg.head_dim, cfg.n_layers
    we, se = welt(cfg), side_elt(cfg)
    kve = 4 if cfg.wdtype == syn.F32 else 2
    NS = cfg.top_k + cfg.n_shared
    sc = 4 if cfg.wdtype == syn.FP8 else 0                 # per-row fp32 scales
    out = {}
    n = lambda k: stats.get(k, {}).get("launches", 0)
    u = lambda k: stats.get(k, {}).get("units", 0)
    out["qkv_rope_kvwrite"] = n("qkv_rope_kvwrite") * (cfg.qkv_rows * (h * we + sc) + T * h * 4 + T * cfg.n_q_heads * d * 4
                                                       + T * 2 * cfg.n_kv_heads * d * kve)
    out["attn_splitkv"] = L * ctx_sum * 2 * cfg.n_kv_heads * d * kve
    out["oproj_residual"] = n("oproj_residual") * (h * (cfg.n_q_heads * d * we + sc) + 2 * T * h * 4 + T * cfg.n_q_heads * d * 4)
    out["router_topk_permute"] = n("router_topk_permute") * (cfg.n_experts * h * se + 2 * T * h * 4)
    out["expert_gateup_swiglu"] = u("expert_gateup_swiglu") * 2 * cfg.inter * (h * we + sc) + \
        n("expert_gateup_swiglu") * (T * h * 4 + T * NS * cfg.inter * 4)
    out["expert_down"] = u("expert_down") * h * (cfg.inter * we + sc) + \
        n("expert_down") * (T * NS * cfg.inter * 4 + T * NS * h * 4)
    out["expert_combine"] = n("expert_combine") * (T * NS * h * 4 + 2 * T * h * 4)
    out["lmhead_argmax_commit"] = n("lmhead_argmax_commit") * (cfg.vocab * h * se + T * h * 4)
    return out


# --------------------------------------------------------------------------- #
# CPU oracle timing (cpu_baseline leg and --impl reference)
# --------------------------------------------------------------------------- #
def oracle_rate(w, prompt, wl, max_steps: int, warmup: int, budget_s: float, seq: int = 0) -> dict:
    """Committed tokens/s of the oracle's speculative loop (prefill excluded),
    over up to max_steps verify steps after `warmup` steps, stopping once
    budget_s seconds of timed steps have run."""
    import oracle
    K = wl.n_draft
    t0 = time.time()
    om = oracle.OracleModel(w)
    t_load = time.time() - t0
    n_ref = 1 + (warmup + max_steps) * (K + 1) + K + 1
    # greedy reference of the oracle itself (untimed), for the synthetic drafter
    cache = oracle.KVCache(om.cfg)
    x = oracle.prompt_embeddings(om, prompt)
    t0 = time.time()
    lg = oracle.forward(om, cache, x, np.arange(len(x)))
    t_prefill = time.time() - t0
    base_cache = cache.copy()
    ref = [int(np.argmax(lg[-1]))]
    t0 = time.time()
    while len(ref) < n_ref and time.time() - t0 < 4 * budget_s:
        lg = oracle.forward(om, cache, om.tok_embed[[ref[-1]]], np.array([cache.length]))
        ref.append(int(np.argmax(lg[0])))
    drafter = syn.Drafter(wl.drafter, wl.q, om.cfg.vocab, seed=2)
    cache = base_cache
    toks = [ref[0]]
    steps = committed = 0
    t_run = 0.0
    for s in range(warmup + max_steps):
        if len(toks) + K + 1 > len(ref):
            break
        d = [int(t) for t in drafter.propose(ref, len(toks), K, seq, s)]
        t1 = time.perf_counter()
        base = cache.length
        g = np.argmax(oracle.verify_rows(om, cache, toks[-1], d), -1)
        a, bonus = oracle.accept(d, g)
        cache.truncate(base + a + 1)
        dt = time.perf_counter() - t1
        toks += d[:a] + [bonus]
        if s >= warmup:
            t_run += dt
            steps += 1
            committed += a + 1
            if t_run > budget_s:
                break
    return {"tok_s": committed / t_run if t_run else 0.0, "steps": steps, "committed": committed,
            "s_per_step": t_run / max(steps, 1), "prefill_s": t_prefill, "load_s": t_load,
            "cores": os.cpu_count()}


def run_reference(args):
    ws, rank, _ = dist_env()
    wl = syn.WORKLOADS[args.workload]
    if rank != 0:
        return
    w = syn.generate_weights(wl.model, 0)
    prompt = syn.make_prompts(wl, n_seq=1)[0]
    steps = min(args.steps, 64)
    r = oracle_rate(w, prompt, wl, steps, min(args.warmup, 2), budget_s=60.0)
    value = r["tok_s"]
    line = {
        "impl": "reference", "metric": "committed tokens/s (greedy speculative verify, excl. prefill)",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": r["steps"], "warmup": min(args.warmup, 2),
        "ms_per_step": r["s_per_step"] * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "model": wl.model.name, "batch": wl.batch, "n_draft": wl.n_draft},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
                         "sample": f"{r['steps']} verify steps after the oracle's own prefill of one "
                                   f"{prompt.length}-row prompt (prefill {r['prefill_s']:.1f}s excluded)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def traffic_for(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, when it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(kernel)
    if not e:
        return None
    src = os.path.join(ROOT, "lossless_speculative_decoding_gb300", "csrc", e["source"])
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != e["sha256"]:
        return None
    return e["bytes_per_launch"]


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from lossless_speculative_decoding_gb300 import build as libbuild
    libbuild.build()
    from lossless_speculative_decoding_gb300 import binding as B
    from lossless_speculative_decoding_gb300.runtime import SpecModel

    wl = syn.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses
        wl = dataclasses.replace(wl, model=syn.scaled(wl.model, n_layers=args.layers))
    cfg = wl.model
    if wl.batch != 1:
        raise SystemExit(f"bench.py runs the batch-1 workloads; {wl.name} has batch {wl.batch}")
    K = wl.n_draft
    W, KS, P = args.warmup, args.steps, max(1, args.profile_steps)
    t_setup = time.time()
    w = syn.generate_weights(cfg, 0)
    prompt = syn.make_prompts(wl, n_seq=1, seed=1 + rank)[0]
    total = W + KS + P
    n_ref = 1 + total * (K + 1) + K + 1
    max_ctx = prompt.length + n_ref + 2 * (K + 1)
    pages = -(-max_ctx // wl.page_size) + 4
    gm = SpecModel(cfg, w.arrays, page_size=wl.page_size, n_pages=pages, max_seqs=1, max_ctx=max_ctx,
                   max_draft=K)
    st = gm.stream
    h = gm.h

    # 1) the GPU's own non-speculative greedy trajectory (drafter reference)
    ref = [gm.prefill(0, prompt.visual, prompt.tokens)]
    while len(ref) < n_ref:
        ref.append(gm.verify(0, [])[1])
    ref = np.array(ref, np.int32)
    gm.release(0)
    drafter = syn.Drafter(wl.drafter, wl.q, cfg.vocab, seed=2)
    drafts, agree, n_before = syn.draft_schedule(drafter, ref, total, K, seq=rank)

    # 2) device-resident run: inputs in HBM, graph replay per step
    first = gm.prefill(0, prompt.visual, prompt.tokens)
    assert first == ref[0]
    B.spec_reserve_seq(h, 0, min(max_ctx, prompt.length + n_ref + K + 1))
    with torch.cuda.stream(st):
        d_drafts = torch.from_numpy(drafts.reshape(-1).copy()).cuda()
        d_seq = torch.zeros(1, dtype=torch.int32, device="cuda")
        d_nd = torch.full((1,), K, dtype=torch.int32, device="cuda")
        d_acc = torch.zeros(total, dtype=torch.int32, device="cuda")
        d_bon = torch.zeros(total, dtype=torch.int32, device="cuda")
    st.synchronize()
    esz = 4

    def dev_step(s):
        B.spec_verify_step_batch_dev(h, 1, d_seq, d_drafts.data_ptr() + s * K * esz, d_nd,
                                     d_acc.data_ptr() + s * esz, d_bon.data_ptr() + s * esz)

    for s in range(W):
        dev_step(s)
    st.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for s in range(W, W + KS):
        dev_step(s)
    e1.record(st)
    e1.synchronize()
    clk = clocks.stop()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    acc = d_acc.cpu().numpy()
    committed = int((acc[W:W + KS] + 1).sum())
    ms_all, committed_all = aggregate(ms, committed, device="cuda")

    # 3) profiled steps (events around every kernel launch) on the same sequence
    stats = B.spec_profile_steps_dev(h, 1, d_seq, d_drafts.data_ptr() + (W + KS) * K * esz, d_nd, P, K)
    B.spec_sync_seqs(h)
    gen = gm.tokens(0)
    n_done = int(n_before[total - 1] + agree[total - 1] + 1) if total else 1
    lossless = bool(np.array_equal(gen[:n_done], ref[:n_done]))
    acc_ok = bool(np.array_equal(acc[:W + KS], agree[:W + KS]))
    gm.release(0)

    # 4) end to end through the host C-ABI call (H2D drafts, D2H results each step)
    gm.prefill(0, prompt.visual, prompt.tokens)
    for s in range(W):
        B.spec_verify_step_batch(h, [0], drafts[s], [K])
    h2d0, d2h0 = B.spec_io_bytes(h)
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    e2e_committed = 0
    for s in range(W, W + KS):
        a, _ = B.spec_verify_step_batch(h, [0], drafts[s], [K])
        e2e_committed += int(a[0]) + 1
    e2e_s = time.perf_counter() - t0
    h2d1, d2h1 = B.spec_io_bytes(h)
    e2e_ok = bool(np.array_equal(gm.tokens(0)[:len(ref)], ref[:len(gm.tokens(0))]))
    gm.release(0)
    e2e_s, e2e_committed = aggregate(e2e_s, e2e_committed, device="cuda")

    # 5) roofline of the dominant kernel and of the whole step
    peaks = measured_peaks()
    T = K + 1
    ctx_sum = float(sum(prompt.length + n_before[s] for s in range(W + KS, total)))
    cb = class_bytes(cfg, stats, T, ctx_sum, P)
    dom = max((k for k in stats if k in cb), key=lambda k: stats[k]["ms"])
    dom_bytes_per_launch = cb[dom] / max(stats[dom]["launches"], 1)
    dom_ms_per_launch = stats[dom]["ms"] / max(stats[dom]["launches"], 1)
    achieved = dom_bytes_per_launch / (dom_ms_per_launch * 1e-3) / 1e9
    step_bytes = sum(cb.values()) / P
    prof_ms = sum(v["ms"] for v in stats.values()) / P
    t_roof_us = step_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    ms_per_step = ms_all / KS
    launches = B.spec_step_launches(h, 1) + 1     # + the staging kernel
    share = {k: round(v["ms"] / max(sum(x["ms"] for x in stats.values()), 1e-9), 4) for k, v in stats.items()}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        r = oracle_rate(w, prompt, wl, max_steps=KS, warmup=1, budget_s=args.cpu_budget_s)
        cpu = {"value": r["tok_s"], "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
               "sample": f"{r['steps']} oracle verify steps (T={T} rows each) after one warm-up step, "
                         f"same workload and drafter; oracle prefill of the {prompt.length}-row prompt "
                         f"({r['prefill_s']:.1f}s) excluded"}

    if rank == 0:
        line = {
            "metric": "committed tokens/s (greedy speculative verify, excl. prefill)",
            "value": committed_all / (ms_all * 1e-3),
            "unit": "tokens/s", "n_gpus": ws, "steps": KS, "warmup": W,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {syn.F32: "f32", syn.BF16: "bf16", syn.FP8: "e4m3 weights / f32 activations"}[cfg.wdtype],
            "data": "synthetic (random-init weights, N(0,1) visual rows, seeded drafter)",
            "config": {"workload": wl.name, "model": cfg.name, "layers": cfg.n_layers, "batch": wl.batch, "n_draft": K,
                       "draft_match_prob": wl.q, "prompt_rows": prompt.length, "page_size": wl.page_size,
                       "tau": committed / KS, "l2": "weights read per step (>2 GB) exceed the 126 MB L2",
                       "parallelism": f"replicas x{ws}"},
            "verify_step_us": ms_per_step * 1e3,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": traffic_for(dom), "peak_source": peaks["source"],
                         "bytes_per_launch": dom_bytes_per_launch, "us_per_launch": dom_ms_per_launch * 1e3},
            "step_roofline": {"bytes_per_step": step_bytes, "t_roof_us": t_roof_us,
                              "t_meas_us": ms_per_step * 1e3, "frac": t_roof_us / (ms_per_step * 1e3),
                              "profiled_kernel_us_per_step": prof_ms * 1e3, "kernel_share": share},
            "e2e": {"value": e2e_committed / e2e_s, "unit": "tokens/s",
                    "h2d_bytes_per_step": (h2d1 - h2d0) / KS, "d2h_bytes_per_step": (d2h1 - d2h0) / KS},
            "gpu_launches": launches * KS,
            "clocks": clk,
            "checks": {"lossless_vs_gpu_greedy": lossless, "acceptance_matches_schedule": acc_ok,
                       "e2e_tokens_match": e2e_ok},
            "setup_s": round(time.time() - t_setup, 1),
        }
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    gm.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
