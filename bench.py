"""Benchmark of one EAGLE draft-and-verify round (the whole hot path) on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one round over the workload's batch: every draft layer (FC, decoder
layer, LM head, child selection), the tree expansion/rerank, tree-masked
verification attention for one target layer, acceptance and the commit --
all libeagle kernels.  The target model itself is not part of the method; its
logits are the seeded synthetic stand-in, computed once in setup from the
round's own draft logits (the round is deterministic, so every timed step
rebuilds the same tree).

Prints one JSON line.  `value` = tree nodes verified per second over all
GPUs (N independent replicas, one process per GPU, no collective on the
data path); `e2e` = the same metric through the public API with the step's
inputs copied from pinned host memory and its results read back every step.
`--impl reference` times the CPU oracle (rank 0 only) on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import eagle_synth as S  # noqa: E402

METRIC = "EAGLE draft+verify round µs and tree nodes/s at 7B shape; % of HBM roofline"
ALPHA = (0.9, 0.7, 0.6, 0.6, 0.6, 0.6)   # injected per-layer acceptance profile

# DRAM bytes (read + write) per gemm_stream_kernel launch at 7b_static26,
# averaged over the 30 launches of one round in one ncu capture.  Reported
# only while the kernel's sources hash to the ones the counters were taken on.
GEMM_TRAFFIC = {"workload": "7b_static26", "bytes_per_launch": 125014434,
                "sources": ("gemm.cu", "sm100.cuh", "common.cuh"),
                "sha256": "def55ace163e92a3cac411c25b915ac037ded975bda1936123cf921abd0dff26"}


def gemm_traffic(workload: str):
    h = hashlib.sha256()
    for f in GEMM_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "eagle_feature_level_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if workload == GEMM_TRAFFIC["workload"] and h.hexdigest() == GEMM_TRAFFIC["sha256"]:
        return GEMM_TRAFFIC["bytes_per_launch"]
    return None


def expected_tokens(depth: int) -> float:
    total, run = 1.0, 1.0
    for a in ALPHA[:depth]:
        run *= a
        total += run
    return total


def describe(w) -> str:
    lens = f"prefix {w.prefix_len}" if w.prefix_len else f"prefix U{{{w.prefix_range[0]}..{w.prefix_range[1]}}}"
    tree = (f"EAGLE-2 tree k={w.top_k} depth {w.depth} keep {w.top_m}" if w.tree == "eagle2"
            else f"static {w.top_m}-node tree depth {w.depth}")
    temps = "greedy" if all(t <= 0 for t in w.temps) else ("T=" + "/".join(str(t) for t in w.temps))
    return (f"{w.name}: d={w.d} {w.n_q_heads}q/{w.n_kv_heads}kv x {w.head_dim}, MLP {w.d_ff}, V={w.vocab}, "
            f"batch {w.batch}, {lens}, {tree}, {temps}, bf16 weights")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc = index, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.samples = []
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 6:
                self.samples.append(parts)

    def summary(self):
        if not getattr(self, "samples", None):
            return None
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[2 + i].lower() == "active"})
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(w, inp) -> float:
    from eagle_feature_level_gb300.workload import weight_bytes_per_forward
    from eagle_feature_level_gb300.runtime import plan_for
    plan = plan_for(w.tree, w.top_k, w.depth, w.top_m)
    kv_row = 2 * w.n_kv_heads * w.head_dim * 2                       # K and V, bf16
    n_fwd = plan.n_layers
    draft_kv = sum(inp["draft_len"]) * kv_row
    verify_kv = sum(inp["prefix_len"]) * kv_row
    return n_fwd * weight_bytes_per_forward(w) + n_fwd * draft_kv + verify_kv


def cpu_baseline(w, seed, W, inp, budget_s=20.0, max_rounds=None, warmup=0):
    """The oracle as it stands, on the host cores: full rounds of request 0
    (after up to `warmup` untimed rounds, at most ~30 s of them)."""
    from oracle.layer import DraftWeights
    from oracle.round import numpy_inputs, run_round
    Wc = {k: v.detach().cpu() for k, v in W.items()}
    ic = numpy_inputs({k: (v.detach().cpu() if torch.is_tensor(v) else v) for k, v in inp.items()})
    Wd = DraftWeights(Wc, w)
    warm, t_w = 0, time.perf_counter()
    while warm < warmup and time.perf_counter() - t_w < 30.0:
        run_round(Wd, w, ic, requests=[0])
        warm += 1
    rounds, t0 = 0, time.perf_counter()
    while True:
        run_round(Wd, w, ic, requests=[0])
        rounds += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_rounds and rounds >= max_rounds):
            break
    nodes = w.top_m
    return {"value": nodes * rounds / el, "unit": "tree nodes/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rounds} full rounds of request 0 of {w.name} ({el:.1f} s, numpy fp64, BLAS threads "
                      f"= host cores)", "warmup_rounds": warm}, rounds, el


def cpu_single_thread(workload: str, budget_s: float):
    """The oracle's bounded sample on one host thread: a child process (its
    BLAS limited to one thread from start-up) that rebuilds the inputs from
    the seeds.  Bounded; returns its result dict, or a reason."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-sample", "--workload", workload,
                            "--cpu-budget", str(budget_s)], env=env, capture_output=True, text=True,
                           timeout=budget_s * 6 + 120)
        line = [x for x in r.stdout.splitlines() if x.startswith("{")]
        return json.loads(line[-1]) if line else {"unavailable": (r.stderr or "no output").strip()[-200:]}
    except Exception as exc:                               # reported, not fatal
        return {"unavailable": str(exc)[:200]}


def run_cpu_sample(args):
    w = S.WORKLOADS[args.workload]
    seed = S.WORKLOAD_SEEDS[args.workload]
    W = S.draft_weights(w, seed, device="cpu")
    inp = S.round_inputs(w, seed, device="cpu")
    base, _, _ = cpu_baseline(w, seed, W, inp, budget_s=args.cpu_budget)
    base.pop("warmup_rounds", None)
    base["cores"] = 1
    base["sample"] = base["sample"].replace("BLAS threads = host cores", "BLAS threads = 1")
    print(json.dumps(base), flush=True)


def run_reference(args):
    rank, world, local = dist_setup(args.gpus)
    if rank != 0:
        return
    w = S.WORKLOADS[args.workload]
    seed = S.WORKLOAD_SEEDS[args.workload]
    W = S.draft_weights(w, seed, device="cpu")
    inp = S.round_inputs(w, seed, device="cpu")
    base, rounds, el = cpu_baseline(w, seed, W, inp, budget_s=90.0, max_rounds=max(1, args.steps),
                                    warmup=args.warmup)
    warm = base.pop("warmup_rounds")
    ms = 1000.0 * el / rounds
    line = {"metric": METRIC, "value": base["value"], "unit": "tree nodes/s", "n_gpus": args.gpus,
            "steps": rounds, "warmup": warm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(w), "sample": base["sample"]},
            "cpu_baseline": base,
            "e2e": {"value": base["value"], "unit": "tree nodes/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    from eagle_feature_level_gb300 import _binding as B
    from eagle_feature_level_gb300.workload import gemm_weight_bytes, make_round, standin
    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = S.WORKLOADS[args.workload]
    seed = S.WORKLOAD_SEEDS[args.workload]
    W = S.draft_weights(w, seed, device=dev)
    inp = S.round_inputs(w, seed, device=dev)
    eng, rd = make_round(w, inp, dev)
    wc = eng.weights(W)
    # setup: one round computes the synthetic target's logits for this tree
    rd.run(wc, target_fn=standin(inp))
    torch.cuda.synchronize()
    status = eng.status()
    if status:
        raise RuntimeError(f"device status {B.STATUS.get(status, status)} after setup round")
    accept_len = [int(x) for x in rd.accept_len.cpu()]
    c0 = B.eagle_launch_count(eng.ctx)
    rd.run(wc)                                   # one eager round: launch count per round
    torch.cuda.synchronize()
    per_round = B.eagle_launch_count(eng.ctx) - c0
    # the whole round as one CUDA graph: no host work between the kernels
    graph = rd.capture(wc)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K rounds, inputs resident in HBM ----
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    launches = per_round * args.steps
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    nodes_per_round = w.batch * w.top_m
    value = world * nodes_per_round * args.steps / (ms_total / 1e3)

    # ---- per-kernel durations inside the untraced round ----
    # The same round captured with launch timestamps: every kernel records
    # (%globaltimer) when its first CTA passed the wait for its predecessors
    # and when its last CTA left.  Kernel i's exclusive window runs from its
    # own release to the next kernel's release (the last one's to its exit):
    # the windows tile the round, so they sum to the round's device time and
    # keep the programmatic overlap between kernels intact.
    cap = per_round + 8
    stamps = torch.empty(3 * cap, dtype=torch.int64, device=dev)
    B.eagle_stamps_enable(eng.ctx, stamps.data_ptr(), cap)
    sgraph = rd.capture(wc)
    names = B.eagle_stamps_disable(eng.ctx)
    k_st = min(max(args.steps, 5), 50)
    n = len(names)
    excl = [0.0] * n
    span = [0.0] * n
    stamped_round = 0.0
    tick = None
    dump = []
    for rep in range(k_st):
        stamps.view(-1, 3)[:, :2].fill_(-1)         # UINT64_MAX: no start / release seen yet
        stamps.view(-1, 3)[:, 2].fill_(0)
        sgraph.replay()
        torch.cuda.synchronize()
        t = [int(x) & 0xFFFFFFFFFFFFFFFF for x in stamps[:3 * n].cpu().tolist()]
        s_, w_, e_ = t[0::3], t[1::3], t[2::3]
        if rep == k_st - 1 and args.dump_stamps:
            dump = [{"kernel": names[i], "start_us": (s_[i] - w_[0]) / 1e3, "release_us": (w_[i] - w_[0]) / 1e3,
                     "exit_us": (e_[i] - w_[0]) / 1e3} for i in range(n)]
        for i in range(n):
            nxt = w_[i + 1] if i + 1 < n else e_[i]
            excl[i] += (nxt - w_[i]) / 1e3
            span[i] += (e_[i] - w_[i]) / 1e3
        stamped_round += (e_[n - 1] - w_[0]) / 1e3
        d = sorted({abs(a - b) for a, b in zip(w_[1:], w_[:-1]) if a != b})
        if d:
            tick = d[0] if tick is None else min(tick, d[0])
    del sgraph
    if dump:
        with open(args.dump_stamps, "w") as fh:
            json.dump(dump, fh, indent=0)
    by_class = {}
    for i, name in enumerate(names):
        c = by_class.setdefault(name, [0, 0.0, 0.0])
        c[0] += 1
        c[1] += excl[i] / k_st
        c[2] += span[i] / k_st
    gb = gemm_weight_bytes(w)
    g_cls = [c for c in gb if c in by_class]
    g_bytes = sum(gb[c] * by_class[c][0] for c in g_cls)                  # per round
    g_us = sum(by_class[c][1] for c in g_cls)
    g_launch = sum(by_class[c][0] for c in g_cls)
    peak, peak_kind = peaks()
    achieved = g_bytes / (g_us / 1e6) / 1e9
    per_contraction = {c: {"us_per_launch": round(by_class[c][1] / by_class[c][0], 2),
                           "gbs": round(gb[c] / (by_class[c][1] / by_class[c][0] / 1e6) / 1e9, 1)}
                       for c in g_cls}
    stage = {
        "draft_us": sum(by_class.get(c, [0, 0.0])[1] for c in
                        ("prep", "gemm_fc", "gemm_qkv", "draft_attn", "gemm_o", "gemm_gateup", "gemm_down",
                         "gemm_lm", "select")),
        "tree_us": by_class.get("tree", [0, 0.0])[1],
        "verify_us": by_class.get("verify_attn", [0, 0.0])[1],
        "accept_us": by_class.get("accept", [0, 0.0])[1],
        "commit_us": by_class.get("commit", [0, 0.0])[1],
    }
    kernel_us = {c: round(v[1], 2) for c, v in sorted(by_class.items())}

    # ---- end to end through the public API with host buffers ----
    # the round's host-facing tensors live in one device allocation per
    # direction (runtime.Round.io_in / io_out): one copy each way per step
    host_in = rd.io_in.detach().to("cpu").pin_memory()
    host_out = torch.empty(rd.io_out.shape, dtype=rd.io_out.dtype, pin_memory=True)
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()
    k_e2e = max(1, min(args.steps, 200))
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        rd.io_in.copy_(host_in, non_blocking=True)
        graph.replay()
        host_out.copy_(rd.io_out, non_blocking=True)
        stream.synchronize()
    el = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e_value = world * nodes_per_round * k_e2e / el

    # ---- CPU baseline (rank 0, N = 1 only) ----
    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base, _, _ = cpu_baseline(w, seed, W, inp, budget_s=args.cpu_budget)
        base.pop("warmup_rounds", None)
        if args.workload in ("tiny_fp32", "7b_static26", "7b_eagle2"):
            base["single_thread"] = cpu_single_thread(args.workload, args.cpu_budget)
        else:
            base["single_thread"] = {"unavailable": "not run: one round of this shape takes minutes on one thread"}

    alg = algorithmic_bytes(w, {"draft_len": inp["draft_len"], "prefix_len": inp["prefix_len"]})
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "tree nodes/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(w), "batch": w.batch, "tree_nodes": w.top_m,
                   "draft_forwards": int(rd.plan.n_layers),
                   "l2": "inputs larger than L2: each draft forward streams "
                         f"{alg / rd.plan.n_layers / 1e6:.0f} MB of weights and KV (L2 = 129 MB)",
                   "parallelism": f"replicas x{world}", "target": "synthetic logits (setup round)"},
        "round_us": 1e3 * ms_step,
        "committed_tokens_per_s": world * w.batch * expected_tokens(w.depth) / (ms_step / 1e3),
        "expected_tokens_per_round": expected_tokens(w.depth),
        "accept_len_observed": accept_len,
        "algorithmic_bytes_per_round": alg,
        "hbm_frac": alg / (ms_step / 1e3) / (peak * 1e9),
        "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "hbm_frac_of_nominal_8tbs": alg / (ms_step / 1e3) / 8.0e12,
        "timing": "stages_us / kernel_us_per_round: exclusive windows of each kernel inside the untraced "
                  "graph replay (kernel-written %globaltimer stamps, mean of "
                  f"{k_st} replays); they sum to stamped_round_us",
        "stamped_round_us": round(stamped_round / k_st, 2),
        "stamp_tick_ns": tick,
        "stages_us": {k: round(v, 2) for k, v in stage.items()},
        "kernel_us_per_round": kernel_us,
        "kernel_span_us_per_round": {c: round(v[2], 2) for c, v in sorted(by_class.items())},
        "roofline": {"kernel": "gemm_stream_kernel (all six draft-layer contractions)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": gemm_traffic(w.name), "launches_per_round": g_launch,
                     "bytes_per_launch": g_bytes / max(g_launch, 1),
                     "us_per_round": round(g_us, 2),
                     "duration": "exclusive window per launch from launch timestamps in the untraced round",
                     "per_contraction": per_contraction},
        "e2e": {"value": e2e_value, "unit": "tree nodes/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": k_e2e},
        "gpu_launches": launches,
        "launches_per_round": per_round,
        "execution": "CUDA graph of the whole round (captured once, replayed per step)",
        "clocks": clocks,
        "cpu_baseline": base,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="7b_static26", choices=list(S.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-oracle-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--dump-stamps", default=None, help="write the last stamped replay's per-launch times (JSON)")
    args = ap.parse_args()
    if args.cpu_oracle_sample:
        run_cpu_sample(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
