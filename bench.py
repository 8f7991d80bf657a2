"""Benchmark of the fused GRPO loss forward + backward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one call of grpo_loss_fwd_bwd over the whole workload (group
advantages, both vocabulary sweeps, the gradient, the reduction).  Default
workload: the large-vocabulary configuration (B=16, T=2048, V=151936, bf16).
Inputs are synthetic (seeded generator) and larger than L2, so no flush is
needed between steps.  Under torchrun every rank runs an independent replica
(the loss of one batch does not shard without its reduction; see the design
notes), so scaling is weak and `value` sums the replicas.

--impl reference times the double-precision CPU oracle (the only reference
implementation of this method) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "active tokens/s and HBM GB/s (% of roofline), fused GRPO fwd+bwd, 1 GB300"
UNIT = "active tokens/s"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "rows_kernel_large_vocab.md")
ROWS_SOURCES = [os.path.join(ROOT, "grad_row_online_gb300", "csrc", f)
                for f in ("grpo_rows.cu", "grpo_rows_common.cuh", "grpo_internal.cuh")]


def rows_source_hash() -> str:
    h = hashlib.sha256()
    for f in ROWS_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the row kernel from the committed ncu summary,
    if it was taken on the current kernel source for this workload."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    src = re.search(r"kernel_source_sha:\s*(\w+)", text)
    wl = re.search(r"workload:\s*(\w+)", text)
    tb = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (src and wl and tb) or src.group(1) != rows_source_hash() or wl.group(1) != workload:
        return None
    return float(tb.group(1))


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------
def device_inputs(w: synth.Workload, device):
    import torch
    X = w.logits_device("policy", device)
    Y = w.logits_device("ref", device)
    acts = torch.from_numpy(w.action_ids()).to(device)
    mask = torch.from_numpy(w.completion_mask()).to(device)
    R = torch.from_numpy(w.rewards()).to(device)
    noise = torch.from_numpy(w.old_noise()).to(device)
    # old_logps = log-prob of the action under the policy + old_sigma * N(0,1),
    # the log-prob taken from PyTorch's fp32 log_softmax (input preparation only)
    old = torch.zeros((w.B, w.T), dtype=torch.float32, device=device)
    flat = mask.view(-1).nonzero().squeeze(1)
    Xf, af, of = X.view(-1, w.V), acts.view(-1), old.view(-1)
    for i in range(0, flat.numel(), 512):
        rows = flat[i:i + 512]
        lsm = torch.log_softmax(Xf[rows].float(), dim=-1)
        of[rows] = lsm.gather(1, af[rows][:, None]).squeeze(1)
        del lsm
    old += w.old_sigma * noise.float() * mask
    bounds = torch.from_numpy(w.group_boundaries()).to(device)
    torch.cuda.synchronize(device)
    return dict(X=X, Y=Y, acts=acts, mask=mask, R=R, old=old, bounds=bounds)


def loss_kwargs(w: synth.Workload, inp):
    kw = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction)
    if w.samples_per_prompt:
        kw["samples_per_prompt"] = w.samples_per_prompt
    else:
        kw["group_boundaries"] = inp["bounds"]
    return kw


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------
def oracle_sample_step(w: synth.Workload, sample_rows: np.ndarray, cache: dict) -> int:
    """One pass of the oracle over `sample_rows` active rows of the workload:
    log-softmax of both rows, the token terms and weights, the gradient rows.
    Input generation is done once and not timed.  Returns tokens processed."""
    import oracle
    if "X" not in cache:
        cache["X"] = w.logit_rows("policy", sample_rows)
        cache["Y"] = w.logit_rows("ref", sample_rows)
        cache["acts"] = w.action_ids().reshape(-1)[sample_rows]
        cache["noise"] = w.old_noise().reshape(-1)[sample_rows]
        cache["A"] = oracle.group_advantages(w.rewards(), w.group_boundaries())
    n = len(sample_rows)
    lse, lp = oracle.log_softmax_rows(cache["X"], w.dtype, cache["acts"])
    _, rl = oracle.log_softmax_rows(cache["Y"], w.dtype, cache["acts"])
    old = (lp + w.old_sigma * cache["noise"]).astype(np.float32)
    mask = np.ones((1, n), np.uint8)
    res = oracle.loss_from_logps(lp[None], rl[None], old[None], mask, cache["A"][:1],
                                 w.eps_lo, w.eps_hi, w.beta, reduction=w.reduction)
    oracle.grad_rows(cache["X"], w.dtype, cache["acts"], lse, res["w"][0])
    return n


def oracle_threads() -> int:
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def cpu_baseline(w: synth.Workload, budget_s: float = 12.0) -> dict:
    active = np.nonzero(w.completion_mask().reshape(-1))[0]
    cores = oracle_threads()
    rows = np.random.default_rng(0).choice(active, min(len(active), max(cores * 2, 16)),
                                           replace=False)
    cache = {}
    oracle_sample_step(w, rows[:2], {})  # load the library
    t0 = time.perf_counter()
    n = oracle_sample_step(w, rows, cache)
    first = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(first, 1e-3)) - 1)
    t0 = time.perf_counter()
    for _ in range(reps):
        n += oracle_sample_step(w, rows, cache)
    el = first + time.perf_counter() - t0
    return {"value": n / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} random active rows of {w.name} (policy+ref log-softmax, "
                      f"token terms, gradient rows), {reps + 1} passes, {el:.1f} s"}


# ---------------------------------------------------------------------------
def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, w, ws, rank):
    if rank != 0:
        return
    cores = oracle_threads()
    active = np.nonzero(w.completion_mask().reshape(-1))[0]
    rows = np.random.default_rng(0).choice(active, min(len(active), max(cores, 8)), replace=False)
    cache = {}
    oracle_sample_step(w, rows, cache)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle_sample_step(w, rows, cache)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = len(rows) * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: {len(rows)} random active rows of {w.name}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w: synth.Workload) -> dict:
    act = int(w.completion_mask().sum())
    cfg = {"workload": f"{w.name}: B={w.B} T={w.T} V={w.V} {w.dtype}", "B": w.B, "T": w.T,
           "V": w.V, "active_tokens": act, "samples_per_prompt": w.samples_per_prompt or None,
           "reduction": ["token_mean", "sequence_mean"][w.reduction],
           "parallelism": "replicas", "l2": "inputs larger than L2 (no flush needed)"}
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large_vocab",
                    choices=["fused", "large_vocab", "var_groups"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=int, default=0,
                    help="shorter rows per sequence (lengths scaled alike): small profiling case")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    w = synth.WORKLOADS[args.workload]
    if args.T:
        lo, hi = w.len_range
        w = w.with_(name=w.name, T=args.T, len_range=(max(1, lo * args.T // w.T), hi * args.T // w.T))

    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, ws, rank)
        return

    import torch
    import grad_row_online_gb300 as g
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    inp = device_inputs(w, device)
    kw = loss_kwargs(w, inp)
    B, T, V = w.B, w.T, w.V
    s_in = 2 if w.dtype == "bf16" else 4
    active = int(inp["mask"].sum().item())
    grad = torch.empty_like(inp["X"])
    out3 = torch.empty(3, dtype=torch.float32, device=device)
    wsp = torch.empty(g.grpo_workspace_size(B, T), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(prof=None):
        g.grpo_loss_fwd_bwd(inp["X"], inp["Y"], inp["acts"], inp["old"], inp["mask"], inp["R"],
                            grad=grad, out3=out3, workspace=wsp, profile=prof, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    assert g.grpo_read_device_status(wsp) == 0

    # row-kernel events, created up front (recorded by the library)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        a.record(); b.record()
    torch.cuda.synchronize(device)

    uuid = getattr(torch.cuda.get_device_properties(device), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    barrier(ws)
    torch.cuda.synchronize(device)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_stop.record(stream)
    torch.cuda.synchronize(device)
    barrier(ws)
    clk = clocks.stop() if rank == 0 else None
    elapsed_ms = t_start.elapsed_time(t_stop)
    rows_ms = [a.elapsed_time(b) for a, b in evs]
    elapsed_ms = max_over_ranks(elapsed_ms, ws, device)
    ms_per_step = elapsed_ms / args.steps
    value = active * args.steps * ws / (elapsed_ms / 1e3)

    # ---- end to end: pinned host inputs -> device -> loss -> host ----
    e2e_steps = min(args.e2e_steps, args.steps)
    host = {}
    for k, v in inp.items():
        host[k] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
        host[k].copy_(v)
    h2d = sum(v.numel() * v.element_size() for k, v in host.items() if k != "bounds")
    loss_host = torch.empty(3, dtype=torch.float32).pin_memory()
    dev_in = {k: torch.empty_like(v) for k, v in inp.items()}
    dev_in["bounds"] = inp["bounds"]
    kw_e = loss_kwargs(w, dev_in)

    def e2e_step():
        for k in ("X", "Y", "acts", "old", "mask", "R"):
            dev_in[k].copy_(host[k], non_blocking=True)
        g.grpo_loss_fwd_bwd(dev_in["X"], dev_in["Y"], dev_in["acts"], dev_in["old"],
                            dev_in["mask"], dev_in["R"], grad=grad, out3=out3, workspace=wsp,
                            **kw_e)
        loss_host.copy_(out3, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(device)
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    e2e_value = active * e2e_steps * ws / (e2e_ms / 1e3)

    if rank != 0:
        barrier(ws)
        return

    alg_bytes = 4.0 * V * s_in * active  # policy read twice, ref once, grad written once
    rows_avg_s = statistics.mean(rows_ms) / 1e3
    peak, peak_kind = measured_peak()
    achieved = alg_bytes / rows_avg_s / 1e9
    traffic = profiled_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "rows_kernel (fused sweeps)", "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": alg_bytes, "avg_launch_ms": rows_avg_s * 1e3},
        "step_gbs_algorithmic": alg_bytes / (ms_per_step / 1e3) / 1e9,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 12, "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    barrier(ws)


if __name__ == "__main__":
    main()
