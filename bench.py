"""Benchmark of the fused GRPO loss forward + backward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one call of grpo_loss_fwd_bwd over the whole workload (group
advantages, both vocabulary sweeps, the gradient, the reduction).  Default
workload: the large-vocabulary configuration (B=16, T=2048, V=151936, bf16).
Inputs are synthetic (seeded generator) and larger than L2, so no flush is
needed between steps (the logps-only workload rotates over copies whose total
is larger than L2).  The timed steps are queued behind a head start of plain
device work, so the device events time the device and not the Python call
overhead of short steps; `e2e` times the whole host path.  Under torchrun
every rank runs an independent replica (the loss of one batch does not shard
without its reduction), so scaling is weak and `value` sums the replicas.

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
CSRC = os.path.join(ROOT, "grad_row_online_gb300", "csrc")
# workload -> (committed ncu summary, sources of the kernel it profiles)
PROFILES = {
    "large_vocab": ("rows_kernel_large_vocab.md",
                    ("grpo_rows.cu", "grpo_rows_common.cuh", "grpo_internal.cuh")),
    "fused": ("rows_kernel_fused.md",
              ("grpo_rows.cu", "grpo_rows_common.cuh", "grpo_internal.cuh")),
    "logps": ("logps_kernel_logps.md", ("grpo_logps.cu", "grpo_internal.cuh")),
    "logps_full": ("logps_kernel_logps_full.md", ("grpo_logps.cu", "grpo_internal.cuh")),
    "large_vocab/gspo": ("gspo_kernels_large_vocab.md",
                         ("grpo_rows.cu", "grpo_rows_common.cuh", "grpo_internal.cuh",
                          "grpo_reduce.cu")),
    "large_vocab/skip_masked": ("rows_kernel_large_vocab_skip_masked.md",
                                ("grpo_rows.cu", "grpo_rows_common.cuh", "grpo_internal.cuh")),
    "large_vocab/tp2": ("vocab_kernels_large_vocab_tp2.md",
                        ("grpo_vocab.cu", "grpo_rows.cu", "grpo_rows_common.cuh",
                         "grpo_internal.cuh", "grpo_reduce.cu", "grpo_prep.cu")),
}


def profile_key(w, variant: str = "default", skip_masked: bool = False, tp: int = 0) -> str:
    """The committed profile a bench line's traffic comes from.  On the logits
    path the loss variants run the same row kernel and move the same bytes,
    except GSPO (two passes); the masked-row mode and the vocabulary-parallel
    path move other bytes; the logps path's variants run another kernel
    instantiation."""
    if tp:
        return f"{w.name}/tp{tp}"
    if skip_masked:
        return f"{w.name}/skip_masked"
    if variant == "gspo" or (w.V == 0 and variant != "default"):
        return f"{w.name}/{variant}"
    return w.name


_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(text: str) -> str:
    """The source with its comments removed and every run of blanks outside
    string and character literals made one space (the literals kept as they
    are)."""
    out, code, pos = [], [], 0
    for m in _TOKENS.finditer(text):
        code.append(text[pos:m.start()])
        if m.group(0)[0] in "\"'":
            out.append(re.sub(r"\s+", " ", "".join(code)))
            out.append(m.group(0))
            code = []
        else:
            code.append(" ")
        pos = m.end()
    code.append(text[pos:])
    out.append(re.sub(r"\s+", " ", "".join(code)))
    return "".join(out).strip()


def source_hash(files) -> str:
    """Hash of the code of the kernel sources (comments and layout do not
    count), the key under which a profile's traffic figure stays valid."""
    h = hashlib.sha256()
    for f in files:
        h.update(_code_only(open(os.path.join(CSRC, f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the workload's main kernel from its committed
    ncu summary, if that was taken on the current kernel source."""
    if workload not in PROFILES:
        return None
    name, files = PROFILES[workload]
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    src = re.search(r"^kernel_source_sha:\s*(\w+)", text, re.M)
    wl = re.search(r"^workload:\s*([\w/]+)", text, re.M)
    tb = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not (src and wl and tb) or src.group(1) != source_hash(files) or wl.group(1) != workload:
        return None
    return float(tb.group(1))


# GB300's nominal HBM3e bandwidth (~8 TB/s); the roofline fraction is taken
# against the measured copy rate, and against this figure beside it
NOMINAL_HBM_GBS = 8000.0


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


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


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


def aggregate_value(active: int, steps: int, world: int, elapsed_ms_max: float) -> float:
    """Whole-job throughput: the active tokens every rank processed over the
    slowest rank's time (replicas: each rank runs the full workload)."""
    return active * steps * world / (elapsed_ms_max / 1e3)


# ---------------------------------------------------------------------------
# the oracle as the reference arm / CPU baseline
# ---------------------------------------------------------------------------
def oracle_logps_step(w: synth.Workload, cache: dict) -> int:
    """One pass of the oracle over the whole logps-only workload (inputs
    generated once, not timed).  Returns tokens processed."""
    import oracle
    if "lp" not in cache:
        cache["lp"], cache["old"], cache["ref"] = w.logps_inputs()
        cache["mask"] = w.completion_mask()
        cache["R"], cache["gb"] = w.rewards(), w.group_boundaries()
    A = oracle.group_advantages(cache["R"], cache["gb"])
    oracle.loss_from_logps(cache["lp"], cache["ref"], cache["old"], cache["mask"], A, w.eps_lo,
                           w.eps_hi, w.beta, reduction=w.reduction)
    return int(cache["mask"].sum())


def reference_sample(w: synth.Workload):
    """(step function, sample description) of the oracle on a bounded sample."""
    cores = oracle_threads()
    if w.V == 0:
        cache = {}
        return (lambda: oracle_logps_step(w, cache)), f"the whole {w.name} workload per step"
    active = np.nonzero(w.completion_mask().reshape(-1))[0]
    rows = np.random.default_rng(0).choice(active, min(len(active), max(cores * 2, 16)),
                                           replace=False)
    cache = {}
    return (lambda: oracle_sample_step(w, rows, cache)), \
        f"{len(rows)} random active rows of {w.name} per step (policy+ref log-softmax, token " \
        f"terms, gradient rows)"


def cpu_baseline(w: synth.Workload, budget_s: float = 12.0) -> dict:
    step, what = reference_sample(w)
    step()  # load the library, generate the inputs
    n, t0, passes = 0, time.perf_counter(), 0
    while True:
        n += step()
        passes += 1
        el = time.perf_counter() - t0
        if el > budget_s or passes >= 10000:
            break
    return {"value": n / el, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "cpu_model": cpu_model(), "sample": f"{what}; {passes} passes, {el:.1f} s"}


def run_reference(args, w, ws, rank):
    if rank != 0:
        return
    step, what = reference_sample(w)
    step()
    times, n = [], 0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        k = step()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
            n += k
    total = sum(times)
    value = n / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(),
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": what},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def l2_note(w: synth.Workload) -> str:
    if w.V:
        return "inputs larger than L2 (no flush needed)"
    # logps, old, ref, grad (f32) and the mask per slot, rewards per sequence
    per_copy = w.B * w.T * (4 * 4 + 1) + 4 * w.B
    return (f"inputs rotate over {LogpsCase.COPIES} copies "
            f"({LogpsCase.COPIES * per_copy / 1e6:.0f} MB, larger than L2)")


# loss variants a run may time (keyword arguments of the two entry points);
# "default" is the GRPO loss of the operator page
VARIANTS = {
    "default": {},
    "k1": {"kl": "k1"},
    "k2": {"kl": "k2"},
    "dual-clip": {"dual_clip_c": 3.0},
    "cispo": {"surrogate": "cispo"},
    "fixed-constant": {"reduction": "fixed_constant"},  # C = B*T, set per workload
    "gspo": {"ratio_level": "sequence", "reduction": "sequence_mean"},
}


def variant_kwargs(name: str, w: synth.Workload) -> dict:
    kw = dict(VARIANTS[name])
    if kw.get("reduction") == "fixed_constant":
        kw["norm_constant"] = float(w.B * w.T)
    return kw


def workload_config(w: synth.Workload, variant: str = "default",
                    skip_masked: bool = False) -> dict:
    act = int(w.completion_mask().sum())
    note = l2_note(w)
    cfg = {"workload": f"{w.name}: B={w.B} T={w.T}" + (f" V={w.V} {w.dtype}" if w.V else " logps f32"),
           "B": w.B, "T": w.T, "V": w.V or None, "active_tokens": act,
           "storage_dtype": w.dtype if w.V else "f32",
           "samples_per_prompt": w.samples_per_prompt or None,
           "reduction": ["token_mean", "sequence_mean"][w.reduction],
           "parallelism": "replicas", "l2": note,
           "timing": "device events around the steps, queued behind a head start of "
                     "plain device work so that host call overhead is not timed; the "
                     "main kernel timed by events in a second pass of the same steps"}
    if variant != "default":
        cfg["variant"] = variant
        if "reduction" in VARIANTS[variant]:
            cfg["reduction"] = VARIANTS[variant]["reduction"]
    if skip_masked:
        cfg["masked_grad_rows"] = "skipped (GRPO_SKIP_MASKED_GRAD_ROWS)"
    if not w.V:
        cfg["workspace"] = ("one workspace for every step; calls after the first skip the "
                            "header reset (GRPO_FLAG_WORKSPACE_CLEAN)")
    return cfg


# ---------------------------------------------------------------------------
# the two boundaries under test
# ---------------------------------------------------------------------------
def active_runs(mask) -> list:
    """[begin, end) ranges of consecutive active slots of a [B, T] host mask,
    over the flattened rows (a run may continue into the next sequence)."""
    flat = (np.asarray(mask).reshape(-1) != 0).astype(np.int8)
    edges = np.diff(np.concatenate([[0], flat, [0]]))
    return list(zip(np.flatnonzero(edges == 1).tolist(), np.flatnonzero(edges == -1).tolist()))


def logits_side_bytes(w, active: int, s_in: int, skip_masked: bool) -> dict:
    """The roofline's secondary figures for a logits workload: the strict
    lower bound (the policy read once, as if each row stayed on chip:
    3 V s_in per active token) and the side streams outside the algorithmic
    bytes (action id, behaviour log-prob and mask per token; the zero fill of
    the masked rows' gradient unless they are skipped)."""
    masked = w.B * w.T - active
    return {"strict_bytes_per_launch": 3.0 * w.V * s_in * active,
            "side_bytes_per_launch": 13.0 * active + (0.0 if skip_masked else
                                                      float(w.V * s_in * masked))}


class ReadBack:
    """The end-to-end steps' read-back on a second stream: step i's outputs go
    to the host while step i+1's inputs come in (the two directions of the
    host link at once), and the call of step i+1 waits for that read-back
    before it overwrites the outputs.  With two device input sets
    (`pipe_init`), the copies in run on a third stream too, into the set the
    previous call did not read, so that they also overlap the calls."""

    PIPELINE = ("; three streams: step i+1's inputs are copied into a second device input set "
                "while step i's call runs, and step i's read-back overlaps step i+1's copies in "
                "(a call waits for its inputs and for the previous read-back; the copies into an "
                "input set wait for the call that last read it)")

    def rb_init(self):
        import torch
        self.side = torch.cuda.Stream(device=self.device)
        self.rb_done = None
        self.cin = None

    def pipe_init(self, make_set):
        """Two device input sets and the copy-in stream."""
        import torch
        self.rb_init()
        self.cin = torch.cuda.Stream(device=self.device)
        self.sets = [make_set(), make_set()]
        self.used = [None, None]
        self.k_set = 0

    def pipe_next(self) -> int:
        """The input set of the next step, once the call that last read it is done."""
        j = self.k_set % 2
        self.k_set += 1
        if self.used[j] is not None:
            self.cin.wait_event(self.used[j])
        return j

    def pipe_ready(self):
        """The current stream waits for the copies in queued so far."""
        import torch
        ev = torch.cuda.Event()
        ev.record(self.cin)
        torch.cuda.current_stream().wait_event(ev)

    def pipe_called(self, j: int):
        import torch
        self.used[j] = torch.cuda.Event()
        self.used[j].record(torch.cuda.current_stream())

    def e2e_begin(self):
        """The side streams start after the work queued so far (the start event)."""
        import torch
        for st in (self.side, self.cin):
            if st is not None:
                st.wait_stream(torch.cuda.current_stream())

    def rb_before_call(self):
        import torch
        if self.rb_done is not None:
            torch.cuda.current_stream().wait_event(self.rb_done)

    def rb_stream(self):
        """The side stream, made to wait for the work queued so far."""
        import torch
        self.side.wait_stream(torch.cuda.current_stream())
        return torch.cuda.stream(self.side)

    def rb_end(self):
        import torch
        self.rb_done = torch.cuda.Event()
        self.rb_done.record(self.side)

    def e2e_join(self):
        import torch
        for st in (self.side, self.cin):
            if st is not None:
                torch.cuda.current_stream().wait_stream(st)


class LogitsCase(ReadBack):
    """grpo_loss_fwd_bwd on a logits workload (inputs larger than L2)."""

    launches_per_step = 3  # prep, rows, reduce
    kernel = "rows_kernel (fused sweeps)"

    def __init__(self, w, device, variant="default", skip_masked=False):
        import torch
        import grad_row_online_gb300 as g
        self.g, self.w, self.device = g, w, device
        self.inp = device_inputs(w, device)
        self.kw = loss_kwargs(w, self.inp)
        self.kw.update(variant_kwargs(variant, w))
        if skip_masked:
            self.kw["skip_masked_grad_rows"] = True
        if variant == "gspo":
            self.launches_per_step = 4  # prep, sweep 1, per-sequence step, sweep 2
            self.kernel = "gspo_sweep1_kernel + reduce_kernel + gspo_sweep2_kernel"
        self.active = int(self.inp["mask"].sum().item())
        self.grad = torch.empty_like(self.inp["X"])
        self.out3 = torch.empty(3, dtype=torch.float32, device=device)
        self.wsp = torch.empty(g.grpo_workspace_size(w.B, w.T), dtype=torch.uint8, device=device)
        s_in = 2 if w.dtype == "bf16" else 4
        # policy read twice, ref once, grad written once, per active row
        self.alg_bytes = 4.0 * w.V * s_in * self.active
        self.extra_bytes = logits_side_bytes(w, self.active, s_in, skip_masked)

    def step(self, k=0, prof=None):
        i = self.inp
        self.g.grpo_loss_fwd_bwd(i["X"], i["Y"], i["acts"], i["old"], i["mask"], i["R"],
                                 grad=self.grad, out3=self.out3, workspace=self.wsp, profile=prof,
                                 **self.kw)

    e2e_copy = ("in: the logits rows the call reads (runs of active tokens, found from the "
                "host mask inside each step: masked rows are never read), the other inputs "
                "whole; out: the loss outputs and the gradient rows of the active tokens into a "
                "pinned host gradient buffer (the masked rows' gradient is zero by contract: "
                "the host buffer is zeroed once before the timed steps)" + ReadBack.PIPELINE)

    def e2e_setup(self):
        import torch
        self.host = {}
        for k, v in self.inp.items():
            self.host[k] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
            self.host[k].copy_(v)
        self.pipe_init(lambda: {k: torch.empty_like(v) for k, v in self.inp.items()})
        # the same call as the resident steps (variant, masked-row mode), on the copied
        # inputs; the group boundaries are configuration, not a step's data
        self.kw_e = dict(self.kw)
        self.loss_host = torch.empty(3, dtype=torch.float32).pin_memory()
        self.mask_host = self.host["mask"].numpy()
        self.runs = active_runs(self.mask_host)
        self.grad_host = torch.zeros(self.grad.shape, dtype=self.grad.dtype, pin_memory=True)
        rows = sum(e - b for b, e in self.runs)
        row_bytes = self.w.V * self.host["X"].element_size()
        h2d = 2 * rows * row_bytes + sum(self.host[k].numel() * self.host[k].element_size()
                                         for k in ("acts", "old", "mask", "R"))
        return h2d, rows * row_bytes + 12

    def e2e_check(self):
        """The host gradient's active rows equal the device gradient's (sampled
        rows), and its masked rows are still zero."""
        import torch
        V = self.w.V
        act = np.flatnonzero(self.mask_host.reshape(-1))
        rng = np.random.default_rng(1)
        pick = np.unique(np.concatenate([act[:4], act[-4:], rng.choice(act, min(64, len(act)),
                                                                      replace=False)]))
        dev_rows = self.grad.view(-1, V)[torch.as_tensor(pick, device=self.grad.device)].cpu()
        if not torch.equal(dev_rows, self.grad_host.view(-1, V)[torch.as_tensor(pick)]):
            raise RuntimeError("the end-to-end gradient rows differ from the device's")
        masked = np.flatnonzero(self.mask_host.reshape(-1) == 0)
        if len(masked) and bool(self.grad_host.view(-1, V)[torch.as_tensor(masked[:64])].any()):
            raise RuntimeError("masked rows of the host gradient are not zero")

    def e2e_step(self):
        import torch
        j = self.pipe_next()
        d, h, V = self.sets[j], self.host, self.w.V
        xd, yd = d["X"].view(-1, V), d["Y"].view(-1, V)
        xh, yh = h["X"].view(-1, V), h["Y"].view(-1, V)
        runs = active_runs(self.mask_host)
        with torch.cuda.stream(self.cin):
            for b, e in runs:
                xd[b:e].copy_(xh[b:e], non_blocking=True)
                yd[b:e].copy_(yh[b:e], non_blocking=True)
            for k in ("acts", "old", "mask", "R"):
                d[k].copy_(h[k], non_blocking=True)
        self.pipe_ready()
        self.rb_before_call()
        self.g.grpo_loss_fwd_bwd(d["X"], d["Y"], d["acts"], d["old"], d["mask"], d["R"],
                                 grad=self.grad, out3=self.out3, workspace=self.wsp, **self.kw_e)
        self.pipe_called(j)
        with self.rb_stream():
            self.loss_host.copy_(self.out3, non_blocking=True)
            gd, gh = self.grad.view(-1, V), self.grad_host.view(-1, V)
            for b, e in runs:
                gh[b:e].copy_(gd[b:e], non_blocking=True)
        self.rb_end()


class VocabCase(ReadBack):
    """The vocabulary-parallel path on a logits workload, emulated with `tp`
    slices on one GPU: every slice's partials, the rank-order exchange
    (a concatenation and a sum, as the collectives would leave them), the
    loss, every slice's gradient.  Each "rank" holds its own contiguous slice,
    prepared before the timed region; the timed step is the work of all
    ranks, done one after the other on the one GPU."""

    kernel = "vocab path: partials + merge + reduce + gradient (whole step)"

    def __init__(self, w, device, variant="default", tp=1):
        import torch
        import grad_row_online_gb300 as g
        self.g, self.w, self.device = g, w, device
        inp = device_inputs(w, device)
        C = g.grpo_vocab_chunk()
        nck = (w.V + C - 1) // C
        cuts = [min(w.V, C * (nck * r // tp)) for r in range(tp + 1)]
        self.bounds = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
        self.Xs = [inp["X"][:, :, a:b].contiguous() for a, b in self.bounds]
        self.Ys = [inp["Y"][:, :, a:b].contiguous() for a, b in self.bounds]
        self.grads = [torch.empty_like(x) for x in self.Xs]
        del inp["X"], inp["Y"]
        torch.cuda.empty_cache()
        self.inp = inp
        self.kw = loss_kwargs(w, inp)
        self.kw.update(variant_kwargs(variant, w))
        self.active = int(inp["mask"].sum().item())
        self.launches_per_step = 2 * len(self.bounds) + 3  # partials, prep, merge, reduce, grads
        self.wsp = torch.empty(g.grpo_workspace_size(w.B, w.T), dtype=torch.uint8, device=device)
        s_in = 2 if w.dtype == "bf16" else 4
        # policy and ref read once for the partials, policy once more and the
        # gradient written once for the slices: 4 V s per active row, as the fused path
        self.alg_bytes = 4.0 * w.V * s_in * self.active
        self.extra_bytes = logits_side_bytes(w, self.active, s_in, False)

    def step(self, k=0, prof=None):
        import torch
        g, i, w = self.g, self.inp, self.w
        if prof is not None:
            prof[0].record()
        parts = [g.grpo_vocab_partials(x, y, i["acts"], i["mask"], a)
                 for (a, _), x, y in zip(self.bounds, self.Xs, self.Ys)]
        part_p = torch.cat([p["part_p"] for p in parts])
        part_r = torch.cat([p["part_r"] for p in parts])
        act = torch.stack([p["action_logits"] for p in parts]).sum(0)
        res = g.grpo_vocab_loss(part_p, part_r, act, w.V, i["acts"], i["old"], i["mask"], i["R"],
                                workspace=self.wsp, **self.kw)
        for (a, _), x, gr in zip(self.bounds, self.Xs, self.grads):
            g.grpo_vocab_grad(x, i["acts"], i["mask"], a, res["lse_w"], grad=gr)
        if prof is not None:
            prof[1].record()
        self.out3 = res["out3"]

    e2e_copy = ("in: every slice's logits rows the calls read (runs of active tokens), the "
                "other inputs whole; out: the loss outputs and every slice's gradient rows of the "
                "active tokens into pinned host buffers (masked rows are zero by contract)"
                + ReadBack.PIPELINE)

    def e2e_setup(self):
        import torch
        self.small = ("acts", "old", "mask", "R")
        self.host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
                     for t in self.Xs + self.Ys]
        self.host_small = {k: torch.empty(self.inp[k].shape, dtype=self.inp[k].dtype,
                                          pin_memory=True).copy_(self.inp[k])
                           for k in self.small}
        self.pipe_init(lambda: ([torch.empty_like(t) for t in self.Xs + self.Ys],
                                {k: torch.empty_like(self.inp[k]) for k in self.small}))
        self.loss_host = torch.empty(3, dtype=torch.float32).pin_memory()
        self.mask_host = self.host_small["mask"].numpy()
        self.grads_host = [torch.zeros(t.shape, dtype=t.dtype, pin_memory=True)
                           for t in self.grads]
        rows = sum(e - b for b, e in active_runs(self.mask_host))
        h2d = (rows * sum(t.shape[-1] * t.element_size() for t in self.host)
               + sum(t.numel() * t.element_size() for t in self.host_small.values()))
        return h2d, rows * sum(t.shape[-1] * t.element_size() for t in self.grads) + 12

    def e2e_check(self):
        import torch
        act = np.flatnonzero(self.mask_host.reshape(-1))[:64]
        for gd, gh in zip(self.grads, self.grads_host):
            a = gd.view(-1, gd.shape[-1])[torch.as_tensor(act, device=gd.device)].cpu()
            if not torch.equal(a, gh.view(-1, gh.shape[-1])[torch.as_tensor(act)]):
                raise RuntimeError("the end-to-end gradient rows differ from the device's")

    def e2e_step(self):
        import torch
        n = len(self.Xs)
        runs = active_runs(self.mask_host)
        j = self.pipe_next()
        dev_in, dev_small = self.sets[j]
        with torch.cuda.stream(self.cin):
            for d, h in zip(dev_in, self.host):  # every slice: the rows the calls read
                dv, hv = d.view(-1, d.shape[-1]), h.view(-1, h.shape[-1])
                for b, e in runs:
                    dv[b:e].copy_(hv[b:e], non_blocking=True)
            for k in self.small:
                dev_small[k].copy_(self.host_small[k], non_blocking=True)
        self.Xs, self.Ys = dev_in[:n], dev_in[n:]
        self.inp = dict(self.inp, **dev_small)
        self.pipe_ready()
        self.rb_before_call()
        self.step()
        self.pipe_called(j)
        self.out3.record_stream(self.side)  # allocated by this step, read on the side stream
        with self.rb_stream():
            self.loss_host.copy_(self.out3, non_blocking=True)
            for gd, gh in zip(self.grads, self.grads_host):  # every slice's active gradient rows
                dv, hv = gd.view(-1, gd.shape[-1]), gh.view(-1, gh.shape[-1])
                for b, e in runs:
                    hv[b:e].copy_(dv[b:e], non_blocking=True)
        self.rb_end()


class LogpsCase(ReadBack):
    """grpo_loss_from_logps on the logps-only workload.  One copy of its
    inputs (54 MB) fits in L2, so the timed steps rotate over COPIES copies
    (with their own gradient buffers): a step's inputs were last touched
    COPIES - 1 steps earlier, with more than L2's capacity read and written
    since."""

    COPIES = 4
    CTAS_PER_SM = 7  # the logps kernel's residency (128 threads of 72 registers, 27 KB shared memory)

    def __init__(self, w, device, variant="default", skip_masked=False):
        import torch
        import grad_row_online_gb300 as g
        self.g, self.w, self.device = g, w, device
        # one cooperative launch when every sequence's CTA is resident at once,
        # else the separate advantage / count pass first
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        if w.B <= self.CTAS_PER_SM * sms:
            self.launches_per_step = 1
            self.kernel = "logps_kernel (one launch: advantages, counts, loss and gradient)"
        else:
            self.launches_per_step = 2
            self.kernel = "logps_kernel (after prep_kernel)"
        self.vkw = variant_kwargs(variant, w)
        lp, old, ref = w.logps_inputs()
        host = dict(lp=lp, old=old, ref=ref, mask=w.completion_mask(), R=w.rewards())
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.copies = [{k: t(v) for k, v in host.items()} for _ in range(self.COPIES)]
        for c in self.copies:
            c["grad"] = torch.empty((w.B, w.T), dtype=torch.float32, device=device)
        self.inp = self.copies[0]
        self.grad = self.inp["grad"]
        self.active = int(self.inp["mask"].sum().item())
        self.out3 = torch.empty(3, dtype=torch.float32, device=device)
        self.wsp = torch.empty(g.grpo_workspace_size(w.B, w.T), dtype=torch.uint8, device=device)
        self.ws_clean = False  # the first call resets the header
        self.overlap_launch = False  # --overlap-launch: GRPO_FLAG_OVERLAP_LAUNCH
        # logp / old / ref of active tokens, the mask, dL/dlogp of every slot
        self.alg_bytes = 12.0 * self.active + 5.0 * w.B * w.T
        self.extra_bytes = {}

    def _call(self, i, prof=None):
        w = self.w
        kw = dict(reduction=w.reduction)
        kw.update(self.vkw)
        # one workspace for every step: each call leaves its header clean, so
        # every call after the first skips the reset (GRPO_FLAG_WORKSPACE_CLEAN)
        self.g.grpo_loss_from_logps(i["lp"], i["old"], i["ref"], i["mask"], i["R"],
                                    samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                    clip_eps_hi=w.eps_hi, beta=w.beta, grad=i["grad"],
                                    out3=self.out3, workspace=self.wsp, profile=prof,
                                    workspace_clean=self.ws_clean,
                                    overlap_launch=self.overlap_launch, **kw)
        self.ws_clean = True

    def step(self, k=0, prof=None):
        self._call(self.copies[k % self.COPIES], prof)

    def e2e_setup(self):
        import torch
        self.host = {}
        for k, v in self.inp.items():
            if k == "grad":
                continue
            self.host[k] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
            self.host[k].copy_(v)
        self.pipe_init(lambda: {k: torch.empty_like(v) for k, v in self.inp.items()})
        self.loss_host = torch.empty(3, dtype=torch.float32).pin_memory()
        self.grad_host = torch.empty(self.grad.shape, dtype=torch.float32, pin_memory=True)
        return (sum(v.numel() * v.element_size() for v in self.host.values()),
                self.grad_host.numel() * 4 + 12)

    e2e_copy = ("in: every input whole; out: the loss outputs and dL/dlogp of every slot "
                "into pinned host memory" + ReadBack.PIPELINE)

    def e2e_step(self):
        import torch
        j = self.pipe_next()
        d = self.sets[j]
        with torch.cuda.stream(self.cin):
            for k in self.host:
                d[k].copy_(self.host[k], non_blocking=True)
        self.pipe_ready()
        self.rb_before_call()
        self._call(d)
        self.pipe_called(j)
        with self.rb_stream():
            self.loss_host.copy_(self.out3, non_blocking=True)
            self.grad_host.copy_(d["grad"], non_blocking=True)
        self.rb_end()

    def e2e_check(self):
        import torch
        if not torch.equal(self.grad_host, self.inp["grad"].cpu()):
            raise RuntimeError("the end-to-end dL/dlogp differs from the device-resident steps'")


def head_start(device, seconds: float):
    """Queue about `seconds` of plain device work (zero-fills of a 1 GB
    buffer) ahead of the timed region, so that the host has enqueued the
    timed steps before the device reaches them: the events then time the
    device, not the Python call overhead of short steps."""
    import torch
    buf = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    seconds = min(seconds, 0.05)
    n = max(1, int(seconds / 160e-6) + 1)  # one 1 GB fill takes about 160 us
    for _ in range(n):
        buf.zero_()
    return buf


def run_gpu(args, w, ws, rank, local):
    import torch
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.tp:
        case = VocabCase(w, device, args.variant, args.tp)
    else:
        case = (LogpsCase if w.V == 0 else LogitsCase)(w, device, args.variant, args.skip_masked)
    if args.overlap_launch:
        if not isinstance(case, LogpsCase):
            raise SystemExit("--overlap-launch applies to the logps workloads")
        case.overlap_launch = True
    stream = torch.cuda.current_stream(device)

    t0 = time.perf_counter()
    for k in range(args.warmup):
        case.step(k)
    host_per_step = (time.perf_counter() - t0) / max(args.warmup, 1)
    torch.cuda.synchronize(device)
    assert case.g.grpo_read_device_status(case.wsp) == 0

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record()  # created now, recorded again inside the timed region
        return e
    kev = [(ev(), ev()) for _ in range(args.steps)]   # main kernel (recorded by the library)
    e_start, e_stop = ev(), ev()
    torch.cuda.synchronize(device)

    uuid = getattr(torch.cuda.get_device_properties(device), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    barrier(ws)
    torch.cuda.synchronize(device)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    # the timed steps: nothing but the library calls between the two events
    hs = head_start(device, 2.0 * host_per_step * args.steps + 1e-3)
    e_start.record(stream)
    for k in range(args.steps):
        case.step(k)
    e_stop.record(stream)
    torch.cuda.synchronize(device)
    # the same steps again, with the library's events around the main kernel
    # of every call (the roofline's per-launch time; the events themselves
    # would add a few microseconds to a step of the logps workload)
    hs = head_start(device, 2.0 * host_per_step * args.steps + 1e-3)
    for k in range(args.steps):
        case.step(k, kev[k])
    # and once more with an event between consecutive steps: the spread of
    # the step times (the headline stays the event-free first pass)
    sev = [ev() for _ in range(args.steps + 1)]
    torch.cuda.synchronize(device)
    hs = head_start(device, 2.0 * host_per_step * args.steps + 1e-3)
    sev[0].record(stream)
    for k in range(args.steps):
        case.step(k)
        sev[k + 1].record(stream)
    torch.cuda.synchronize(device)
    barrier(ws)
    clk = clocks.stop() if rank == 0 else None
    del hs
    elapsed_ms = e_start.elapsed_time(e_stop)
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    step_ms = [a.elapsed_time(b) for a, b in zip(sev[:-1], sev[1:])]
    elapsed_ms = max_over_ranks(elapsed_ms, ws, device)
    ms_per_step = elapsed_ms / args.steps
    value = aggregate_value(case.active, args.steps, ws, elapsed_ms)

    # ---- end to end: pinned host inputs -> device -> loss -> host ----
    e2e_steps = min(args.e2e_steps, args.steps)
    resident_out3 = case.out3.clone()  # the loss of the device-resident steps
    h2d, d2h = case.e2e_setup()
    case.e2e_step()
    torch.cuda.synchronize(device)
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    case.e2e_begin()
    for _ in range(e2e_steps):
        case.e2e_step()
    case.e2e_join()  # the last step's read-back
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, device)
    e2e_value = aggregate_value(case.active, e2e_steps, ws, e2e_ms)
    if not torch.equal(case.out3, resident_out3):  # the same inputs, copied in
        raise RuntimeError("the end-to-end steps' loss differs from the device-resident steps'")
    if not torch.equal(case.loss_host, resident_out3.cpu()):
        raise RuntimeError("the loss read back to the host differs from the device's")
    case.e2e_check()

    if rank != 0:
        barrier(ws)
        return
    kern_avg_s = statistics.mean(kernel_ms) / 1e3
    peak, peak_kind = measured_peak()
    achieved = case.alg_bytes / kern_avg_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        # the arithmetic type of the path (fp32 with float-pair and fp64 steps; the
        # logits' storage type is in config["storage_dtype"])
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": dict(workload_config(w, args.variant, args.skip_masked),
                                            **({"launch": "GRPO_FLAG_OVERLAP_LAUNCH: dispatched "
                                                "while the previous step ends, not "
                                                "cooperative"} if args.overlap_launch else {}),
                                            **({"vocab_slices": args.tp} if args.tp else {})),
        "median_ms": statistics.median(step_ms), "min_ms": min(step_ms),
        "max_ms": max(step_ms),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_vs_nominal": achieved / NOMINAL_HBM_GBS,
                     "launch_ms": {"median": statistics.median(kernel_ms),
                                   "min": min(kernel_ms), "max": max(kernel_ms)},
                     "traffic": profiled_traffic(profile_key(w, args.variant,
                                                             args.skip_masked, args.tp)),
                     "kernel": case.kernel, "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": case.alg_bytes, "avg_launch_ms": kern_avg_s * 1e3,
                     **({"strict_frac": case.extra_bytes["strict_bytes_per_launch"] / kern_avg_s
                         / 1e9 / peak, **case.extra_bytes} if case.extra_bytes else {})},
        "step_gbs_algorithmic": case.alg_bytes / (ms_per_step / 1e3) / 1e9,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                **({"copies": case.e2e_copy} if getattr(case, "e2e_copy", None) else {})},
        "gpu_launches": case.launches_per_step * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    barrier(ws)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="large_vocab",
                    choices=["fused", "large_vocab", "var_groups", "logps", "logps_full"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", default="default", choices=list(VARIANTS),
                    help="loss variant to time (default: the operator page's GRPO loss)")
    ap.add_argument("--tp", type=int, default=0,
                    help="time the vocabulary-parallel path with this many slices (on one GPU)")
    ap.add_argument("--overlap-launch", action="store_true",
                    help="logps workloads: GRPO_FLAG_OVERLAP_LAUNCH (nothing else runs on the GPU)")
    ap.add_argument("--skip-masked", action="store_true",
                    help="leave masked gradient rows untouched (GRPO_SKIP_MASKED_GRAD_ROWS)")
    ap.add_argument("--T", type=int, default=0,
                    help="shorter rows per sequence (lengths scaled alike): small profiling case")
    ap.add_argument("--B", type=int, default=0,
                    help="fewer sequences (the same length mix): small profiling case")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    w = synth.WORKLOADS[args.workload]
    if args.T:
        lo, hi = w.len_range
        w = w.with_(name=w.name, T=args.T, len_range=(max(1, lo * args.T // w.T), hi * args.T // w.T))
    if args.B:
        assert not w.samples_per_prompt or args.B % w.samples_per_prompt == 0, \
            "B must be a multiple of samples_per_prompt"
        w = w.with_(name=w.name, B=args.B, holes=w.holes * args.B // w.B)

    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, ws, rank)
        return
    run_gpu(args, w, ws, rank, local)


if __name__ == "__main__":
    main()
