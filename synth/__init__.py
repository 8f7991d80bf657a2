"""Seeded synthetic inputs for the GRPO loss workloads.

This module draws random numbers and nothing else: it holds no arithmetic of
the GRPO method.  Both sides of every parity comparison (the oracle under
``oracle/`` and the CUDA library) receive inputs from here.

Every element is a pure function of ``(seed, stream, index)`` (see
``synth_core.h``), so the host build (C, gcc) and the device build (CUDA) give
the same bits, and any row of a tensor that is too large for host memory can
be regenerated on its own.

The workloads follow the sizes and value distributions stated for the fused
GRPO loss benchmarks: ``N(0, s)`` means a normal with standard deviation
``s``.  The one input that depends on the method -- the behaviour log-prob
``old_logps = exact policy log-prob of the action + N(0, 0.05)`` -- is not
formed here: this module supplies the ``N(0,1)`` deviates (``old_noise``) and
the caller adds them to a log-prob it computed itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth_host.so")
_CUDA_SO = os.path.join(_HERE, "libsynth_cuda.so")

STREAM_POLICY, STREAM_SPIKE, STREAM_REF, STREAM_ACTION = 1, 2, 3, 4
STREAM_OLD, STREAM_REWARD, STREAM_LENGTH, STREAM_GROUP = 5, 6, 7, 8
STREAM_LOGP, STREAM_REFLOGP, STREAM_HOLE, STREAM_MISC = 9, 10, 11, 12

DTYPE_CODE = {"f32": 0, "bf16": 1}


# --------------------------------------------------------------------------
# build / load
# --------------------------------------------------------------------------
def build_commands(arch: str = "103a") -> list[list[str]]:
    """Compiler invocations that produce the two generator libraries."""
    host = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
            "-ffp-contract=off", "-fno-fast-math",
            os.path.join(_HERE, "synth_host.c"), "-o", _HOST_SO, "-lm"]
    cuda = ["nvcc", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-O3",
            "-fmad=false", "-shared", "-Xcompiler", "-fPIC",
            os.path.join(_HERE, "synth_cuda.cu"), "-o", _CUDA_SO]
    return [host, cuda]


def build() -> None:
    procs = [subprocess.Popen(c) for c in build_commands()]
    for p, c in zip(procs, build_commands()):
        if p.wait() != 0:
            raise RuntimeError("synth build failed: " + " ".join(c))


_host_lib = None
_cuda_lib = None


def host_lib():
    global _host_lib
    if _host_lib is None:
        if not os.path.exists(_HOST_SO):
            raise RuntimeError(f"{_HOST_SO} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(_HOST_SO)
        i64, u64, u32, dbl, vp = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                  ctypes.c_double, ctypes.c_void_p)
        lib.synth_host_logit_rows.argtypes = [u64, ctypes.c_int, ctypes.c_int, vp, i64,
                                              i64, dbl, dbl, dbl, dbl, vp]
        lib.synth_host_normal.argtypes = [u64, u32, i64, i64, vp]
        lib.synth_host_uniform.argtypes = [u64, u32, i64, i64, u32, vp]
        lib.synth_host_below.argtypes = [u64, u32, i64, i64, u32, u64, vp]
        _host_lib = lib
    return _host_lib


def cuda_lib():
    global _cuda_lib
    if _cuda_lib is None:
        if not os.path.exists(_CUDA_SO):
            raise RuntimeError(f"{_CUDA_SO} missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(_CUDA_SO)
        lib.synth_cuda_logits.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_double,
                                          ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_cuda_logits.restype = ctypes.c_int
        _cuda_lib = lib
    return _cuda_lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# --------------------------------------------------------------------------
# primitive draws (host)
# --------------------------------------------------------------------------
def normal(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        host_lib().synth_host_normal(seed, stream, start, n, _ptr(out))
    return out


def uniform(seed: int, stream: int, start: int, n: int, draw: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        host_lib().synth_host_uniform(seed, stream, start, n, draw, _ptr(out))
    return out


def below(seed: int, stream: int, start: int, n: int, bound: int, draw: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if n:
        host_lib().synth_host_below(seed, stream, start, n, draw, bound, _ptr(out))
    return out


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One synthetic GRPO-loss workload: shapes, distributions, loss knobs."""
    name: str
    B: int
    T: int
    V: int = 0                      # 0 for the logps-only workload
    dtype: str = "f32"              # storage dtype of the logits ("f32" | "bf16")
    seed: int = 0
    sigma: float = 1.0              # policy logits ~ N(0, sigma)
    spike_p: float = 0.0            # probability of a +spike_mag spike
    spike_mag: float = 0.0
    ref_sigma: float = 0.1          # ref = policy + N(0, ref_sigma)
    old_sigma: float = 0.05         # old = exact logp + N(0, old_sigma)
    samples_per_prompt: int = 0     # uniform groups (0 -> CSR groups)
    csr_size_range: tuple = (2, 16)  # CSR group sizes U{lo..hi}
    reward: str = "bernoulli"       # "bernoulli" | "normal"
    reward_p: float = 0.5
    zero_group: bool = False        # force group 0 all-zero, redraw the others
    mask: str = "prefix"            # "prefix" | "full"
    len_range: tuple = (1, 1)       # prefix length U{lo..hi}
    holes: int = 0                  # number of rows made fully masked
    eps_lo: float = 0.2
    eps_hi: float = 0.2
    beta: float = 0.04
    reduction: int = 0              # 0 token mean, 1 sequence mean
    logp_mean: float = -2.0         # logps-only workload: logp ~ N(mean, sd)
    logp_sigma: float = 0.5
    ref_logp_sigma: float = 0.05

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def rows(self) -> int:
        return self.B * self.T

    # ---- group structure -------------------------------------------------
    def group_boundaries(self) -> np.ndarray:
        """CSR offsets [G+1] (also returned for uniform groups)."""
        if self.samples_per_prompt > 0:
            assert self.B % self.samples_per_prompt == 0
            return np.arange(0, self.B + 1, self.samples_per_prompt, dtype=np.int64)
        lo, hi = self.csr_size_range
        sizes, total, j = [], 0, 0
        while True:
            s = lo + int(below(self.seed, STREAM_GROUP, j, 1, hi - lo + 1)[0])
            j += 1
            if total + s > self.B:
                break
            sizes.append(s)
            total += s
        rem = self.B - total
        if rem >= 2 or (rem == 1 and not sizes):
            sizes.append(rem)
        elif rem == 1:
            sizes[-1] += 1
        return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)

    # ---- [B] and [B,T] inputs --------------------------------------------
    def lengths(self) -> np.ndarray:
        if self.mask == "full":
            L = np.full(self.B, self.T, dtype=np.int64)
        else:
            lo, hi = self.len_range
            L = lo + below(self.seed, STREAM_LENGTH, 0, self.B, hi - lo + 1)
        if self.holes:
            chosen, j = [], 0
            while len(chosen) < min(self.holes, self.B):
                r = int(below(self.seed, STREAM_HOLE, j, 1, self.B)[0])
                j += 1
                if r not in chosen:
                    chosen.append(r)
            L[chosen] = 0
        return L

    def completion_mask(self) -> np.ndarray:
        L = self.lengths()
        return (np.arange(self.T)[None, :] < L[:, None]).astype(np.uint8)

    def action_ids(self) -> np.ndarray:
        return below(self.seed, STREAM_ACTION, 0, self.rows, self.V).reshape(self.B, self.T)

    def rewards(self) -> np.ndarray:
        gb = self.group_boundaries()
        if self.reward == "normal":
            return normal(self.seed, STREAM_REWARD, 0, self.B).astype(np.float32)
        R = np.zeros(self.B, dtype=np.float32)
        for g in range(len(gb) - 1):
            lo, hi = int(gb[g]), int(gb[g + 1])
            if self.zero_group and g == 0:
                continue
            for draw in range(1000):
                r = (uniform(self.seed, STREAM_REWARD, lo, hi - lo, draw) < self.reward_p)
                if not self.zero_group or hi - lo < 2 or 0 < r.sum() < hi - lo:
                    break
            R[lo:hi] = r.astype(np.float32)
        return R

    def old_noise(self) -> np.ndarray:
        """N(0,1) deviates, [B,T]; old_logps = logp + old_sigma * noise."""
        return normal(self.seed, STREAM_OLD, 0, self.rows).reshape(self.B, self.T)

    # ---- logps-only workload -----------------------------------------------
    def logps_inputs(self):
        """(logps, old_logps, ref_logps) as float32 [B,T]."""
        n = self.rows
        lp = (self.logp_mean + self.logp_sigma * normal(self.seed, STREAM_LOGP, 0, n)).astype(np.float32)
        old = (lp.astype(np.float64) + self.old_sigma * normal(self.seed, STREAM_OLD, 0, n)).astype(np.float32)
        ref = (lp.astype(np.float64) + self.ref_logp_sigma * normal(self.seed, STREAM_REFLOGP, 0, n)).astype(np.float32)
        shp = (self.B, self.T)
        return lp.reshape(shp), old.reshape(shp), ref.reshape(shp)

    # ---- logits -----------------------------------------------------------
    def logit_rows(self, which: str, rows) -> np.ndarray:
        """Host copy of the given rows (flat row index b*T+t) of the policy
        ("policy") or reference ("ref") logits: float32 or uint16 (bf16 bits)."""
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        npdt = np.uint16 if self.dtype == "bf16" else np.float32
        out = np.empty((len(rows), self.V), dtype=npdt)
        if len(rows):
            host_lib().synth_host_logit_rows(self.seed, DTYPE_CODE[self.dtype],
                                             int(which == "ref"), _ptr(rows), len(rows), self.V,
                                             self.sigma, self.spike_p, self.spike_mag,
                                             self.ref_sigma, _ptr(out))
        return out

    def logits_host(self, which: str) -> np.ndarray:
        """The whole [B,T,V] tensor on the host (small workloads only)."""
        return self.logit_rows(which, np.arange(self.rows)).reshape(self.B, self.T, self.V)

    def logits_device(self, which: str, device="cuda"):
        """The whole [B,T,V] tensor generated directly in device memory."""
        import torch
        tdt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        out = torch.empty((self.B, self.T, self.V), dtype=tdt, device=device)
        stream = torch.cuda.current_stream(out.device).cuda_stream
        rc = cuda_lib().synth_cuda_logits(self.seed, DTYPE_CODE[self.dtype], int(which == "ref"),
                                          out.numel(), self.sigma, self.spike_p, self.spike_mag,
                                          self.ref_sigma, out.data_ptr(), stream)
        if rc != 0:
            raise RuntimeError(f"synth_cuda_logits failed with CUDA error {rc}")
        return out


# The five workloads of the fused GRPO loss benchmark.
WORKLOADS = {
    # 2 prompts x 4 samples, T=16, V=64, fp32 logits ~N(0,1)
    "tiny": Workload("tiny", B=8, T=16, V=64, dtype="f32", seed=0, sigma=1.0,
                     ref_sigma=0.1, samples_per_prompt=4, reward_p=0.5,
                     len_range=(4, 16), eps_lo=0.2, eps_hi=0.2, beta=0.04),
    # logps-only loss: 128 prompts x 8, T=4096, ragged prefixes in [T/4, T]
    "logps": Workload("logps", B=1024, T=4096, V=0, seed=1, samples_per_prompt=8,
                      reward_p=0.3, len_range=(1024, 4096), eps_lo=0.2, eps_hi=0.2,
                      beta=0.04),
    # fused logits path: 8 prompts x 8, T=1024, V=32768, bf16 ~N(0,2)
    "fused": Workload("fused", B=64, T=1024, V=32768, dtype="bf16", seed=2, sigma=2.0,
                      ref_sigma=0.1, samples_per_prompt=8, reward_p=0.5,
                      len_range=(128, 1024), eps_lo=0.2, eps_hi=0.2, beta=0.04),
    # large vocabulary: 2 prompts x 8, T=2048, V=151936, bf16 ~N(0,3) + 1% spikes of +8
    "large_vocab": Workload("large_vocab", B=16, T=2048, V=151936, dtype="bf16", seed=3,
                            sigma=3.0, spike_p=0.01, spike_mag=8.0, ref_sigma=0.2,
                            samples_per_prompt=8, reward_p=0.4, zero_group=True,
                            len_range=(256, 2048), eps_lo=0.2, eps_hi=0.28, beta=0.04),
    # variable CSR groups over 64 sequences, T=512, V=128256, fp32 ~N(0,2), sequence mean
    "var_groups": Workload("var_groups", B=64, T=512, V=128256, dtype="f32", seed=4,
                           sigma=2.0, ref_sigma=0.1, samples_per_prompt=0,
                           csr_size_range=(2, 16), reward="normal", len_range=(16, 512),
                           holes=4, eps_lo=0.2, eps_hi=0.2, beta=0.04, reduction=1),
}
# the logps-only workload is also run with a full mask
WORKLOADS["logps_full"] = WORKLOADS["logps"].with_(name="logps_full", mask="full")
