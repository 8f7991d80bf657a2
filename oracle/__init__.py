"""TEST INFRASTRUCTURE: the double-precision CPU oracle of the GRPO loss.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library in ``grad_row_online_gb300``; the two meet only through inputs drawn
by ``synth``.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this file
marshals numpy arrays and composes the C steps in the order the GRPO loss
defines them:

  1. group advantages from the rewards           (``group_advantages``)
  2. log-softmax of the policy / reference rows  (``log_softmax_rows``)
  3. ratio, clipped surrogate (or CISPO, or the dual clip), the KL estimator
     (k3, k1 or k2), weights, the two-level reduction, dL/dlogp and the clip
     counters                                     (``loss_from_logps``)
  4. dL/dlogits = w (onehot - softmax)            (``grad_rows``)

Parity pins: every function here is checked against closed forms, library
special cases, invariants, finite differences and hand-worked fixtures in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")

F32, BF16, F16, F64 = 0, 1, 2, 3
DTYPE_CODE = {"f32": F32, "bf16": BF16, "f16": F16, "f64": F64}
TOKEN_MEAN, SEQUENCE_MEAN, FIXED_CONSTANT = 0, 1, 2
KL_TYPES = {"k3": 0, "k1": 1, "k2": 2}
SURROGATES = {"clip": 0, "cispo": 1}


def build_commands() -> list[list[str]]:
    return [["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
             "-fno-fast-math", os.path.join(_HERE, "oracle.c"), "-o", _SO, "-lm"]]


def build() -> None:
    for c in build_commands():
        subprocess.run(c, check=True)


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError(f"{_SO} missing: run __graft_entry__.build()")
        L = ctypes.CDLL(_SO)
        i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        L.oracle_group_advantages.argtypes = [vp, i64, vp, i64, dbl, ci, vp]
        L.oracle_group_advantages.restype = ci
        L.oracle_log_softmax_rows.argtypes = [vp, ci, i64, i64, vp, vp, vp]
        L.oracle_loss_from_logps.argtypes = [i64, i64, vp, vp, vp, vp, vp, dbl, dbl, dbl, dbl,
                                             ci, ci, ci, dbl, dbl, ci, vp, vp, vp, vp, vp]
        L.oracle_grad_rows.argtypes = [vp, ci, i64, i64, vp, vp, vp, ci, vp, vp]
        L.oracle_lse_partial.argtypes = [vp, ci, i64, i64, i64, i64, vp, vp]
        L.oracle_lse_merge.argtypes = [i64, i64, vp, vp, vp]
        L.oracle_round_to.argtypes = [vp, i64, ci, vp]
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def _storage_np(dtype: str):
    return {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16, "f64": np.float64}[dtype]


# --------------------------------------------------------------------------
def group_advantages(rewards, bounds, adv_eps: float = 1e-6, eps_add: bool = False) -> np.ndarray:
    """Group-normalised advantages A[B] (double)."""
    r = _c(rewards, np.float32)
    b = _c(bounds, np.int64)
    A = np.zeros(r.shape[0], dtype=np.float64)
    rc = lib().oracle_group_advantages(_p(r), r.shape[0], _p(b), b.shape[0] - 1,
                                       float(adv_eps), int(eps_add), _p(A))
    if rc == 1:
        raise ValueError("invalid group boundaries")
    if rc == 2:
        raise ValueError("non-finite reward")
    return A


def log_softmax_rows(rows, dtype: str, actions=None):
    """rows: [n, V] storage array (float32 / uint16 bits / float64).
    Returns (lse[n], logp[n] or None)."""
    rows = _c(rows, _storage_np(dtype))
    n, V = rows.shape
    lse = np.empty(n, dtype=np.float64)
    logp = None
    a = None
    if actions is not None:
        a = _c(actions, np.int64)
        logp = np.empty(n, dtype=np.float64)
    lib().oracle_log_softmax_rows(_p(rows), DTYPE_CODE[dtype], n, V, _p(a), _p(lse), _p(logp))
    return lse, logp


def loss_from_logps(logp, ref_logp, old, mask, A, eps_lo, eps_hi, beta,
                    grad_scale: float = 1.0, reduction: int = TOKEN_MEAN, kl: str = "k3",
                    surrogate: str = "clip", dual_clip_c: float | None = None,
                    norm_constant: float | None = None, ratio_level: str = "token"):
    """Loss, per-sequence totals and dL/dlogp from per-token log-probs.
    logp / ref_logp / old: [B,T] (any float type, widened to double);
    ref_logp may be None (no KL term).  Variants: kl in {"k3", "k1", "k2"},
    surrogate in {"clip", "cispo"}, the dual clip constant c > 1, and the
    fixed-constant normaliser (reduction FIXED_CONSTANT with norm_constant),
    and ratio_level "sequence" (GSPO: one ratio per sequence, sequence mean
    only, not with CISPO)."""
    lp = _c(logp, np.float64)
    B, T = lp.shape
    rl = None if ref_logp is None else _c(ref_logp, np.float64)
    od = _c(old, np.float64)
    m = _c(mask, np.uint8)
    Ad = _c(A, np.float64)
    if reduction == FIXED_CONSTANT and not (norm_constant and norm_constant > 0):
        raise ValueError("the fixed-constant normaliser needs norm_constant > 0")
    if dual_clip_c is not None and (dual_clip_c <= 1.0 or surrogate != "clip"):
        raise ValueError("the dual clip needs c > 1 and the clipped surrogate")
    if ratio_level not in ("token", "sequence"):
        raise ValueError("ratio_level is 'token' or 'sequence'")
    if ratio_level == "sequence" and (reduction != SEQUENCE_MEAN or surrogate != "clip"):
        raise ValueError("sequence-level ratios need the sequence mean and the clipped surrogate")
    out3 = np.zeros(3, dtype=np.float64)
    per_seq = np.zeros(3 * B, dtype=np.float64)
    w = np.zeros((B, T), dtype=np.float64)
    ratio = np.zeros((B, T), dtype=np.float64)
    counts = np.zeros(3, dtype=np.int64)
    lib().oracle_loss_from_logps(B, T, _p(lp), _p(rl), _p(od), _p(m), _p(Ad), float(eps_lo),
                                 float(eps_hi), float(beta), float(grad_scale), int(reduction),
                                 KL_TYPES[kl], SURROGATES[surrogate], float(dual_clip_c or 0.0),
                                 float(norm_constant or 0.0), int(ratio_level == "sequence"),
                                 _p(out3), _p(per_seq), _p(w), _p(ratio), _p(counts))
    return {"loss": out3[0], "policy_loss": out3[1], "kl": out3[2],
            "per_seq_policy": per_seq[:B], "per_seq_kl": per_seq[B:2 * B],
            "per_seq_active": per_seq[2 * B:], "w": w, "ratio": ratio,
            "clip_counts": counts}


def lse_vocab_parallel(rows, dtype: str, bounds) -> np.ndarray:
    """The rows' logsumexp from vocabulary slices [bounds[k], bounds[k+1]):
    a partial normaliser per slice, merged in slice order (the vocab-parallel
    logprob of the distributed loss)."""
    rows = _c(rows, _storage_np(dtype))
    n, V = rows.shape
    K = len(bounds) - 1
    M = np.empty((K, n), dtype=np.float64)
    Z = np.empty((K, n), dtype=np.float64)
    for k in range(K):
        mk = np.empty(n, dtype=np.float64)
        zk = np.empty(n, dtype=np.float64)
        lib().oracle_lse_partial(_p(rows), DTYPE_CODE[dtype], n, V, int(bounds[k]),
                                 int(bounds[k + 1]), _p(mk), _p(zk))
        M[k], Z[k] = mk, zk
    lse = np.empty(n, dtype=np.float64)
    lib().oracle_lse_merge(n, K, _p(M), _p(Z), _p(lse))
    return lse


def grad_rows(rows, dtype: str, actions, lse, w, out_dtype: str | None = None,
              want_f64: bool = True):
    """dL/dlogits for the given rows.  Returns (rounded storage array,
    unrounded float64 array, or None when want_f64 is False)."""
    out_dtype = out_dtype or dtype
    rows = _c(rows, _storage_np(dtype))
    n, V = rows.shape
    a = _c(actions, np.int64)
    l = _c(lse, np.float64)
    wd = _c(w, np.float64)
    out = np.empty((n, V), dtype=_storage_np(out_dtype))
    f64 = np.empty((n, V), dtype=np.float64) if want_f64 else None
    lib().oracle_grad_rows(_p(rows), DTYPE_CODE[dtype], n, V, _p(a), _p(l), _p(wd),
                           DTYPE_CODE[out_dtype], _p(out), _p(f64))
    return out, f64


def round_to(x, dtype: str) -> np.ndarray:
    """Round doubles to a storage dtype, nearest-even."""
    xd = _c(x, np.float64)
    out = np.empty(xd.shape, dtype=_storage_np(dtype))
    lib().oracle_round_to(_p(xd), xd.size, DTYPE_CODE[dtype], _p(out))
    return out


def widen(a, dtype: str) -> np.ndarray:
    """Storage array -> exact float64 values."""
    a = np.asarray(a)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    return a.astype(np.float64)


def fused(policy, ref, dtype: str, actions, old, mask, rewards, bounds, eps_lo, eps_hi,
          beta, adv_eps: float = 1e-6, eps_add: bool = False, grad_scale: float = 1.0,
          reduction: int = TOKEN_MEAN, out_dtype: str | None = None, want_grad: bool = True,
          **variant):
    """The whole fused path for in-memory [B,T,V] inputs (small sizes).
    `variant` (kl, surrogate, dual_clip_c, norm_constant) goes to
    loss_from_logps unchanged.

    Masked rows are never read: their logits, actions and old_logps may hold
    anything.  Returns a dict with loss, policy_loss, kl, per-sequence
    totals, advantages, per-token logp / ref_logp / ratio / w and, when
    asked, the gradient rounded to out_dtype (and unrounded)."""
    B, T, V = policy.shape
    m = np.asarray(mask).astype(np.uint8)
    A = group_advantages(rewards, bounds, adv_eps, eps_add)
    act = np.nonzero(m.reshape(-1))[0]
    pol_rows = np.asarray(policy).reshape(B * T, V)[act]
    acts = np.asarray(actions).reshape(-1)[act]
    lse_p, lp = log_softmax_rows(pol_rows, dtype, acts)
    logp = np.zeros(B * T)
    logp[act] = lp
    ref_logp = np.zeros(B * T)
    if ref is not None:
        ref_rows = np.asarray(ref).reshape(B * T, V)[act]
        _, rlp = log_softmax_rows(ref_rows, dtype, acts)
        ref_logp[act] = rlp
    oldd = np.zeros(B * T)
    oldd[act] = np.asarray(old, dtype=np.float64).reshape(-1)[act]
    res = loss_from_logps(logp.reshape(B, T), None if ref is None else ref_logp.reshape(B, T),
                          oldd.reshape(B, T), m, A, eps_lo, eps_hi, beta, grad_scale, reduction,
                          **variant)
    res["A"] = A
    res["logp"] = logp.reshape(B, T)
    res["ref_logp"] = ref_logp.reshape(B, T)
    res["lse"] = np.zeros(B * T)
    res["lse"][act] = lse_p
    if want_grad:
        od = out_dtype or dtype
        g = np.zeros((B * T, V), dtype=_storage_np(od))
        g64 = np.zeros((B * T, V), dtype=np.float64)
        if len(act):
            gr, g64r = grad_rows(pol_rows, dtype, acts, lse_p, res["w"].reshape(-1)[act], od)
            g[act] = gr
            g64[act] = g64r
        res["grad"] = g.reshape(B, T, V)
        res["grad_f64"] = g64.reshape(B, T, V)
    return res
