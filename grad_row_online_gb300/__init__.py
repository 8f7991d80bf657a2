"""GB300 (sm_103a) fused GRPO loss: Python binding of libgrpo_gb300.so.

Argument marshalling only: every step of the loss runs in the library's CUDA
kernels (see ``include/grpo.h`` for the exact contract).  PyTorch provides
device memory and the current stream.  If the library is missing this module
raises; there is no fallback.

    import grad_row_online_gb300 as g
    res = g.grpo_loss_fwd_bwd(policy_logits, ref_logits, action_ids, old_logps,
                              completion_mask, rewards, samples_per_prompt=8,
                              clip_eps=0.2, beta=0.04)
    res["loss"], res["policy_loss"], res["kl"], res["grad"]
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = ["grpo_workspace_size", "grpo_group_adv", "grpo_loss_fwd_bwd", "grpo_loss_fwd_bwd_static",
           "grpo_loss_from_logps", "grpo_count_active", "grpo_loss_finalize", "Shard",
           "totals_buffer", "SEQ_TOTAL_BYTES", "grpo_vocab_chunk", "grpo_vocab_partials",
           "grpo_vocab_loss", "grpo_vocab_grad",
           "grpo_read_device_status", "grpo_status_string", "GrpoError", "library_path",
           "GRPO_ADV_EPS_ADD", "GRPO_SKIP_MASKED_GRAD_ROWS"]

GRPO_ADV_EPS_ADD = 1
GRPO_SKIP_MASKED_GRAD_ROWS = 2
GRPO_FLAG_SEPARATE_PREP = 4  # grpo_loss_from_logps: advantages / counts as their own launch
GRPO_FLAG_WORKSPACE_CLEAN = 8  # grpo_loss_from_logps: the header is clean, skip its reset
GRPO_FLAG_OVERLAP_LAUNCH = 16  # grpo_loss_from_logps: dispatch while the previous kernel ends
GRPO_FLAG_TEST_STALLED_COPY = 0x80000000  # test hook (see include/grpo.h)
GRPO_FLAG_TEST_STALLED_BARRIER = 0x40000000  # test hook (see include/grpo.h)
GRPO_ERR_ACTION_RANGE = 16  # device-detected status bits (grpo_read_device_status)
GRPO_ERR_CSR = 32
GRPO_ERR_NONFINITE_REWARD = 64
GRPO_ERR_TIMEOUT = 128
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
_REDUCTIONS = {"token_mean": 0, "sequence_mean": 1, "fixed_constant": 2}
_KL_TYPES = {"k3": 0, "k1": 1, "k2": 2}
_SURROGATES = {"clip": 0, "cispo": 1}


SEQ_TOTAL_BYTES = 32  # one grpo_seq_total_t record


class Shard:
    """A data-parallel shard of the batch: the call's token arguments cover
    sequences [seq_begin, seq_begin + B) of a batch whose rewards and groups
    are passed whole; ``global_counts`` (int64 [2] on the device: N, S of
    the batch) sets the token weights, and the call writes its per-sequence
    totals into ``totals`` (``totals_buffer(B)``) instead of the loss."""

    def __init__(self, seq_begin: int, global_counts: torch.Tensor, totals: torch.Tensor):
        self.seq_begin = int(seq_begin)
        self.global_counts = global_counts
        self.totals = totals


def totals_buffer(B: int, device="cuda") -> torch.Tensor:
    """Device memory for B per-sequence total records (uint8 [B, 32])."""
    return torch.empty((B, SEQ_TOTAL_BYTES), dtype=torch.uint8, device=device)


class GrpoError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {grpo_status_string(code)} (status {code})")
        self.code = code


class _Groups(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int64), ("samples_per_prompt", ctypes.c_int32),
                ("_reserved", ctypes.c_int32), ("group_boundaries", ctypes.c_void_p),
                ("num_groups", ctypes.c_int64)]


class _Profile(ctypes.Structure):
    _fields_ = [("start", ctypes.c_void_p), ("stop", ctypes.c_void_p)]


class _Shard(ctypes.Structure):
    _fields_ = [("seq_begin", ctypes.c_int64), ("global_counts", ctypes.c_void_p),
                ("totals_out", ctypes.c_void_p)]


class _Params(ctypes.Structure):
    _fields_ = [("clip_eps_lo", ctypes.c_float), ("clip_eps_hi", ctypes.c_float),
                ("beta", ctypes.c_float), ("adv_eps", ctypes.c_float),
                ("grad_scale", ctypes.c_float), ("reduction", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("kl_type", ctypes.c_int32),
                ("surrogate", ctypes.c_int32), ("dual_clip_c", ctypes.c_float),
                ("norm_constant", ctypes.c_float), ("ratio_level", ctypes.c_int32),
                ("profile", ctypes.POINTER(_Profile)), ("shard", ctypes.POINTER(_Shard)),
                ("clip_counts", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(_build.LIB)
        vp, i64, f32, u32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32,
                                 ctypes.c_size_t)
        L.grpo_workspace_size.argtypes = [i64, i64, i64]
        L.grpo_workspace_size.restype = sz
        L.grpo_group_adv.argtypes = [vp, ctypes.POINTER(_Groups), f32, u32, vp, vp, sz, vp]
        L.grpo_group_adv.restype = ctypes.c_int
        L.grpo_loss_fwd_bwd.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, vp, vp, vp, vp,
                                        ctypes.POINTER(_Groups), ctypes.POINTER(_Params), vp, vp,
                                        vp, vp, vp, vp, sz, vp]
        L.grpo_loss_fwd_bwd.restype = ctypes.c_int
        L.grpo_loss_fwd_bwd_static.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, vp, vp, vp,
                                               vp, ctypes.POINTER(_Groups),
                                               ctypes.POINTER(_Params), vp, vp, vp, vp, vp, vp]
        L.grpo_loss_fwd_bwd_static.restype = ctypes.c_int
        L.grpo_loss_from_logps.argtypes = [vp, vp, vp, vp, i64, i64, vp, ctypes.POINTER(_Groups),
                                           ctypes.POINTER(_Params), vp, vp, vp, vp, vp, sz, vp]
        L.grpo_loss_from_logps.restype = ctypes.c_int
        L.grpo_count_active.argtypes = [vp, i64, i64, vp, vp]
        L.grpo_count_active.restype = ctypes.c_int
        L.grpo_loss_finalize.argtypes = [vp, i64, vp, ctypes.POINTER(_Params), vp, vp]
        L.grpo_loss_finalize.restype = ctypes.c_int
        L.grpo_vocab_chunk.argtypes = []
        L.grpo_vocab_chunk.restype = sz
        L.grpo_vocab_partials.argtypes = [vp, vp, ctypes.c_int, i64, i64, i64, i64, vp, vp, vp,
                                          vp, vp, vp]
        L.grpo_vocab_partials.restype = ctypes.c_int
        L.grpo_vocab_loss.argtypes = [vp, vp, i64, vp, i64, vp, vp, vp, i64, i64, vp,
                                      ctypes.POINTER(_Groups), ctypes.POINTER(_Params), vp, vp, vp,
                                      vp, vp, vp, sz, vp]
        L.grpo_vocab_loss.restype = ctypes.c_int
        L.grpo_vocab_grad.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, vp, vp, vp, vp, u32,
                                      vp]
        L.grpo_vocab_grad.restype = ctypes.c_int
        L.grpo_read_device_status.argtypes = [vp, vp]
        L.grpo_read_device_status.restype = ctypes.c_int
        L.grpo_status_string.argtypes = [ctypes.c_int]
        L.grpo_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def grpo_status_string(code: int) -> str:
    return lib().grpo_status_string(int(code)).decode()


def grpo_workspace_size(B: int, T: int, num_groups: int = 0) -> int:
    return int(lib().grpo_workspace_size(B, T, num_groups))


# --------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _groups(B: int, samples_per_prompt: int, group_boundaries) -> tuple[_Groups, object]:
    g = _Groups()
    g.num_seqs = B
    g.samples_per_prompt = int(samples_per_prompt or 0)
    keep = None
    if group_boundaries is not None:
        gb = group_boundaries
        if not isinstance(gb, torch.Tensor):
            gb = torch.tensor(list(gb), dtype=torch.int64, device="cuda")
        _dev(gb, "group_boundaries", torch.int64)
        g.group_boundaries = gb.data_ptr()
        g.num_groups = gb.numel() - 1
        keep = gb
    return g, keep


def _params(clip_eps, clip_eps_hi, beta, adv_eps, grad_scale, reduction, flags, profile,
            kl="k3", surrogate="clip", dual_clip_c=None, norm_constant=None, clip_counts=None,
            shard: Optional[Shard] = None, ratio_level: str = "token"):
    p = _Params()
    p.ratio_level = {"token": 0, "sequence": 1}[ratio_level]
    if shard is not None:
        _dev(shard.global_counts, "global_counts", torch.int64)
        _dev(shard.totals, "totals", torch.uint8)
        p._shard = _Shard(shard.seq_begin, shard.global_counts.data_ptr(), shard.totals.data_ptr())
        p.shard = ctypes.pointer(p._shard)
    p.kl_type = _KL_TYPES[kl]
    p.surrogate = _SURROGATES[surrogate]
    p.dual_clip_c = float(dual_clip_c or 0.0)
    p.norm_constant = float(norm_constant or 0.0)
    if clip_counts is not None:
        _dev(clip_counts, "clip_counts", torch.int64)
        p.clip_counts = clip_counts.data_ptr()
    p.clip_eps_lo = float(clip_eps)
    p.clip_eps_hi = float(clip_eps if clip_eps_hi is None else clip_eps_hi)
    p.beta = float(beta)
    p.adv_eps = float(adv_eps)
    p.grad_scale = float(grad_scale)
    p.reduction = _REDUCTIONS[reduction] if isinstance(reduction, str) else int(reduction)
    p.flags = int(flags)
    prof = None
    if profile is not None:
        prof = _Profile(profile[0].cuda_event if hasattr(profile[0], "cuda_event") else profile[0],
                        profile[1].cuda_event if hasattr(profile[1], "cuda_event") else profile[1])
        p.profile = ctypes.pointer(prof)
    return p, prof


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _workspace(B, T, G, workspace, device):
    need = grpo_workspace_size(B, T, G)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace, need


def _check(code: int, what: str):
    if code != 0:
        raise GrpoError(code, what)


def _check_logits_call(policy_logits, ref_logits, action_ids, old_logps, completion_mask,
                       rewards, sharded: bool):
    """Device, dtype, layout and shape checks shared by the logits entry
    points; returns (B, T, V, mask as uint8)."""
    if not isinstance(policy_logits, torch.Tensor) or policy_logits.dtype not in _DTYPES:
        raise ValueError(f"unsupported logits dtype {getattr(policy_logits, 'dtype', None)}")
    _dev(policy_logits, "policy_logits")
    _dev(ref_logits, "ref_logits", policy_logits.dtype)
    if policy_logits.dim() != 3 or ref_logits.shape != policy_logits.shape:
        raise ValueError("policy_logits and ref_logits must both be [B, T, V]")
    B, T, V = policy_logits.shape
    _dev(action_ids, "action_ids", torch.int64)
    _dev(old_logps, "old_logps", torch.float32)
    _dev(rewards, "rewards", torch.float32)
    mask = _dev(completion_mask, "completion_mask")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    elif mask.dtype != torch.uint8:
        raise ValueError("completion_mask must be bool or uint8")
    if action_ids.shape != (B, T) or old_logps.shape != (B, T) or mask.shape != (B, T):
        raise ValueError("action_ids, old_logps and completion_mask must be [B, T]")
    if not sharded and rewards.shape != (B,):
        raise ValueError("rewards must be [B]")
    devs = {t.device for t in (ref_logits, action_ids, old_logps, rewards, mask)}
    if devs != {policy_logits.device}:
        raise ValueError("every tensor must be on the device of policy_logits")
    return B, T, V, mask


# --------------------------------------------------------------------------
def grpo_group_adv(rewards: torch.Tensor, *, samples_per_prompt: int = 0, group_boundaries=None,
                   adv_eps: float = 1e-6, eps_add: bool = False, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Group-normalised advantages [B] (f32)."""
    _dev(rewards, "rewards", torch.float32)
    B = rewards.numel()
    g, keep = _groups(B, samples_per_prompt, group_boundaries)
    out = torch.empty(B, dtype=torch.float32, device=rewards.device) if out is None else out
    ws, need = _workspace(B, 0, 0, workspace, rewards.device)
    rc = lib().grpo_group_adv(_ptr(rewards), ctypes.byref(g), float(adv_eps),
                              GRPO_ADV_EPS_ADD if eps_add else 0, _ptr(out), _ptr(ws),
                              ws.numel(), _stream(stream))
    _check(rc, "grpo_group_adv")
    return out


def grpo_loss_fwd_bwd(policy_logits: torch.Tensor, ref_logits: torch.Tensor,
                      action_ids: torch.Tensor, old_logps: torch.Tensor,
                      completion_mask: torch.Tensor, rewards: torch.Tensor, *,
                      samples_per_prompt: int = 0, group_boundaries=None, clip_eps: float = 0.2,
                      clip_eps_hi: Optional[float] = None, beta: float = 0.04,
                      adv_eps: float = 1e-6, eps_add: bool = False, grad_scale: float = 1.0,
                      reduction="token_mean", grad=True, skip_masked_grad_rows: bool = False,
                      want_per_seq: bool = False, want_logps: bool = False,
                      want_adv: bool = False, out3: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None,
                      profile=None, kl: str = "k3", surrogate: str = "clip",
                      dual_clip_c: Optional[float] = None, norm_constant: Optional[float] = None,
                      want_clip_counts: bool = False, shard: Optional[Shard] = None,
                      ratio_level: str = "token") -> dict:
    """Fused GRPO loss forward + dL/dlogits.

    ``grad``: True (allocate), a tensor to write into (may be
    ``policy_logits`` itself for an in-place gradient), or None/False
    (forward only).  Variants: ``kl`` in {"k3", "k1", "k2"}, ``surrogate``
    in {"clip", "cispo"}, ``dual_clip_c`` (> 1), ``reduction=
    "fixed_constant"`` with ``norm_constant``, ``ratio_level="sequence"``
    (GSPO, with ``reduction="sequence_mean"``).  Returns a dict of device
    tensors: ``out3`` ([loss, policy_loss, kl]), ``loss``, ``policy_loss``,
    ``kl`` (0-d views), ``grad``, and the optional ``per_seq`` [3,B],
    ``logps`` [B,T], ``adv`` [B], ``clip_counts`` [3] (int64: clipped at the
    upper bound, at the lower bound, by the dual clip).  With ``shard``
    (see ``Shard``) ``rewards`` and the groups span the whole batch, the
    token tensors the shard's sequences, and ``out3`` is not written."""
    B, T, V, mask = _check_logits_call(policy_logits, ref_logits, action_ids, old_logps,
                                       completion_mask, rewards, shard is not None)
    dev = policy_logits.device
    g, keep = _groups(rewards.numel() if shard is not None else B, samples_per_prompt,
                      group_boundaries)
    counts = torch.empty(3, dtype=torch.int64, device=dev) if want_clip_counts else None
    p, prof = _params(clip_eps, clip_eps_hi, beta, adv_eps, grad_scale, reduction,
                      (GRPO_ADV_EPS_ADD if eps_add else 0)
                      | (GRPO_SKIP_MASKED_GRAD_ROWS if skip_masked_grad_rows else 0), profile,
                      kl, surrogate, dual_clip_c, norm_constant, counts, shard, ratio_level)
    if grad is True:
        grad_t = torch.empty_like(policy_logits)
    elif grad is None or grad is False:
        grad_t = None
    else:
        grad_t = _dev(grad, "grad", policy_logits.dtype)
        if grad_t.shape != policy_logits.shape:
            raise ValueError("grad must have the shape of policy_logits")
    out3 = torch.empty(3, dtype=torch.float32, device=dev) if out3 is None else out3
    per_seq = torch.empty((3, B), dtype=torch.float32, device=dev) if want_per_seq else None
    logps = torch.empty((B, T), dtype=torch.float32, device=dev) if want_logps else None
    adv = torch.empty(B, dtype=torch.float32, device=dev) if want_adv else None
    ws, need = _workspace(rewards.numel() if shard is not None else B, T, 0, workspace, dev)
    rc = lib().grpo_loss_fwd_bwd(_ptr(policy_logits), _ptr(ref_logits), _DTYPES[policy_logits.dtype],
                                 B, T, V, _ptr(action_ids), _ptr(old_logps), _ptr(mask),
                                 _ptr(rewards), ctypes.byref(g), ctypes.byref(p), _ptr(grad_t),
                                 _ptr(out3), _ptr(per_seq), _ptr(logps), _ptr(adv), _ptr(ws),
                                 ws.numel(), _stream(stream))
    _check(rc, "grpo_loss_fwd_bwd")
    return {"out3": out3, "loss": out3[0], "policy_loss": out3[1], "kl": out3[2],
            "grad": grad_t, "per_seq": per_seq, "logps": logps, "adv": adv,
            "clip_counts": counts, "workspace": ws}


def grpo_loss_fwd_bwd_static(policy_logits: torch.Tensor, ref_logits: torch.Tensor,
                             action_ids: torch.Tensor, old_logps: torch.Tensor,
                             completion_mask: torch.Tensor, rewards: torch.Tensor, *,
                             samples_per_prompt: int = 0, group_boundaries=None,
                             clip_eps: float = 0.2, clip_eps_hi: Optional[float] = None,
                             beta: float = 0.04, adv_eps: float = 1e-6, eps_add: bool = False,
                             grad_scale: float = 1.0, reduction="token_mean",
                             grad: Optional[torch.Tensor] = None, out3: Optional[torch.Tensor] = None,
                             stream=None) -> int:
    """grpo_loss_fwd_bwd with the library's fixed scratch memory instead of a
    workspace, for callers that cannot allocate device memory at the call
    (e.g. inside CUDA graph capture).  Every output is caller-provided:
    `out3` ([3] f32) and, optionally, `grad` (like policy_logits);
    `group_boundaries`, if given, must already be an int64 device tensor.
    The arguments are checked as in grpo_loss_fwd_bwd (ValueError).  Returns
    the status code (0 = ok); nothing is allocated by this call."""
    B, T, V, mask = _check_logits_call(policy_logits, ref_logits, action_ids, old_logps,
                                       completion_mask, rewards, False)
    if out3 is None:
        raise ValueError("out3 ([3] float32 on the device) is required")
    _dev(out3, "out3", torch.float32)
    if out3.shape != (3,) or out3.device != policy_logits.device:
        raise ValueError("out3 must be [3] on the device of policy_logits")
    if grad is not None:
        _dev(grad, "grad", policy_logits.dtype)
        if grad.shape != policy_logits.shape or grad.device != policy_logits.device:
            raise ValueError("grad must have the shape and device of policy_logits")
    if group_boundaries is not None and not isinstance(group_boundaries, torch.Tensor):
        raise ValueError("group_boundaries must be an int64 device tensor here (a list would "
                         "need an allocation and a host-to-device copy)")
    g, keep = _groups(B, samples_per_prompt, group_boundaries)
    p, prof = _params(clip_eps, clip_eps_hi, beta, adv_eps, grad_scale, reduction,
                      GRPO_ADV_EPS_ADD if eps_add else 0, None)
    return int(lib().grpo_loss_fwd_bwd_static(
        _ptr(policy_logits), _ptr(ref_logits), _DTYPES[policy_logits.dtype], B, T, V,
        _ptr(action_ids), _ptr(old_logps), _ptr(mask), _ptr(rewards), ctypes.byref(g),
        ctypes.byref(p), _ptr(grad), _ptr(out3), None, None, None, _stream(stream)))


def grpo_loss_from_logps(logps: torch.Tensor, old_logps: torch.Tensor,
                         ref_logps: Optional[torch.Tensor], completion_mask: torch.Tensor,
                         rewards: torch.Tensor, *, samples_per_prompt: int = 0,
                         group_boundaries=None, clip_eps: float = 0.2,
                         clip_eps_hi: Optional[float] = None, beta: float = 0.04,
                         adv_eps: float = 1e-6, eps_add: bool = False, grad_scale: float = 1.0,
                         reduction="token_mean", grad=True, want_per_seq: bool = False,
                         want_adv: bool = False, out3: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None,
                         profile=None, kl: str = "k3", surrogate: str = "clip",
                         dual_clip_c: Optional[float] = None,
                         norm_constant: Optional[float] = None,
                         want_clip_counts: bool = False, shard: Optional[Shard] = None,
                         ratio_level: str = "token", workspace_clean: bool = False,
                         overlap_launch: bool = False, extra_flags: int = 0) -> dict:
    """GRPO loss from per-token log-probs; ``grad`` gives dL/dlogp [B,T].
    Variants, outputs and ``shard`` as in grpo_loss_fwd_bwd.
    ``workspace_clean``: the given ``workspace`` was last used by a
    grpo_loss_from_logps call that succeeded (or was zeroed), so its header
    is clean and the call skips resetting it (GRPO_FLAG_WORKSPACE_CLEAN; a
    workspace allocated here is never clean).  ``overlap_launch``: the
    one-launch form is dispatched while the previous kernel on the stream
    ends instead of cooperatively; the caller states that no other kernel
    holds SMs for long meanwhile (GRPO_FLAG_OVERLAP_LAUNCH, include/grpo.h).
    ``extra_flags``
    are raw grpo_params_t flag bits (e.g. GRPO_FLAG_TEST_STALLED_COPY)."""
    _dev(logps, "logps", torch.float32)
    B, T = logps.shape
    _dev(old_logps, "old_logps", torch.float32)
    if ref_logps is not None:
        _dev(ref_logps, "ref_logps", torch.float32)
    _dev(rewards, "rewards", torch.float32)
    mask = _dev(completion_mask, "completion_mask")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    dev = logps.device
    Bg = rewards.numel() if shard is not None else B
    g, keep = _groups(Bg, samples_per_prompt, group_boundaries)
    counts = torch.empty(3, dtype=torch.int64, device=dev) if want_clip_counts else None
    p, prof = _params(clip_eps, clip_eps_hi, beta, adv_eps, grad_scale, reduction,
                      (GRPO_ADV_EPS_ADD if eps_add else 0)
                      | (GRPO_FLAG_WORKSPACE_CLEAN if workspace_clean and workspace is not None
                         else 0) | (GRPO_FLAG_OVERLAP_LAUNCH if overlap_launch else 0)
                      | int(extra_flags), profile, kl,
                      surrogate, dual_clip_c, norm_constant, counts, shard, ratio_level)
    if grad is True:
        grad_t = torch.empty((B, T), dtype=torch.float32, device=dev)
    elif grad is None or grad is False:
        grad_t = None
    else:
        grad_t = _dev(grad, "grad", torch.float32)
    out3 = torch.empty(3, dtype=torch.float32, device=dev) if out3 is None else out3
    per_seq = torch.empty((3, B), dtype=torch.float32, device=dev) if want_per_seq else None
    adv = torch.empty(B, dtype=torch.float32, device=dev) if want_adv else None
    ws, need = _workspace(Bg, T, 0, workspace, dev)
    rc = lib().grpo_loss_from_logps(_ptr(logps), _ptr(old_logps), _ptr(ref_logps), _ptr(mask),
                                    B, T, _ptr(rewards), ctypes.byref(g), ctypes.byref(p),
                                    _ptr(grad_t), _ptr(out3), _ptr(per_seq), _ptr(adv), _ptr(ws),
                                    ws.numel(), _stream(stream))
    _check(rc, "grpo_loss_from_logps")
    return {"out3": out3, "loss": out3[0], "policy_loss": out3[1], "kl": out3[2],
            "grad": grad_t, "per_seq": per_seq, "adv": adv, "clip_counts": counts,
            "workspace": ws}


def grpo_count_active(completion_mask: torch.Tensor, out: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """N (active tokens) and S (sequences with one) of a [B,T] mask, as an
    int64 [2] device tensor: a shard's contribution to the batch counts."""
    mask = _dev(completion_mask, "completion_mask")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    B, T = mask.shape
    out = torch.empty(2, dtype=torch.int64, device=mask.device) if out is None else out
    _check(lib().grpo_count_active(_ptr(mask), B, T, _ptr(out), _stream(stream)),
           "grpo_count_active")
    return out


def grpo_loss_finalize(totals: torch.Tensor, global_counts: torch.Tensor, *, beta: float = 0.04,
                       reduction="token_mean", norm_constant: Optional[float] = None,
                       out3: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """[loss, policy_loss, kl] from the whole batch's per-sequence totals
    (every shard's ``totals`` concatenated in shard order, uint8 [B, 32])
    and the batch counts -- bit-identical to the unsharded call."""
    _dev(totals, "totals", torch.uint8)
    _dev(global_counts, "global_counts", torch.int64)
    B = totals.shape[0]
    p, _ = _params(0.2, None, beta, 1e-6, 1.0, reduction, 0, None, norm_constant=norm_constant)
    out3 = torch.empty(3, dtype=torch.float32, device=totals.device) if out3 is None else out3
    _check(lib().grpo_loss_finalize(_ptr(totals), B, _ptr(global_counts), ctypes.byref(p),
                                    _ptr(out3), _stream(stream)), "grpo_loss_finalize")
    return out3


# --------------------------------------------------------------------------
# vocabulary parallelism (see include/grpo.h): partials -> exchange -> loss ->
# gradient slices
def grpo_vocab_chunk() -> int:
    return int(lib().grpo_vocab_chunk())


def grpo_vocab_partials(policy_slice: torch.Tensor, ref_slice: torch.Tensor,
                        action_ids: torch.Tensor, completion_mask: torch.Tensor, v_begin: int,
                        stream=None) -> dict:
    """This rank's partial normalisers: ``part_p`` / ``part_r`` (float32
    [chunks, B*T, 4] records) and ``action_logits`` ([2, B*T], 0 where the
    slice does not hold the action)."""
    if policy_slice.dtype not in _DTYPES:
        raise ValueError(f"unsupported logits dtype {policy_slice.dtype}")
    _dev(policy_slice, "policy_slice")
    _dev(ref_slice, "ref_slice", policy_slice.dtype)
    B, T, Vk = policy_slice.shape
    _dev(action_ids, "action_ids", torch.int64)
    mask = _dev(completion_mask, "completion_mask")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    C = grpo_vocab_chunk()
    nck = (Vk + C - 1) // C
    dev = policy_slice.device
    part_p = torch.empty((nck, B * T, 4), dtype=torch.float32, device=dev)
    part_r = torch.empty((nck, B * T, 4), dtype=torch.float32, device=dev)
    act = torch.empty((2, B * T), dtype=torch.float32, device=dev)
    _check(lib().grpo_vocab_partials(_ptr(policy_slice), _ptr(ref_slice),
                                     _DTYPES[policy_slice.dtype], B, T, Vk, int(v_begin),
                                     _ptr(action_ids), _ptr(mask), _ptr(part_p), _ptr(part_r),
                                     _ptr(act), _stream(stream)), "grpo_vocab_partials")
    return {"part_p": part_p, "part_r": part_r, "action_logits": act}


def grpo_vocab_loss(part_p: torch.Tensor, part_r: torch.Tensor, action_logits: torch.Tensor,
                    V: int, action_ids: torch.Tensor, old_logps: torch.Tensor,
                    completion_mask: torch.Tensor, rewards: torch.Tensor, *,
                    samples_per_prompt: int = 0, group_boundaries=None, clip_eps: float = 0.2,
                    clip_eps_hi: Optional[float] = None, beta: float = 0.04,
                    adv_eps: float = 1e-6, eps_add: bool = False, grad_scale: float = 1.0,
                    reduction="token_mean", want_per_seq: bool = False, want_logps: bool = False,
                    want_adv: bool = False, workspace: Optional[torch.Tensor] = None,
                    stream=None, kl: str = "k3", surrogate: str = "clip",
                    dual_clip_c: Optional[float] = None, norm_constant: Optional[float] = None,
                    want_clip_counts: bool = False, shard: Optional[Shard] = None,
                    ratio_level: str = "token") -> dict:
    """The loss from every slice's partials (concatenated in rank order) and
    the summed action logits.  Returns ``out3``, ``lse_w`` ([2, B*T] double:
    logsumexp and dL/dlogp per row, for grpo_vocab_grad) and the optional
    outputs of grpo_loss_fwd_bwd."""
    B, T = action_ids.shape
    dev = action_ids.device
    for t, n in ((part_p, "part_p"), (part_r, "part_r")):
        _dev(t, n, torch.float32)
    _dev(action_logits, "action_logits", torch.float32)
    _dev(old_logps, "old_logps", torch.float32)
    _dev(rewards, "rewards", torch.float32)
    mask = _dev(completion_mask, "completion_mask")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    Bg = rewards.numel() if shard is not None else B
    g, keep = _groups(Bg, samples_per_prompt, group_boundaries)
    counts = torch.empty(3, dtype=torch.int64, device=dev) if want_clip_counts else None
    p, prof = _params(clip_eps, clip_eps_hi, beta, adv_eps, grad_scale, reduction,
                      GRPO_ADV_EPS_ADD if eps_add else 0, None, kl, surrogate, dual_clip_c,
                      norm_constant, counts, shard, ratio_level)
    out3 = torch.empty(3, dtype=torch.float32, device=dev)
    lse_w = torch.empty((2, B * T), dtype=torch.float64, device=dev)
    per_seq = torch.empty((3, B), dtype=torch.float32, device=dev) if want_per_seq else None
    logps = torch.empty((B, T), dtype=torch.float32, device=dev) if want_logps else None
    adv = torch.empty(B, dtype=torch.float32, device=dev) if want_adv else None
    ws, need = _workspace(Bg, T, 0, workspace, dev)
    _check(lib().grpo_vocab_loss(_ptr(part_p), _ptr(part_r), part_p.shape[0], _ptr(action_logits),
                                 int(V), _ptr(action_ids), _ptr(old_logps), _ptr(mask), B, T,
                                 _ptr(rewards), ctypes.byref(g), ctypes.byref(p), _ptr(lse_w),
                                 _ptr(out3), _ptr(per_seq), _ptr(logps), _ptr(adv), _ptr(ws),
                                 ws.numel(), _stream(stream)), "grpo_vocab_loss")
    return {"out3": out3, "loss": out3[0], "policy_loss": out3[1], "kl": out3[2],
            "lse_w": lse_w, "per_seq": per_seq, "logps": logps, "adv": adv,
            "clip_counts": counts, "workspace": ws}


def grpo_vocab_grad(policy_slice: torch.Tensor, action_ids: torch.Tensor,
                    completion_mask: torch.Tensor, v_begin: int, lse_w: torch.Tensor, *,
                    grad: Optional[torch.Tensor] = None, skip_masked_grad_rows: bool = False,
                    stream=None) -> torch.Tensor:
    """This rank's slice of dL/dlogits ([B, T, Vk], the dtype of the slice)."""
    _dev(policy_slice, "policy_slice")
    B, T, Vk = policy_slice.shape
    mask = _dev(completion_mask, "completion_mask")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    _dev(lse_w, "lse_w", torch.float64)
    grad = torch.empty_like(policy_slice) if grad is None else _dev(grad, "grad",
                                                                   policy_slice.dtype)
    _check(lib().grpo_vocab_grad(_ptr(policy_slice), _DTYPES[policy_slice.dtype], B, T, Vk,
                                 int(v_begin), _ptr(action_ids), _ptr(mask), _ptr(lse_w),
                                 _ptr(grad), GRPO_SKIP_MASKED_GRAD_ROWS if skip_masked_grad_rows
                                 else 0, _stream(stream)), "grpo_vocab_grad")
    return grad


def grpo_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises and returns the device status word of a workspace."""
    return int(lib().grpo_read_device_status(_ptr(workspace), _stream(stream)))
