"""Inputs and oracle expectations for the parity tests.

Inputs come from ``synth`` (seeded); the behaviour log-prob
``old_logps = exact policy log-prob of the action + old_sigma * N(0,1)`` takes
its exact log-prob from the oracle.  Nothing here reads a CUDA result to build
an input or an expectation.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

BF16_MIN_NORMAL_EXP = -126
ACTIVE_CHUNK = 256


# ---------------------------------------------------------------------------
# tolerances
# ---------------------------------------------------------------------------
def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the storage dtype at |x| (x already rounded to it)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    if dtype == "f32":
        return np.spacing(a.astype(np.float32)).astype(np.float64)
    prec, emin = (8, -126) if dtype == "bf16" else (11, -14)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # zero: the spacing of the subnormals, as for every value below 2^emin
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return np.ldexp(1.0, (e - (prec - 1)).astype(np.int64))


_PREC = {"f32": (24, -126), "bf16": (8, -126), "f16": (11, -14)}


def ulp_device(o: torch.Tensor, dtype: str) -> torch.Tensor:
    """ulp() on the device: o holds float64 values exactly representable in
    the storage dtype."""
    prec, emin = _PREC[dtype]
    _, e = torch.frexp(o.abs())  # |o| = m 2^e, m in [1/2, 1): floor(log2|o|) = e - 1
    e = torch.where(o != 0, torch.clamp(e - 1, min=emin), torch.full_like(e, emin))
    return torch.ldexp(torch.ones_like(o), (e - (prec - 1)).to(o.dtype))


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.widen(a, dtype)


def torch_storage(t: torch.Tensor) -> np.ndarray:
    """Device/host tensor -> numpy storage array (float32, or uint16 bits)."""
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.uint16).numpy()
    return t.numpy()


def assert_scalar(got: float, want: float, what: str, rel: float = 1e-5):
    assert abs(got - want) <= rel * abs(want) + 1e-12, f"{what}: gpu {got!r} oracle {want!r}"


# ---------------------------------------------------------------------------
# small cases: everything in host memory
# ---------------------------------------------------------------------------
def make_case(w: synth.Workload, dtype: str | None = None) -> dict:
    """Host inputs of a workload.  dtype "f16" stores the f32 draws as f16."""
    dtype = dtype or w.dtype
    base = w.with_(dtype="bf16" if dtype == "bf16" else "f32")
    X = base.logits_host("policy")
    Y = base.logits_host("ref")
    if dtype == "f16":
        X = torch.from_numpy(X).half().view(torch.uint16).numpy()
        Y = torch.from_numpy(Y).half().view(torch.uint16).numpy()
    acts = w.action_ids()
    mask = w.completion_mask()
    _, lp = oracle.log_softmax_rows(X.reshape(-1, w.V), dtype, acts.reshape(-1))
    old = (lp.reshape(w.B, w.T) + w.old_sigma * w.old_noise()).astype(np.float32)
    return dict(w=w, dtype=dtype, X=X, Y=Y, acts=acts, mask=mask, old=old, R=w.rewards(),
                bounds=w.group_boundaries())


def expect(case: dict, *, eps_lo=None, eps_hi=None, beta=None, reduction=None, eps_add=False,
           grad_scale=1.0, ref_is_policy=False, want_grad=True) -> dict:
    w = case["w"]
    return oracle.fused(case["X"], case["X"] if ref_is_policy else case["Y"], case["dtype"],
                        case["acts"], case["old"], case["mask"], case["R"], case["bounds"],
                        w.eps_lo if eps_lo is None else eps_lo,
                        w.eps_hi if eps_hi is None else eps_hi,
                        w.beta if beta is None else beta, eps_add=eps_add, grad_scale=grad_scale,
                        reduction=w.reduction if reduction is None else reduction,
                        want_grad=want_grad)


def to_device(case: dict, device="cuda") -> dict:
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[case["dtype"]]

    def logits(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if case["dtype"] != "f32":
            t = t.view(tdt)
        return t.to(device)

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return dict(X=logits(case["X"]), Y=logits(case["Y"]), acts=t(case["acts"]),
                old=t(case["old"]), mask=t(case["mask"]), R=t(case["R"]),
                bounds=t(case["bounds"]))


def clip_band_rows(exp: dict, eps_lo: float, eps_hi: float, band: float = 1e-6) -> np.ndarray:
    """Active tokens whose oracle ratio sits within `band` (relative) of a clip
    bound: there the fp32 and fp64 evaluations may take different branches of
    the clipped surrogate, and both gradients are correct readings."""
    r = exp["ratio"]
    lo = 1.0 - float(np.float32(eps_lo))
    hi = 1.0 + float(np.float32(eps_hi))
    return (np.abs(r - lo) <= band * lo) | (np.abs(r - hi) <= band * hi)


def assert_grad_rows(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "grad",
                     alt: np.ndarray | None = None):
    """|gpu - oracle_rounded| <= ulp_dtype(oracle_rounded) + 1e-9 elementwise;
    rows listed in `alt` may match the alternative expectation instead."""
    g = storage_to_f64(got, dtype)
    o = storage_to_f64(want, dtype)
    err = np.abs(g - o)
    tol = ulp(o, dtype) + 1e-9
    bad = err > tol
    if alt is not None:
        oa = storage_to_f64(alt, dtype)
        bad &= np.abs(g - oa) > ulp(oa, dtype) + 1e-9
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance, e.g. "
                             + ", ".join(f"{tuple(i)} gpu={g[tuple(i)]:.9g} oracle={o[tuple(i)]:.9g}"
                                         for i in idx))


def assert_grad_rows_streamed(w: synth.Workload, X: torch.Tensor, grad: torch.Tensor,
                              exp: dict, rows: np.ndarray, chunk: int = 256) -> int:
    """Every element of the gradient rows `rows` (flat row indices) against
    the oracle, |gpu - oracle_rounded| <= ulp_dtype(oracle_rounded) + 1e-9,
    in chunks: the policy rows are copied to the host for the oracle, whose
    rounded rows go back to the device for the comparison.  Returns the
    number of elements checked."""
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.dtype]
    Xf, Gf = X.view(-1, w.V), grad.view(-1, w.V)
    wflat = exp["w"].reshape(-1)
    n = 0
    for i in range(0, len(rows), chunk):
        r = rows[i:i + chunk]
        idx = torch.as_tensor(r, device=X.device)
        xs = torch_storage(Xf[idx])
        want, _ = oracle.grad_rows(xs, w.dtype, exp["acts"][r], exp["lse"][r], wflat[r],
                                   want_f64=False)
        wt = torch.from_numpy(want).to(X.device)
        if w.dtype != "f32":
            wt = wt.view(tdt)
        o = wt.to(torch.float64)
        g = Gf[idx].to(torch.float64)
        bad = (g - o).abs() > ulp_device(o, w.dtype) + 1e-9
        if bool(bad.any()):
            k = torch.nonzero(bad)[:5].cpu().numpy()
            raise AssertionError(
                f"{w.name} grad: {int(bad.sum())} elements out of tolerance in rows "
                f"{r[0]}..{r[-1]}, e.g. " + ", ".join(
                    f"row {r[a]} col {b} gpu={float(g[a, b]):.9g} oracle={float(o[a, b]):.9g}"
                    for a, b in k))
        n += len(r) * w.V
    return n


# ---------------------------------------------------------------------------
# full-size workloads: inputs generated in device memory, oracle streamed
# ---------------------------------------------------------------------------
def device_logits(w: synth.Workload):
    """Policy and reference logits of a workload, generated on the device."""
    X = w.logits_device("policy")
    Y = w.logits_device("ref")
    torch.cuda.synchronize()
    return X, Y


def check_device_generator(w: synth.Workload, X, Y, rows) -> None:
    """The device generator must give the host generator's bits."""
    for which, T in (("policy", X), ("ref", Y)):
        got = torch_storage(T.view(-1, w.V)[torch.as_tensor(rows, device=T.device)])
        want = w.logit_rows(which, rows)
        assert np.array_equal(got, want), f"device generator differs from host ({which})"


def stream_oracle(w: synth.Workload, X, Y, chunk: int = 1024) -> dict:
    """Oracle log-softmax of every active row, streamed in row chunks copied
    from the generated device tensors, then the loss from the log-probs."""
    mask = w.completion_mask()
    acts = w.action_ids().reshape(-1)
    active = np.nonzero(mask.reshape(-1))[0]
    BT = w.rows
    logp = np.zeros(BT)
    ref_logp = np.zeros(BT)
    lse = np.zeros(BT)
    Xf, Yf = X.view(-1, w.V), Y.view(-1, w.V)
    for i in range(0, len(active), chunk):
        rows = active[i:i + chunk]
        ridx = torch.as_tensor(rows, device=X.device)
        xs = torch_storage(Xf[ridx])
        ys = torch_storage(Yf[ridx])
        l, lp = oracle.log_softmax_rows(xs, w.dtype, acts[rows])
        _, rl = oracle.log_softmax_rows(ys, w.dtype, acts[rows])
        lse[rows] = l
        logp[rows] = lp
        ref_logp[rows] = rl
    old = np.zeros(BT, dtype=np.float32)
    noise = w.old_noise().reshape(-1)
    old[active] = (logp[active] + w.old_sigma * noise[active]).astype(np.float32)
    R = w.rewards()
    bounds = w.group_boundaries()
    A = oracle.group_advantages(R, bounds)
    res = oracle.loss_from_logps(logp.reshape(w.B, w.T), ref_logp.reshape(w.B, w.T),
                                 old.reshape(w.B, w.T), mask, A, w.eps_lo, w.eps_hi, w.beta,
                                 reduction=w.reduction)
    res.update(A=A, logp=logp.reshape(w.B, w.T), lse=lse, mask=mask, acts=acts, old=old.reshape(w.B, w.T),
               R=R, bounds=bounds, active=active)
    return res
