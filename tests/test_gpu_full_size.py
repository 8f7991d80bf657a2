"""Parity at the full benchmark sizes, in the launch configuration the
benchmark times.  Inputs are generated in device memory by the seeded
generator (checked bit for bit against the host generator on sampled rows);
the oracle streams every active row for the loss, the per-sequence totals and
every log-prob, then again for every element of every active gradient row."""
import numpy as np
import pytest
import torch

import grad_row_online_gb300 as g
import oracle
import synth
from workload_inputs import (assert_grad_rows_streamed, assert_scalar, check_device_generator,
                             device_logits, stream_oracle)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    import __graft_entry__
    if not os.path.exists(g.library_path()):
        __graft_entry__.build()


def _run_full(w, X, Y, exp, grad=True):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction,
                want_per_seq=True, want_logps=True, want_adv=True, grad=grad)
    if w.samples_per_prompt:
        args["samples_per_prompt"] = w.samples_per_prompt
    else:
        args["group_boundaries"] = t(exp["bounds"])
    res = g.grpo_loss_fwd_bwd(X, Y, t(exp["acts"].reshape(w.B, w.T)), t(exp["old"]),
                              t(exp["mask"]), t(exp["R"]), **args)
    torch.cuda.synchronize()
    assert g.grpo_read_device_status(res["workspace"]) == 0
    return res


@pytest.mark.parametrize("name", ["fused", "large_vocab", "var_groups"])
def test_full_size_logits_workload(name):
    w = synth.WORKLOADS[name]
    X, Y = device_logits(w)
    rng = np.random.default_rng(7)
    check_device_generator(w, X, Y, rng.choice(w.rows, 8, replace=False))
    exp = stream_oracle(w, X, Y)
    res = _run_full(w, X, Y, exp)

    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    ps = res["per_seq"].cpu().numpy().astype(np.float64)
    assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-4)
    assert np.allclose(ps[1], exp["per_seq_kl"], rtol=1e-5, atol=1e-5)
    assert np.array_equal(ps[2], exp["per_seq_active"])
    m = exp["mask"].astype(bool)
    lp = res["logps"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lp[m] - exp["logp"][m]) <= 4e-6 + 1e-6 * np.abs(exp["logp"][m]))

    # gradient: every element of every active row against the oracle (rows of
    # tokens whose ratio sits at a clip kink may take either branch, and are
    # left out), masked rows all zero
    grad = res["grad"].view(-1, w.V)
    active = exp["active"]
    lo, hi = 1.0 - float(np.float32(w.eps_lo)), 1.0 + float(np.float32(w.eps_hi))
    r = exp["ratio"].reshape(-1)[active]
    kink = (np.abs(r - lo) <= 1e-6 * lo) | (np.abs(r - hi) <= 1e-6 * hi)
    checked = assert_grad_rows_streamed(w, X, res["grad"], exp, active[~kink])
    assert checked == int((~kink).sum()) * w.V and kink.sum() <= 2, kink.sum()
    mrows = torch.as_tensor(np.nonzero(~m.reshape(-1))[0], device="cuda")
    if len(mrows):
        assert grad[mrows].abs().max().item() == 0.0


@pytest.mark.parametrize("name", ["logps", "logps_full"])
def test_full_size_logps_workload(name):
    w = synth.WORKLOADS[name]
    lp, old, ref = w.logps_inputs()
    mask = w.completion_mask()
    R = w.rewards()
    A = oracle.group_advantages(R, w.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, mask, A, w.eps_lo, w.eps_hi, w.beta,
                                 reduction=w.reduction)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    res = g.grpo_loss_from_logps(t(lp), t(old), t(ref), t(mask), t(R),
                                 samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                 clip_eps_hi=w.eps_hi, beta=w.beta, want_per_seq=True)
    torch.cuda.synchronize()
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    got = res["grad"].cpu().numpy().astype(np.float64)
    want = exp["w"].astype(np.float32).astype(np.float64)
    r = exp["ratio"]
    band = (np.abs(r - (1 - np.float32(w.eps_lo))) < 1e-6) | (np.abs(r - (1 + np.float32(w.eps_hi))) < 1e-6)
    ok = np.abs(got - want) <= np.spacing(np.abs(want).astype(np.float32)) + 1e-9
    assert np.all(ok | band)
    assert np.array_equal(res["per_seq"][2].cpu().numpy(), exp["per_seq_active"].astype(np.float32))
