"""grpo_loss_fwd_bwd_static: the entry point for callers that cannot
allocate device memory where they compute the loss (for instance inside a
CUDA graph capture, or when another allocator owns the device memory).  It
runs on the library's fixed scratch array instead of a caller workspace.

Checked through the C ABI against grpo_loss_fwd_bwd on the same inputs, on
two calls in a row (the shared scratch keeps the previous call's contents):
both run the same deterministic kernels, so the results must be the same
bits.  One case also goes against the oracle, with the parity tests'
tolerances, and the Python wrapper is checked to validate its arguments
the way the workspace wrapper does.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import grad_row_online_gb300 as g
import synth
from workload_inputs import (assert_grad_rows, assert_scalar, expect, make_case, to_device,
                             torch_storage)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    import __graft_entry__
    if not os.path.exists(g.library_path()):
        __graft_entry__.build()


def _params(w):
    p = g._Params()
    p.clip_eps_lo, p.clip_eps_hi, p.beta = w.eps_lo, w.eps_hi, w.beta
    p.adv_eps, p.grad_scale, p.reduction, p.flags = 1e-6, 1.0, w.reduction, 0
    return p


def _groups(w, dev):
    gr = g._Groups()
    gr.num_seqs = w.B
    gr.samples_per_prompt = w.samples_per_prompt
    gr.group_boundaries = None if w.samples_per_prompt else dev["bounds"].data_ptr()
    gr.num_groups = 0 if w.samples_per_prompt else len(dev["bounds"]) - 1
    return gr


def _static_call(case, dev):
    """One call of the no-allocation entry point through the C ABI."""
    w = case["w"]
    grad = torch.empty_like(dev["X"])
    out3 = torch.empty(3, dtype=torch.float32, device="cuda")
    gr, p = _groups(w, dev), _params(w)
    dt = {"f32": 0, "bf16": 1, "f16": 2}[case["dtype"]]
    rc = g.lib().grpo_loss_fwd_bwd_static(
        dev["X"].data_ptr(), dev["Y"].data_ptr(), dt, w.B, w.T, w.V, dev["acts"].data_ptr(),
        dev["old"].data_ptr(), dev["mask"].data_ptr(), dev["R"].data_ptr(), ctypes.byref(gr),
        ctypes.byref(p), grad.data_ptr(), out3.data_ptr(), None, None, None,
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0, g.grpo_status_string(rc)
    return out3, grad


def _workspace_call(case, dev):
    """The same loss through the workspace entry point."""
    w = case["w"]
    kw = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction)
    if w.samples_per_prompt:
        kw["samples_per_prompt"] = w.samples_per_prompt
    else:
        kw["group_boundaries"] = dev["bounds"]
    res = g.grpo_loss_fwd_bwd(dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"], dev["R"],
                              **kw)
    torch.cuda.synchronize()
    return res["out3"], res["grad"]


CASES = [
    (synth.WORKLOADS["tiny"], "f32"),
    (synth.Workload("csr", B=13, T=6, V=1531, seed=102, sigma=2.0, samples_per_prompt=0,
                    csr_size_range=(2, 5), reward="normal", len_range=(1, 6), holes=2,
                    reduction=1), "bf16"),
]


def test_static_scratch_matches_workspace_entry_point_twice():
    for w, dtype in CASES * 2:  # two rounds: each call follows another on the shared scratch
        case = make_case(w, dtype)
        dev = to_device(case)
        want3, want_g = _workspace_call(case, dev)
        for _ in range(2):
            got3, got_g = _static_call(case, dev)
            assert torch.equal(got3, want3), (w.name, got3, want3)
            assert torch.equal(got_g, want_g), w.name


def test_static_scratch_matches_the_oracle():
    w, dtype = CASES[0]
    case = make_case(w, dtype)
    exp = expect(case)
    got3, got_g = _static_call(case, to_device(case))
    out = got3.cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"static {k}")
    assert_grad_rows(torch_storage(got_g), exp["grad"], dtype, what="static grad")


def _wrapper_args(case, dev):
    w = case["w"]
    kw = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction)
    if w.samples_per_prompt:
        kw["samples_per_prompt"] = w.samples_per_prompt
    else:
        kw["group_boundaries"] = dev["bounds"]
    return kw


def test_static_python_wrapper_matches_and_validates():
    w, dtype = CASES[1]
    case = make_case(w, dtype)
    dev = to_device(case)
    want3, want_g = _workspace_call(case, dev)
    out3 = torch.empty(3, dtype=torch.float32, device="cuda")
    grad = torch.empty_like(dev["X"])
    args = (dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"], dev["R"])
    rc = g.grpo_loss_fwd_bwd_static(*args, grad=grad, out3=out3, **_wrapper_args(case, dev))
    torch.cuda.synchronize()
    assert rc == 0, g.grpo_status_string(rc)
    assert torch.equal(out3, want3) and torch.equal(grad, want_g)
    kw = _wrapper_args(case, dev)
    bad = [
        # int32 action ids would be read as int64 by the kernels
        ((dev["X"], dev["Y"], dev["acts"].int(), dev["old"], dev["mask"], dev["R"]),
         dict(grad=grad, out3=out3)),
        # host tensors
        ((dev["X"], dev["Y"], dev["acts"].cpu(), dev["old"], dev["mask"], dev["R"]),
         dict(grad=grad, out3=out3)),
        # a non-contiguous view
        ((dev["X"], dev["Y"], dev["acts"].t().contiguous().t(), dev["old"], dev["mask"],
          dev["R"]), dict(grad=grad, out3=out3)),
        # outputs of the wrong dtype or shape, or missing
        (args, dict(grad=grad.float() if dtype != "f32" else grad.half(), out3=out3)),
        (args, dict(grad=grad, out3=out3[:2])),
        (args, dict(grad=grad, out3=None)),
    ]
    for a, o in bad:
        with pytest.raises(ValueError):
            g.grpo_loss_fwd_bwd_static(*a, **o, **kw)
    # CSR boundaries given as a list would need an allocation
    kw_list = dict(kw, group_boundaries=case["bounds"].tolist(), samples_per_prompt=0)
    with pytest.raises(ValueError):
        g.grpo_loss_fwd_bwd_static(*args, grad=grad, out3=out3, **kw_list)


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    w = synth.WORKLOADS["tiny"]
    gr, p = g._Groups(), _params(w)
    gr.num_seqs, gr.samples_per_prompt = 8192, 8
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = g.lib().grpo_loss_fwd_bwd_static(fake, fake, 0, 8192, 64, 16, fake, fake, fake, fake,
                                          ctypes.byref(gr), ctypes.byref(p), fake, fake, None,
                                          None, None, None)
    assert rc == 7  # GRPO_ERR_WORKSPACE


def test_static_scratch_limit_counts_the_whole_batch_in_a_shard_call():
    # a shard of 8 sequences of a 8192-sequence batch: the scratch is laid out
    # for the batch, so the call is rejected like the unsharded one
    w = synth.WORKLOADS["tiny"]
    gr, p = g._Groups(), _params(w)
    gr.num_seqs, gr.samples_per_prompt = 8192, 8
    fake = 1 << 20  # never dereferenced: the size check comes first
    sh = g._Shard(0, fake, fake)
    p.shard = ctypes.pointer(sh)
    rc = g.lib().grpo_loss_fwd_bwd_static(fake, fake, 0, 8, 64, 16, fake, fake, fake, fake,
                                          ctypes.byref(gr), ctypes.byref(p), fake, None, None,
                                          None, None, None)
    assert rc == 7  # GRPO_ERR_WORKSPACE
