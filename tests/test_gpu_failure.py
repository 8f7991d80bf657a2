"""Failure detection on the GPU without a fault: the test hook
GRPO_FLAG_TEST_STALLED_COPY makes one asynchronous copy of the logps kernel
under-deliver, so its bounded wait runs out.  The call must come back with
GRPO_ERR_TIMEOUT in the workspace status word and NaN loss outputs, and the
same context must then compute a correct loss."""
import time

import numpy as np
import pytest
import torch

import grad_row_online_gb300 as g
import oracle
import synth
from workload_inputs import assert_scalar

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    import __graft_entry__
    if not os.path.exists(g.library_path()):
        __graft_entry__.build()


W = synth.WORKLOADS["logps"].with_(name="logps_stall", B=16, T=2048, len_range=(2048, 2048))


def _inputs():
    lp, old, ref = W.logps_inputs()
    host = dict(lp=lp, old=old, ref=ref, mask=W.completion_mask(), R=W.rewards())
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in host.items()}


def _call(t, ws, **kw):
    return g.grpo_loss_from_logps(t["lp"], t["old"], t["ref"], t["mask"], t["R"],
                                  samples_per_prompt=W.samples_per_prompt, clip_eps=W.eps_lo,
                                  clip_eps_hi=W.eps_hi, beta=W.beta, workspace=ws, **kw)


def test_a_stalled_copy_times_out_and_the_context_survives():
    t = _inputs()
    ws = torch.empty(g.grpo_workspace_size(W.B, W.T), dtype=torch.uint8, device="cuda")
    t0 = time.time()
    bad = _call(t, ws, extra_flags=g.GRPO_FLAG_TEST_STALLED_COPY)
    status = g.grpo_read_device_status(ws)  # synchronises
    took = time.time() - t0
    assert status & g.GRPO_ERR_TIMEOUT
    assert torch.isnan(bad["out3"]).all()
    assert took < 30.0
    # the same context and workspace, without the hook: a correct loss
    good = _call(t, ws)
    assert g.grpo_read_device_status(ws) == 0
    lp, old, ref = W.logps_inputs()
    A = oracle.group_advantages(W.rewards(), W.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, W.completion_mask(), A, W.eps_lo, W.eps_hi,
                                 W.beta)
    out = good["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)
