"""The logps path in one launch: when every sequence's CTA fits on the GPU at
once, grpo_loss_from_logps runs a single cooperative kernel whose CTAs scan
their own mask rows, form their own advantages and meet at a grid barrier
before reading the batch counts N and S.  Against the separate advantage /
count pass (GRPO_FLAG_SEPARATE_PREP) it must give the same bits for every
output -- loss outputs, gradient, per-sequence totals, advantages, clip
counts -- on the staged, register and scalar row paths, uniform and CSR
groups, every reduction and the loss variants.  Batches too large for one
wave take the separate pass by themselves; device-detected errors are still
reported; a barrier wait that runs out is reported and leaves the context
usable."""
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


BASE = synth.WORKLOADS["logps"].with_(name="onelaunch", B=48, T=64, len_range=(0, 64),
                                      samples_per_prompt=8, old_sigma=0.3, ref_logp_sigma=0.1)
CSR = BASE.with_(name="onelaunch_csr", samples_per_prompt=0, csr_size_range=(1, 9),
                 reward="normal")


def _tensors(w):
    lp, old, ref = w.logps_inputs()
    host = dict(lp=lp, old=old, ref=ref, mask=w.completion_mask(), R=w.rewards())
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in host.items()}
    t["bounds"] = (torch.from_numpy(w.group_boundaries()).cuda()
                   if not w.samples_per_prompt else None)
    return t


def _call(w, t, flags=0, **kw):
    args = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, want_per_seq=True,
                want_adv=True, want_clip_counts=True, extra_flags=flags)
    if w.samples_per_prompt:
        args["samples_per_prompt"] = w.samples_per_prompt
    else:
        args["group_boundaries"] = t["bounds"]
    args.update(kw)
    res = g.grpo_loss_from_logps(t["lp"], t["old"], t["ref"], t["mask"], t["R"], **args)
    torch.cuda.synchronize()
    return res


OUTS = ("out3", "grad", "per_seq", "adv", "clip_counts")
OPTIONS = {
    "token-mean": dict(),
    "sequence-mean": dict(reduction="sequence_mean"),
    "fixed-k2-dual": dict(reduction="fixed_constant", norm_constant=50.0, kl="k2",
                          dual_clip_c=1.4),
    "cispo-k1": dict(surrogate="cispo", kl="k1"),
    "cispo": dict(surrogate="cispo"),
    "dual": dict(dual_clip_c=1.4),
    "k1": dict(kl="k1"),
    "k2-sequence-mean": dict(kl="k2", reduction="sequence_mean"),
    "gspo": dict(reduction="sequence_mean", ratio_level="sequence"),
}


@pytest.mark.parametrize("opt", list(OPTIONS))
@pytest.mark.parametrize("T", [64, 100, 37])  # staged, register and scalar row paths
@pytest.mark.parametrize("w", [BASE, CSR], ids=["uniform", "csr"])
def test_one_launch_equals_the_separate_pass(w, T, opt):
    w = w.with_(T=T, len_range=(0, T))
    t = _tensors(w)
    one = _call(w, t, **OPTIONS[opt])
    two = _call(w, t, flags=g.GRPO_FLAG_SEPARATE_PREP, **OPTIONS[opt])
    assert g.grpo_read_device_status(one["workspace"]) == 0
    for k in OUTS:
        assert torch.equal(one[k], two[k]), k


def test_one_launch_parity_with_the_oracle():
    w = CSR.with_(reduction=1)
    t = _tensors(w)
    res = _call(w, t, reduction="sequence_mean")
    lp, old, ref = w.logps_inputs()
    A = oracle.group_advantages(w.rewards(), w.group_boundaries())
    assert np.array_equal(res["adv"].cpu().numpy(), A.astype(np.float32))
    exp = oracle.loss_from_logps(lp, ref, old, w.completion_mask(), A, w.eps_lo, w.eps_hi, w.beta,
                                 reduction=1)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)


def test_a_batch_larger_than_one_wave_takes_the_separate_pass():
    # 1,304 sequences: more CTAs than GB300 holds at once (8 per SM x 152)
    w = BASE.with_(name="onelaunch_big", B=1304, T=32, len_range=(0, 32))
    t = _tensors(w)
    one = _call(w, t)
    two = _call(w, t, flags=g.GRPO_FLAG_SEPARATE_PREP)
    for k in OUTS:
        assert torch.equal(one[k], two[k]), k
    lp, old, ref = w.logps_inputs()
    A = oracle.group_advantages(w.rewards(), w.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, w.completion_mask(), A, w.eps_lo, w.eps_hi, w.beta)
    out = one["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)


def test_device_errors_in_one_launch():
    w = BASE
    t = _tensors(w)
    R = t["R"].clone()
    R[13] = float("nan")
    res = _call(w, dict(t, R=R))
    assert g.grpo_read_device_status(res["workspace"]) == g.GRPO_ERR_NONFINITE_REWARD
    assert torch.isnan(res["out3"]).all()
    # a CSR whose groups do not end at B (checked over the grid, group by group)
    wc = CSR
    tc = _tensors(wc)
    bad = tc["bounds"].clone()
    bad[-1] = wc.B - 1
    res = _call(wc, dict(tc, bounds=bad))
    assert g.grpo_read_device_status(res["workspace"]) == g.GRPO_ERR_CSR
    assert torch.isnan(res["out3"]).all()
    res = _call(wc, tc, workspace=res["workspace"])
    assert g.grpo_read_device_status(res["workspace"]) == 0


def test_a_stalled_barrier_times_out_and_the_context_survives():
    w = BASE
    t = _tensors(w)
    t0 = time.time()
    bad = _call(w, t, flags=g.GRPO_FLAG_TEST_STALLED_BARRIER)
    status = g.grpo_read_device_status(bad["workspace"])
    assert status == g.GRPO_ERR_TIMEOUT
    assert torch.isnan(bad["out3"]).all()
    assert time.time() - t0 < 30.0
    good = _call(w, t, workspace=bad["workspace"])
    assert g.grpo_read_device_status(good["workspace"]) == 0
    ref = _call(w, t, flags=g.GRPO_FLAG_SEPARATE_PREP)
    for k in OUTS:
        assert torch.equal(good[k], ref[k]), k


@pytest.mark.parametrize("flags", [0, g.GRPO_FLAG_SEPARATE_PREP], ids=["one-launch", "two-launch"])
def test_clean_workspace_calls_give_the_same_bits(flags):
    # every call leaves the header clean, so a loop of calls on one workspace
    # may skip its reset (GRPO_FLAG_WORKSPACE_CLEAN): same bits as a fresh
    # workspace, for every option, on both forms, after errors and timeouts
    ws = torch.empty(g.grpo_workspace_size(CSR.B, 100, 0), dtype=torch.uint8, device="cuda")
    _call(BASE, _tensors(BASE), flags=flags, workspace=ws)  # leaves it clean
    for w in (BASE, CSR):
        for T in (64, 100):
            wt = w.with_(T=T, len_range=(0, T))
            t = _tensors(wt)
            for opt in OPTIONS.values():
                got = _call(wt, t, flags=flags, workspace=ws, workspace_clean=True, **opt)
                assert g.grpo_read_device_status(ws) == 0
                want = _call(wt, t, flags=flags, **opt)
                for k in OUTS:
                    assert torch.equal(got[k], want[k]), k
    # a device-detected error is reported by its own call, and the next clean
    # call is clean
    t = _tensors(BASE)
    R = t["R"].clone()
    R[5] = float("inf")
    bad = _call(BASE, dict(t, R=R), flags=flags, workspace=ws, workspace_clean=True)
    assert g.grpo_read_device_status(ws) == g.GRPO_ERR_NONFINITE_REWARD
    assert torch.isnan(bad["out3"]).all()
    good = _call(BASE, t, flags=flags, workspace=ws, workspace_clean=True)
    assert g.grpo_read_device_status(ws) == 0
    want = _call(BASE, t, flags=flags)
    for k in OUTS:
        assert torch.equal(good[k], want[k]), k
    if flags == 0:
        # a barrier wait that runs out still leaves the header clean
        bad = _call(BASE, t, flags=g.GRPO_FLAG_TEST_STALLED_BARRIER, workspace=ws,
                    workspace_clean=True)
        assert g.grpo_read_device_status(ws) == g.GRPO_ERR_TIMEOUT
        good = _call(BASE, t, workspace=ws, workspace_clean=True)
        assert g.grpo_read_device_status(ws) == 0
        for k in OUTS:
            assert torch.equal(good[k], want[k]), k


def test_clean_workspace_shard_calls():
    w = BASE
    t = _tensors(w)
    mask = w.completion_mask()
    counts = torch.tensor([int(mask.sum()), int((mask.sum(1) > 0).sum())], dtype=torch.int64,
                          device="cuda")
    ws = torch.zeros(g.grpo_workspace_size(w.B, w.T, 0), dtype=torch.uint8, device="cuda")
    outs = []
    for clean in (False, True, True):
        tot = g.totals_buffer(w.B)
        r = _call(w, t, shard=g.Shard(0, counts, tot), workspace=ws, workspace_clean=clean,
                  want_per_seq=False)
        outs.append((tot, r["grad"], r["clip_counts"]))
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert torch.equal(a, b)


def test_overlap_launch_gives_the_same_bits():
    # GRPO_FLAG_OVERLAP_LAUNCH: the one-launch kernel dispatched while the
    # previous kernel on the stream ends (nothing else runs on this GPU in the
    # test, so every CTA becomes resident); back-to-back calls on one
    # workspace give the cooperative launch's bits
    ws = torch.empty(g.grpo_workspace_size(CSR.B, 100, 0), dtype=torch.uint8, device="cuda")
    for w in (BASE, CSR):
        for T in (64, 100):
            wt = w.with_(T=T, len_range=(0, T))
            t = _tensors(wt)
            for opt in OPTIONS.values():
                want = _call(wt, t, **opt)
                args = dict(clip_eps=wt.eps_lo, clip_eps_hi=wt.eps_hi, beta=wt.beta,
                            want_per_seq=True, want_adv=True, want_clip_counts=True,
                            workspace=ws, overlap_launch=True, **opt)
                if wt.samples_per_prompt:
                    args["samples_per_prompt"] = wt.samples_per_prompt
                else:
                    args["group_boundaries"] = t["bounds"]
                outs = [g.grpo_loss_from_logps(t["lp"], t["old"], t["ref"], t["mask"], t["R"],
                                               workspace_clean=k > 0, **args) for k in range(3)]
                torch.cuda.synchronize()
                assert g.grpo_read_device_status(ws) == 0
                for got in outs:
                    for k in OUTS:
                        assert torch.equal(got[k], want[k]), k
