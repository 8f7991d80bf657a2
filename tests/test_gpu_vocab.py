"""Vocabulary parallelism (tensor parallelism over V), emulated on one GPU:
the vocabulary split into slices at chunk boundaries, every "rank" computing
its partial normalisers and gradient slice from its own contiguous copy of
the slice.  Every split gives bit-identical losses, log-sum-exps, per-sequence
totals and gradients (RL-Kernel "Tensor and Data Parallel": cross-TP bitwise
equality), and the result matches the oracle within the usual tolerances."""
import numpy as np
import pytest
import torch

import grad_row_online_gb300 as g
import oracle
import synth
from workload_inputs import assert_grad_rows, assert_scalar, make_case, to_device, torch_storage

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    import __graft_entry__
    if not os.path.exists(g.library_path()):
        __graft_entry__.build()


C = 4096
# three chunks, the last one partial; spikes; ragged masks; groups of 4
WL = synth.Workload("vocab_tp", B=8, T=6, V=2 * C + 777, seed=131, sigma=2.5, spike_p=0.01,
                    spike_mag=8.0, ref_sigma=0.2, samples_per_prompt=4, reward_p=0.5,
                    len_range=(1, 6), eps_lo=0.2, eps_hi=0.28, beta=0.1, old_sigma=0.2)
SPLITS = {"1": [WL.V], "2": [C, WL.V - C], "3": [C, C, WL.V - 2 * C], "2b": [2 * C, WL.V - 2 * C]}
VARIANTS = {"default": {}, "gspo": dict(ratio_level="sequence", reduction="sequence_mean"),
            "k2-cispo": dict(kl="k2", surrogate="cispo"),
            "seqmean-dual": dict(reduction="sequence_mean", dual_clip_c=1.5)}
_RED = {"token_mean": 0, "sequence_mean": 1}


def _tp_run(dev, widths, v):
    w = WL
    bounds = np.concatenate([[0], np.cumsum(widths)])
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        parts.append(g.grpo_vocab_partials(dev["X"][:, :, a:b].contiguous(),
                                           dev["Y"][:, :, a:b].contiguous(), dev["acts"],
                                           dev["mask"], int(a)))
    part_p = torch.cat([p["part_p"] for p in parts])  # rank order = chunk order
    part_r = torch.cat([p["part_r"] for p in parts])
    act = torch.stack([p["action_logits"] for p in parts]).sum(0)  # one rank holds each
    res = g.grpo_vocab_loss(part_p, part_r, act, w.V, dev["acts"], dev["old"], dev["mask"],
                            dev["R"], samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                            clip_eps_hi=w.eps_hi, beta=w.beta, want_per_seq=True,
                            want_logps=True, want_clip_counts=True, **v)
    grads = [g.grpo_vocab_grad(dev["X"][:, :, a:b].contiguous(), dev["acts"], dev["mask"], int(a),
                               res["lse_w"]) for a, b in zip(bounds[:-1], bounds[1:])]
    torch.cuda.synchronize()
    res["grad"] = torch.cat(grads, dim=2)
    return res


@pytest.mark.parametrize("name", list(VARIANTS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_vocab_parallel_is_bitwise_across_splits_and_matches_the_oracle(dtype, name):
    v = VARIANTS[name]
    w = WL
    case = make_case(w, dtype)
    dev = to_device(case)
    ref = _tp_run(dev, SPLITS["1"], v)
    for split, widths in SPLITS.items():
        got = _tp_run(dev, widths, v)
        for k in ("out3", "lse_w", "per_seq", "logps", "grad", "clip_counts"):
            assert torch.equal(got[k], ref[k]), (split, k)
    kw = {k: v[k] for k in ("kl", "surrogate", "dual_clip_c", "ratio_level") if k in v}
    kw["reduction"] = _RED[v.get("reduction", "token_mean")]
    exp = oracle.fused(case["X"], case["Y"], dtype, case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, **kw)
    out = ref["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    ps = ref["per_seq"].cpu().numpy().astype(np.float64)
    assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-6)
    m = case["mask"].astype(bool)
    lp = ref["logps"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lp[m] - exp["logp"][m]) <= 1e-6 * (1 + np.abs(exp["logp"][m])))
    r = exp["ratio"]
    near = np.zeros(r.shape, bool)
    for b in (0.8, 1.28, 1.5):
        near |= np.abs(r - b) <= 1e-6 * b
    keep = ~near
    assert_grad_rows(torch_storage(ref["grad"])[keep], exp["grad"][keep], dtype,
                     what=f"{name} grad")
    assert list(ref["clip_counts"].cpu().numpy()) == list(exp["clip_counts"]) or near.any()


def test_vocab_parallel_agrees_with_the_fused_path():
    w = WL
    case = make_case(w, "bf16")
    dev = to_device(case)
    tp = _tp_run(dev, SPLITS["3"], {})
    fused = g.grpo_loss_fwd_bwd(dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"],
                                dev["R"], samples_per_prompt=w.samples_per_prompt,
                                clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta)
    torch.cuda.synchronize()
    a = tp["out3"].cpu().numpy().astype(np.float64)
    b = fused["out3"].cpu().numpy().astype(np.float64)
    assert np.allclose(a, b, rtol=2e-5, atol=1e-9)
    diff = (tp["grad"].float() - fused["grad"].float()).abs()
    assert diff.max().item() <= 2 * 2 ** -8 * fused["grad"].float().abs().max().item()


@pytest.mark.parametrize("V,dtype,widths", [(1000, "f32", [1000]), (2 * C, "bf16", [C, C]),
                                            (C + 5, "f16", [C, 5])])
def test_vocab_parallel_edge_vocabularies(V, dtype, widths):
    # a single partial chunk; whole chunks only; a 5-entry last slice; f16
    w = WL.with_(V=V, B=8, T=4, len_range=(0, 4))
    case = make_case(w, dtype)
    dev = to_device(case)
    got = _run_with(w, dev, widths)
    one = _run_with(w, dev, [V])
    for k in ("out3", "lse_w", "grad"):
        assert torch.equal(got[k], one[k]), k
    exp = oracle.fused(case["X"], case["Y"], dtype, case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta)
    out = got["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)
    r = exp["ratio"]
    near = (np.abs(r - 0.8) <= 1e-6) | (np.abs(r - 1.28) <= 1.3e-6)
    assert_grad_rows(torch_storage(got["grad"])[~near], exp["grad"][~near], dtype)


def _run_with(w, dev, widths):
    bounds = np.concatenate([[0], np.cumsum(widths)])
    parts = [g.grpo_vocab_partials(dev["X"][:, :, a:b].contiguous(),
                                   dev["Y"][:, :, a:b].contiguous(), dev["acts"], dev["mask"],
                                   int(a)) for a, b in zip(bounds[:-1], bounds[1:])]
    res = g.grpo_vocab_loss(torch.cat([p["part_p"] for p in parts]),
                            torch.cat([p["part_r"] for p in parts]),
                            torch.stack([p["action_logits"] for p in parts]).sum(0), w.V,
                            dev["acts"], dev["old"], dev["mask"], dev["R"],
                            samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                            clip_eps_hi=w.eps_hi, beta=w.beta)
    res["grad"] = torch.cat([g.grpo_vocab_grad(dev["X"][:, :, a:b].contiguous(), dev["acts"],
                                               dev["mask"], int(a), res["lse_w"])
                             for a, b in zip(bounds[:-1], bounds[1:])], dim=2)
    torch.cuda.synchronize()
    return res


def test_vocab_parallel_masked_rows_and_bad_actions():
    w = WL.with_(V=3000, B=8, T=4, len_range=(0, 4))
    case = make_case(w, "bf16")
    dev = to_device(case)
    # masked rows are never read: poison their logits
    m = dev["mask"].bool()
    dev["X"][~m] = float("nan")
    dev["Y"][~m] = float("inf")
    a = _run_with(w, dev, [3000])
    assert torch.isfinite(a["out3"]).all()
    assert (a["grad"][~m] == 0).all()
    # an active token whose action id no slice holds: device status, NaN loss
    acts = dev["acts"].clone()
    row = int(m.view(-1).nonzero()[0])
    acts.view(-1)[row] = w.V + 7
    dev2 = dict(dev, acts=acts)
    b = _run_with(w, dev2, [3000])
    assert torch.isnan(b["out3"]).all()
    assert g.grpo_read_device_status(b["workspace"]) & 16
