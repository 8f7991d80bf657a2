"""Parity of the loss variants -- KL estimators k1 / k2, the dual clip, CISPO,
the fixed-constant (Dr.GRPO) normaliser, GSPO's sequence-level ratio -- and
of the clip counters, CUDA
library against the oracle, on both boundaries (logits and per-token
log-probs), with ratios spread wide enough that every clip binds."""
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


VARIANTS = {
    "k1": dict(kl="k1"),
    "k2": dict(kl="k2"),
    "dual": dict(dual_clip_c=1.3),
    "cispo": dict(surrogate="cispo"),
    "fixed": dict(reduction="fixed_constant", norm_constant=50.0),
    "k2-dual-seqmean": dict(kl="k2", dual_clip_c=1.25, reduction="sequence_mean"),
    "cispo-k1-fixed": dict(surrogate="cispo", kl="k1", reduction="fixed_constant",
                           norm_constant=7.0),
    "gspo": dict(ratio_level="sequence", reduction="sequence_mean"),
    "gspo-k2-dual": dict(ratio_level="sequence", reduction="sequence_mean", kl="k2",
                         dual_clip_c=1.3),
    "default": dict(),
}
_RED = {"token_mean": 0, "sequence_mean": 1, "fixed_constant": 2}


def _oracle_kw(v: dict, w) -> dict:
    kw = {k: v[k] for k in ("kl", "surrogate", "dual_clip_c", "norm_constant", "ratio_level")
          if k in v}
    kw["reduction"] = _RED[v["reduction"]] if "reduction" in v else w.reduction
    return kw


def _band(exp, eps_lo, eps_hi, dual_c, band=1e-6):
    r = exp["ratio"]
    near = np.zeros(r.shape, bool)
    for b in (1.0 - float(np.float32(eps_lo)), 1.0 + float(np.float32(eps_hi)),
              float(np.float32(dual_c)) if dual_c else None):
        if b is not None:
            near |= np.abs(r - b) <= band * b
    return near


def _check_counts(got, exp, near):
    got = got.cpu().numpy()
    want = exp["clip_counts"]
    assert np.all(np.abs(got - want) <= near.sum()), (got, want, near.sum())


# ---------------------------------------------------------------------------
# the logits boundary
# ---------------------------------------------------------------------------
# ratios spread by old = logp + N(0, 0.4): both bounds and the dual clip bind
WIDE = synth.Workload("wide", B=12, T=10, V=3001, seed=111, sigma=2.0, ref_sigma=0.3,
                      samples_per_prompt=4, reward_p=0.5, len_range=(2, 10), eps_lo=0.2,
                      eps_hi=0.28, beta=0.3, old_sigma=0.4)
TINY_WIDE = synth.WORKLOADS["tiny"].with_(old_sigma=0.4, beta=0.3)


def _run_logits(case, dev, v):
    w = case["w"]
    args = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction,
                samples_per_prompt=w.samples_per_prompt, want_per_seq=True,
                want_clip_counts=True)
    args.update(v)
    res = g.grpo_loss_fwd_bwd(dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"], dev["R"],
                              **args)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("name", list(VARIANTS))
@pytest.mark.parametrize("which,dtype", [("tiny", "f32"), ("wide", "f32"), ("wide", "bf16")])
def test_logits_variants(name, which, dtype):
    v = VARIANTS[name]
    w = TINY_WIDE if which == "tiny" else WIDE
    case = make_case(w, dtype)
    exp = oracle.fused(case["X"], case["Y"], dtype, case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, **_oracle_kw(v, w))
    res = _run_logits(case, to_device(case), v)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    ps = res["per_seq"].cpu().numpy().astype(np.float64)
    assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-6)
    assert np.allclose(ps[1], exp["per_seq_kl"], rtol=1e-5, atol=1e-7)
    near = _band(exp, w.eps_lo, w.eps_hi, v.get("dual_clip_c"))
    _check_counts(res["clip_counts"], exp, near)
    # gradient rows of tokens at a clip kink may take either branch
    got = torch_storage(res["grad"])
    keep = ~near
    assert_grad_rows(got[keep], exp["grad"][keep], dtype, what=f"{name} grad")


@pytest.mark.parametrize("name", ["gspo", "default"])
def test_long_16bit_rows_claimed_token_major(name):
    # bf16 rows long enough for the tensor-memory slice: the row kernel and
    # GSPO's second sweep claim their rows token-major (slot t of every
    # sequence before slot t + 1), which must change no result
    v = VARIANTS[name]
    w = WIDE.with_(name="wide_long", V=90000, T=6, len_range=(1, 6))
    case = make_case(w, "bf16")
    exp = oracle.fused(case["X"], case["Y"], "bf16", case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, **_oracle_kw(v, w))
    res = _run_logits(case, to_device(case), v)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    near = _band(exp, w.eps_lo, w.eps_hi, v.get("dual_clip_c"))
    assert_grad_rows(torch_storage(res["grad"])[~near], exp["grad"][~near], "bf16",
                     what=f"{name} grad")


def test_wide_case_reaches_every_clip():
    case = make_case(WIDE, "f32")
    w = WIDE
    exp = oracle.fused(case["X"], case["Y"], "f32", case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, dual_clip_c=1.3)
    assert np.all(exp["clip_counts"] > 0), exp["clip_counts"]


# ---------------------------------------------------------------------------
# the per-token log-prob boundary
# ---------------------------------------------------------------------------
LOGPS_WIDE = synth.WORKLOADS["logps"].with_(name="logps_wide", B=16, T=64, len_range=(4, 64),
                                           old_sigma=0.4, ref_logp_sigma=0.3, beta=0.3,
                                           eps_hi=0.28)


def _logps_inputs(w, mask_seed=None):
    lp, old, ref = w.logps_inputs()
    mask = w.completion_mask()
    if mask_seed is not None:  # holes and leading masked tokens
        rng = np.random.default_rng(mask_seed)
        mask = (mask * (rng.random(mask.shape) < 0.8)).astype(np.uint8)
    return lp, old, ref, mask, w.rewards()


@pytest.mark.parametrize("name", list(VARIANTS))
@pytest.mark.parametrize("T", [64, 100, 37])  # staged, register and scalar paths
def test_logps_variants(name, T):
    v = VARIANTS[name]
    w = LOGPS_WIDE.with_(T=T, len_range=(4, T))
    lp, old, ref, mask, R = _logps_inputs(w, mask_seed=T)
    A = oracle.group_advantages(R, w.group_boundaries())
    for has_ref in (True, False):  # without a reference the KL term needs beta = 0
        beta = w.beta if has_ref else 0.0
        exp = oracle.loss_from_logps(lp, ref if has_ref else None, old, mask, A, w.eps_lo,
                                     w.eps_hi, beta, **_oracle_kw(v, w))
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        args = dict(samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                    clip_eps_hi=w.eps_hi, beta=beta, reduction=w.reduction,
                    want_per_seq=True, want_clip_counts=True)
        args.update(v)
        res = g.grpo_loss_from_logps(t(lp), t(old), t(ref) if has_ref else None, t(mask), t(R),
                                     **args)
        torch.cuda.synchronize()
        out = res["out3"].cpu().numpy().astype(np.float64)
        for i, k in enumerate(("loss", "policy_loss", "kl")):
            assert_scalar(out[i], exp[k], f"{name} ref={has_ref} {k}")
        ps = res["per_seq"].cpu().numpy().astype(np.float64)
        assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-5)
        near = _band(exp, w.eps_lo, w.eps_hi, v.get("dual_clip_c"))
        _check_counts(res["clip_counts"], exp, near)
        want = exp["w"].astype(np.float32)
        got = res["grad"].cpu().numpy()
        ok = np.abs(got.astype(np.float64) - want) <= np.spacing(np.abs(want)) + 1e-9
        assert np.all(ok | near), np.argwhere(~(ok | near))[:5]


def test_logps_default_counts_on_the_fast_path():
    # the default variant evaluates full 4-token vectors on the packed fast
    # path, which counts clipped tokens by the sign of A
    w = LOGPS_WIDE.with_(B=64, T=512, len_range=(512, 512), old_sigma=0.15, ref_logp_sigma=0.05,
                         beta=0.04)
    lp, old, ref, mask, R = _logps_inputs(w)
    A = oracle.group_advantages(R, w.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, mask, A, w.eps_lo, w.eps_hi, w.beta)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    res = g.grpo_loss_from_logps(t(lp), t(old), t(ref), t(mask), t(R),
                                 samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                 clip_eps_hi=w.eps_hi, beta=w.beta, want_clip_counts=True)
    torch.cuda.synchronize()
    near = _band(exp, w.eps_lo, w.eps_hi, None)
    assert exp["clip_counts"][0] > 0 and exp["clip_counts"][1] > 0
    _check_counts(res["clip_counts"], exp, near)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)


@pytest.mark.parametrize("name", list(VARIANTS))
def test_logps_variants_on_the_fast_path(name):
    # small log ratios: every fully active 4-token vector passes the fast
    # path's range check, so the variants' packed path carries the tokens
    v = VARIANTS[name]
    w = LOGPS_WIDE.with_(B=64, T=512, len_range=(384, 512), old_sigma=0.15,
                         ref_logp_sigma=0.05, beta=0.04)
    lp, old, ref, mask, R = _logps_inputs(w)
    A = oracle.group_advantages(R, w.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, mask, A, w.eps_lo, w.eps_hi, w.beta,
                                 **_oracle_kw(v, w))
    if v.get("dual_clip_c") and not v.get("ratio_level"):  # the dual clip binds on
        assert exp["clip_counts"][2] > 0                     # the fast path too
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = dict(samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi,
                beta=w.beta, reduction=w.reduction, want_per_seq=True, want_clip_counts=True)
    args.update(v)
    res = g.grpo_loss_from_logps(t(lp), t(old), t(ref), t(mask), t(R), **args)
    torch.cuda.synchronize()
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    near = _band(exp, w.eps_lo, w.eps_hi, v.get("dual_clip_c"))
    _check_counts(res["clip_counts"], exp, near)
    want = exp["w"].astype(np.float32)
    got = res["grad"].cpu().numpy()
    ok = np.abs(got.astype(np.float64) - want) <= np.spacing(np.abs(want)) + 1e-9
    assert np.all(ok | near), np.argwhere(~(ok | near))[:5]


@pytest.mark.parametrize("name", ["k1", "k2", "dual", "cispo", "gspo"])
def test_logps_variants_with_every_vector_deferred(name):
    # log ratios ~N(0, 2): nearly every vector fails the fast path's range
    # check, so the variants with a packed path of their own (the clipped
    # surrogate with k1, k2 or the dual clip, CISPO with k3, GSPO with k3) leave each thread's
    # whole share of the row to the general path after the token loop
    v = VARIANTS[name]
    w = LOGPS_WIDE.with_(B=8, T=4096, len_range=(3000, 4096), old_sigma=2.0,
                         ref_logp_sigma=1.0)
    lp, old, ref, mask, R = _logps_inputs(w)
    A = oracle.group_advantages(R, w.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, mask, A, w.eps_lo, w.eps_hi, w.beta,
                                 **_oracle_kw(v, w))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for flags in (0, g.GRPO_FLAG_SEPARATE_PREP):
        args = dict(samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                    clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction,
                    want_per_seq=True, want_clip_counts=True, extra_flags=flags)
        args.update(v)
        res = g.grpo_loss_from_logps(t(lp), t(old), t(ref), t(mask), t(R), **args)
        torch.cuda.synchronize()
        out = res["out3"].cpu().numpy().astype(np.float64)
        for i, k in enumerate(("loss", "policy_loss", "kl")):
            assert_scalar(out[i], exp[k], f"{name} {k}")
        near = _band(exp, w.eps_lo, w.eps_hi, v.get("dual_clip_c"))
        _check_counts(res["clip_counts"], exp, near)
        want = exp["w"].astype(np.float32)
        got = res["grad"].cpu().numpy()
        ok = np.abs(got.astype(np.float64) - want) <= np.spacing(np.abs(want)) + 1e-9
        assert np.all(ok | near), np.argwhere(~(ok | near))[:5]


def test_variant_parameters_are_checked_on_the_host():
    x = torch.zeros((2, 1, 4), device="cuda")
    a = torch.zeros((2, 1), dtype=torch.int64, device="cuda")
    o = torch.zeros((2, 1), device="cuda")
    m = torch.ones((2, 1), dtype=torch.uint8, device="cuda")
    r = torch.tensor([1.0, 0.0], device="cuda")
    for bad in (dict(dual_clip_c=0.5), dict(surrogate="cispo", dual_clip_c=2.0),
                dict(reduction="fixed_constant")):
        with pytest.raises(g.GrpoError):
            g.grpo_loss_fwd_bwd(x, x, a, o, m, r, samples_per_prompt=2, **bad)


def test_gspo_with_empty_sequences_on_both_boundaries():
    # sequences with no active token: rho_i undefined, weight 0, excluded from
    # the sequence mean
    w = WIDE.with_(len_range=(0, 10), holes=3, reduction=1)
    case = make_case(w, "f32")
    assert (case["mask"].sum(1) == 0).sum() >= 3
    v = dict(ratio_level="sequence", reduction="sequence_mean")
    exp = oracle.fused(case["X"], case["Y"], "f32", case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, reduction=1,
                       ratio_level="sequence")
    res = _run_logits(case, to_device(case), v)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)
    near = _band(exp, w.eps_lo, w.eps_hi, None)
    assert_grad_rows(torch_storage(res["grad"])[~near], exp["grad"][~near], "f32")
    # the same tokens through the logps boundary
    lp = exp["logp"].astype(np.float32)
    rf = exp["ref_logp"].astype(np.float32)
    e2 = oracle.loss_from_logps(lp, rf, case["old"], case["mask"], exp["A"], w.eps_lo, w.eps_hi,
                                w.beta, reduction=1, ratio_level="sequence")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    r2 = g.grpo_loss_from_logps(t(lp), t(case["old"]), t(rf), t(case["mask"]), t(case["R"]),
                                samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                clip_eps_hi=w.eps_hi, beta=w.beta, **v)
    torch.cuda.synchronize()
    out = r2["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], e2[k], k)


@pytest.mark.parametrize("name", ["k2", "cispo", "gspo", "dual"])
def test_variants_with_f16_logits(name):
    v = VARIANTS[name]
    w = TINY_WIDE
    case = make_case(w, "f16")
    exp = oracle.fused(case["X"], case["Y"], "f16", case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, **_oracle_kw(v, w))
    res = _run_logits(case, to_device(case), v)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{name} {k}")
    near = _band(exp, w.eps_lo, w.eps_hi, v.get("dual_clip_c"))
    assert_grad_rows(torch_storage(res["grad"])[~near], exp["grad"][~near], "f16")
