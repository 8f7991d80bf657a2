"""Parity of the CUDA library (through its C ABI) with the double-precision
oracle on seeded inputs, at sizes the oracle finishes in seconds: several
512-thread tiles per row, ragged tails, odd vocabularies, every dtype, both
reductions, CSR groups, and the edge cases of the method."""
import numpy as np
import pytest
import torch

import grad_row_online_gb300 as g
import oracle
import synth
from workload_inputs import (assert_grad_rows, assert_scalar, clip_band_rows, expect, make_case,
                             to_device, torch_storage)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    import __graft_entry__
    if not os.path.exists(g.library_path()):
        __graft_entry__.build()


TINY = synth.WORKLOADS["tiny"]
# multi-tile rows with a ragged vector tail, 3 groups of 4, some empty rows
MEDIUM = synth.Workload("medium", B=12, T=10, V=5003, seed=101, sigma=2.0, ref_sigma=0.1,
                        samples_per_prompt=4, reward_p=0.5, len_range=(0, 10),
                        eps_lo=0.2, eps_hi=0.28, beta=0.04)
# CSR groups, sequence mean, continuous rewards, fully masked rows
CSR = synth.Workload("csr", B=13, T=6, V=1531, seed=102, sigma=2.0, samples_per_prompt=0,
                     csr_size_range=(2, 5), reward="normal", len_range=(1, 6), holes=2,
                     reduction=1)


def run(case, dev, **kw):
    w = case["w"]
    args = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta,
                reduction=w.reduction, want_per_seq=True, want_logps=True, want_adv=True)
    if w.samples_per_prompt:
        args["samples_per_prompt"] = w.samples_per_prompt
    else:
        args["group_boundaries"] = dev["bounds"]
    args.update(kw)
    res = g.grpo_loss_fwd_bwd(dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"], dev["R"],
                              **args)
    torch.cuda.synchronize()
    return res


def check(case, res, exp, what=""):
    w = case["w"]
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{what} {k}")
    ps = res["per_seq"].cpu().numpy().astype(np.float64)
    assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-6)
    assert np.allclose(ps[1], exp["per_seq_kl"], rtol=1e-5, atol=1e-7)
    assert np.array_equal(ps[2], exp["per_seq_active"])
    assert np.allclose(res["adv"].cpu().numpy(), exp["A"].astype(np.float32), rtol=1e-6, atol=1e-7)
    m = case["mask"].astype(bool)
    lp = res["logps"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lp[m] - exp["logp"][m]) <= 4e-6 + 1e-6 * np.abs(exp["logp"][m]))
    assert np.all(lp[~m] == 0)
    if res["grad"] is not None:
        got = torch_storage(res["grad"])
        assert_grad_rows(got, exp["grad"], case["dtype"], what=f"{what} grad")


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_tiny_workload(dtype):
    case = make_case(TINY, dtype)
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"tiny/{dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_medium_multi_tile_ragged(dtype):
    case = make_case(MEDIUM, dtype)
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"medium/{dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_csr_groups_sequence_mean(dtype):
    case = make_case(CSR, dtype)
    assert (case["mask"].sum(1) == 0).sum() == 2
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"csr/{dtype}")


@pytest.mark.parametrize("V", [1, 2, 4, 7, 8, 9, 16, 4099, 4100])
def test_small_and_odd_vocabularies(V):
    w = TINY.with_(name=f"v{V}", V=V, seed=200 + V)
    case = make_case(w)
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"V={V}")


# long rows: many vectors per thread, a ragged vector tail, and an unaligned
# long row
@pytest.mark.parametrize("dtype,V", [("f32", 40000), ("bf16", 90000), ("f32", 100000),
                                     ("f32", 200000), ("bf16", 300000), ("f32", 270001)])
def test_long_rows(dtype, V):
    w = TINY.with_(name=f"long{V}", B=4, T=3, V=V, seed=300 + V % 97, sigma=2.0,
                   samples_per_prompt=2, len_range=(1, 3))
    case = make_case(w, dtype)
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"{dtype} V={V}")


# The row kernel keeps the head of a long policy row on chip between its two
# sweeps: 2,816 16-byte vectors in shared memory, then 16 per thread (4,096)
# in tensor memory, when the row has at least 7,680 vectors; the rest is read
# again.  Actions at the edges of each slice, on rows just above and below the
# length threshold, aligned and not.
@pytest.mark.parametrize("dtype,V", [("bf16", 90000), ("f32", 40000), ("bf16", 61440),
                                     ("bf16", 61439), ("f32", 30721), ("f16", 151936)])
def test_actions_at_kept_slice_edges(dtype, V):
    w = TINY.with_(name=f"edges{V}", B=4, T=3, V=V, seed=400 + V % 89, sigma=2.0,
                   samples_per_prompt=2, mask="full")
    case = make_case(w, dtype)
    per = 4 if dtype == "f32" else 8  # elements per vector
    e1, e2 = 2816 * per, 6912 * per
    acts = np.array([0, e1 - 1, e1, e1 + 1, e2 - 1, e2, e2 + 1, V - 1, e1 + per, e2 - per,
                     (e1 + e2) // 2, V // 2], dtype=np.int64)
    case["acts"] = np.minimum(acts, V - 1).reshape(w.B, w.T)
    _, lp = oracle.log_softmax_rows(case["X"].reshape(-1, V), dtype, case["acts"].reshape(-1))
    case["old"] = (lp.reshape(w.B, w.T) + w.old_sigma * w.old_noise()).astype(np.float32)
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"{dtype} V={V} kept-slice edges")


# a full mask: with equal lengths the advantages of a group cancel in the
# policy loss, which is then a small residual of the ratios
@pytest.mark.parametrize("dtype,V", [("f32", 5008), ("bf16", 5008), ("bf16", 90000)])
def test_full_mask_cancellation(dtype, V):
    w = MEDIUM.with_(name="full", V=V, mask="full", B=8 if V > 9000 else 12, T=4 if V > 9000 else 10)
    case = make_case(w, dtype)
    exp = expect(case)
    check(case, run(case, to_device(case)), exp, f"full mask {dtype} V={V}")


def test_a_gradient_step_lowers_the_loss():
    # the gradient the library writes is the derivative of the loss it reports:
    # a small step s of the policy logits against it changes the loss by
    # grad . s to first order (the second-order term is ~1e-5 of it here)
    case = make_case(MEDIUM, "f32")
    dev = to_device(case)
    res = run(case, dev)
    loss0 = float(res["out3"][0])
    grad = res["grad"].clone()
    eta = 1e-5 / float((grad.double() ** 2).sum())  # a predicted decrease of ~1e-5
    x1 = dev["X"] - eta * grad
    step = (x1.double() - dev["X"].double())        # the step as rounded to fp32
    predicted = float((grad.double() * step).sum())
    res1 = run(case, dict(dev, X=x1))
    change = float(res1["out3"][0]) - loss0
    assert predicted < -5e-6
    assert abs(change - predicted) <= 0.02 * abs(predicted), (change, predicted)


def test_token_mean_and_options():
    case = make_case(MEDIUM.with_(reduction=0), "f32")
    dev = to_device(case)
    for kw in (dict(eps_add=True), dict(grad_scale=0.37), dict(beta=0.0), dict(beta=0.5)):
        exp = expect(case, eps_add=kw.get("eps_add", False), grad_scale=kw.get("grad_scale", 1.0),
                     beta=kw.get("beta"))
        check(case, run(case, dev, **kw), exp, str(kw))


@pytest.mark.parametrize("V", [5003, 5008, 90000])  # 90000: the kept tensor-memory slice
def test_forward_only_matches(V):
    case = make_case(MEDIUM.with_(V=V, B=4, T=5) if V > 9000 else MEDIUM.with_(V=V), "bf16")
    dev = to_device(case)
    a = run(case, dev)
    b = run(case, dev, grad=None)
    assert b["grad"] is None
    assert torch.equal(a["out3"], b["out3"])
    assert torch.equal(a["per_seq"], b["per_seq"])


@pytest.mark.parametrize("V", [5003, 5008, 90001, 90000])
def test_in_place_gradient(V):
    case = make_case(MEDIUM.with_(V=V, B=4, T=5) if V > 9000 else MEDIUM.with_(V=V), "bf16")
    dev = to_device(case)
    ref = run(case, dev)
    X = dev["X"].clone()
    res = run(case, dict(dev, X=X), grad=X)
    assert torch.equal(res["out3"], ref["out3"])
    assert torch.equal(X, ref["grad"])


@pytest.mark.parametrize("V", [5003, 5008, 90001, 90000])
def test_skip_masked_grad_rows(V):
    case = make_case(MEDIUM.with_(V=V, B=4, T=5) if V > 9000 else MEDIUM.with_(V=V), "f32")
    dev = to_device(case)
    ref = run(case, dev)
    G = torch.full_like(dev["X"], 7.0)
    run(case, dev, grad=G, skip_masked_grad_rows=True)
    m = dev["mask"].bool()
    assert torch.equal(G[m], ref["grad"][m])
    assert torch.all(G[~m] == 7.0)
    assert torch.all(ref["grad"][~m] == 0.0)


@pytest.mark.parametrize("V", [5003, 5008, 90001, 90000])
def test_identity_ref_is_policy(V):
    case = make_case(MEDIUM.with_(V=V, B=4, T=5) if V > 9000 else MEDIUM.with_(V=V), "bf16")
    dev = to_device(case)
    res = run(case, dict(dev, Y=dev["X"]))
    assert res["out3"][2].item() == 0.0  # KL exactly 0
    assert torch.all(res["per_seq"][1] == 0.0)
    exp = expect(case, ref_is_policy=True)
    check(case, res, exp, "identity")


@pytest.mark.parametrize("V", [5003, 5008, 90001, 90000])
def test_masked_storage_is_never_read(V):
    case = make_case(MEDIUM.with_(V=V, B=4, T=5) if V > 9000 else MEDIUM.with_(V=V), "f32")
    dev = to_device(case)
    ref = run(case, dev)
    m = dev["mask"].bool()
    X, Y = dev["X"].clone(), dev["Y"].clone()
    X[~m] = float("nan")
    Y[~m] = float("inf")
    acts = dev["acts"].clone()
    acts[~m] = -12345
    old = dev["old"].clone()
    old[~m] = float("nan")
    res = run(case, dict(dev, X=X, Y=Y, acts=acts, old=old))
    for k in ("out3", "per_seq", "logps", "adv", "grad"):
        assert torch.equal(res[k], ref[k]), k


@pytest.mark.parametrize("V", [1531, 1536])
def test_bitwise_run_to_run(V):
    case = make_case(CSR.with_(V=V), "f32")
    dev = to_device(case)
    a, b = run(case, dev), run(case, dev)
    for k in ("out3", "per_seq", "logps", "grad"):
        assert torch.equal(a[k], b[k]), k


def test_all_masked_and_empty():
    case = make_case(TINY, "f32")
    dev = to_device(case)
    res = run(case, dict(dev, mask=torch.zeros_like(dev["mask"])))
    assert torch.all(res["out3"] == 0) and torch.all(res["grad"] == 0)
    for B, T in ((0, 4), (4, 0)):
        X = torch.zeros((B, T, 5), device="cuda")
        res = g.grpo_loss_fwd_bwd(X, X, torch.zeros((B, T), dtype=torch.int64, device="cuda"),
                                  torch.zeros((B, T), device="cuda"),
                                  torch.zeros((B, T), dtype=torch.uint8, device="cuda"),
                                  torch.zeros(B, device="cuda"), samples_per_prompt=2 if B else 0,
                                  group_boundaries=None if B else [0])
        torch.cuda.synchronize()
        assert torch.all(res["out3"] == 0)


def test_device_detected_errors():
    case = make_case(TINY, "f32")
    dev = to_device(case)
    acts = dev["acts"].clone()
    acts[0, 0] = TINY.V  # active token (every row has >= 4 active)
    res = run(case, dict(dev, acts=acts))
    assert g.grpo_read_device_status(res["workspace"]) == 16
    assert torch.all(torch.isnan(res["out3"]))
    R = dev["R"].clone()
    R[3] = float("nan")
    res = run(case, dict(dev, R=R))
    assert g.grpo_read_device_status(res["workspace"]) == 64
    assert torch.all(torch.isnan(res["out3"]))
    res = run(case, dev, samples_per_prompt=0, group_boundaries=[0, 5, 5, 8])
    assert g.grpo_read_device_status(res["workspace"]) == 32
    # a clean call on the same workspace resets the status
    res = run(case, dev, workspace=res["workspace"])
    assert g.grpo_read_device_status(res["workspace"]) == 0


def test_group_adv_entry_point():
    w = CSR
    R = torch.from_numpy(w.rewards()).cuda()
    gb = torch.from_numpy(w.group_boundaries()).cuda()
    for eps_add in (False, True):
        A = g.grpo_group_adv(R, group_boundaries=gb, eps_add=eps_add)
        want = oracle.group_advantages(w.rewards(), w.group_boundaries(), eps_add=eps_add)
        assert np.allclose(A.cpu().numpy(), want.astype(np.float32), rtol=1e-6, atol=1e-7)
    R2 = torch.from_numpy(TINY.rewards()).cuda()
    A = g.grpo_group_adv(R2, samples_per_prompt=4)
    want = oracle.group_advantages(TINY.rewards(), TINY.group_boundaries())
    assert np.array_equal(A.cpu().numpy(), want.astype(np.float32))


# ---------------------------------------------------------------------------
# logps-only boundary
# ---------------------------------------------------------------------------
LOGPS_SMALL = synth.WORKLOADS["logps"].with_(name="logps_small", B=24, T=64, len_range=(8, 64))


def _logps_case(w):
    lp, old, ref = w.logps_inputs()
    return dict(lp=lp, old=old, ref=ref, mask=w.completion_mask(), R=w.rewards(),
                bounds=w.group_boundaries())


def _logps_run(w, c, ref=True, **kw):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = dict(clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta, reduction=w.reduction,
                want_per_seq=True, want_adv=True)
    if w.samples_per_prompt:
        args["samples_per_prompt"] = w.samples_per_prompt
    else:
        args["group_boundaries"] = t(c["bounds"])
    args.update(kw)
    res = g.grpo_loss_from_logps(t(c["lp"]), t(c["old"]), t(c["ref"]) if ref else None,
                                 t(c["mask"]), t(c["R"]), **args)
    torch.cuda.synchronize()
    return res


def _logps_check(w, c, res, beta=None, reduction=None, ref=True):
    A = oracle.group_advantages(c["R"], c["bounds"])
    exp = oracle.loss_from_logps(c["lp"], c["ref"] if ref else None, c["old"], c["mask"], A,
                                 w.eps_lo, w.eps_hi, w.beta if beta is None else beta,
                                 reduction=w.reduction if reduction is None else reduction)
    out = res["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], k)
    ps = res["per_seq"].cpu().numpy().astype(np.float64)
    assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-5)
    assert np.array_equal(ps[2], exp["per_seq_active"])
    if res["grad"] is not None:
        want = exp["w"].astype(np.float32)
        r = exp["ratio"]
        band = (np.abs(r - (1 - np.float32(w.eps_lo))) < 1e-6) | (np.abs(r - (1 + np.float32(w.eps_hi))) < 1e-6)
        got = res["grad"].cpu().numpy()
        ok = np.abs(got.astype(np.float64) - want) <= np.spacing(np.abs(want)) + 1e-9
        assert np.all(ok | band), np.argwhere(~(ok | band))[:5]


@pytest.mark.parametrize("mask", ["prefix", "full"])
def test_logps_small(mask):
    w = LOGPS_SMALL.with_(mask=mask)
    c = _logps_case(w)
    _logps_check(w, c, _logps_run(w, c))


def test_logps_odd_T_sequence_mean_and_no_ref():
    w = LOGPS_SMALL.with_(T=37, len_range=(0, 37), reduction=1)
    c = _logps_case(w)
    _logps_check(w, c, _logps_run(w, c))
    _logps_check(w, c, _logps_run(w, c, ref=False, beta=0.0), beta=0.0, ref=False)


def _mask_pattern(B, T, pattern, seed):
    rng = np.random.default_rng(seed)
    t = np.arange(T)[None, :]
    if pattern == "random":  # ~70% active, nonzero bytes of several values
        m = (rng.random((B, T)) < 0.7) * rng.choice([1, 7, 255], size=(B, T))
    elif pattern == "suffix":  # a masked prefix, then active to a ragged end
        lo = rng.integers(0, T, size=B)[:, None]
        hi = rng.integers(0, T + 1, size=B)[:, None]
        m = (t >= lo) & (t < np.maximum(hi, lo + 1))
    else:  # "single": one active token per sequence (none in sequence 0)
        m = t == rng.integers(0, T, size=B)[:, None]
        m[0] = False
    return np.ascontiguousarray(m.astype(np.uint8))


@pytest.mark.parametrize("T", [2064, 100])
@pytest.mark.parametrize("pattern", ["random", "suffix", "single"])
def test_logps_mask_patterns(T, pattern):
    # T=2064: rows staged through shared memory in three 1,024-token chunks
    # (the ring of two wraps, the last chunk is partial); T=100: the register
    # path.  The random mask leaves most vectors partly active: those go to the
    # general path after the token loop, several per thread.
    w = LOGPS_SMALL.with_(B=16, T=T)
    c = _logps_case(w)
    c["mask"] = _mask_pattern(w.B, w.T, pattern, seed=T)
    for reduction in (0, 1):
        _logps_check(w, c, _logps_run(w, c, reduction=reduction), reduction=reduction)


def test_logps_large_weights_take_the_precise_path():
    # 2 sequences, 3 tokens: weights ~0.3, far above the fp32 budget
    w = LOGPS_SMALL.with_(B=8, T=4, len_range=(0, 2))
    c = _logps_case(w)
    _logps_check(w, c, _logps_run(w, c))


@pytest.mark.parametrize("flags", [0, g.GRPO_FLAG_SEPARATE_PREP], ids=["one-launch", "two-launch"])
def test_logps_every_vector_on_the_general_path(flags):
    # log ratios ~N(0, 2): nearly every vector fails the fast path's range
    # check, so each thread evaluates its whole share of the row (eight vectors
    # at T=4096) after the token loop, from its list in the workspace
    w = LOGPS_SMALL.with_(name="logps_general", B=8, T=4096, len_range=(3000, 4096),
                          old_sigma=2.0, ref_logp_sigma=1.0)
    c = _logps_case(w)
    for reduction in (0, 1):
        _logps_check(w, c, _logps_run(w, c, reduction=reduction, extra_flags=flags),
                     reduction=reduction)
