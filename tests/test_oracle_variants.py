"""Pins of the oracle's loss variants -- the KL estimators k1 / k2, the dual
clip, CISPO, the fixed-constant (Dr.GRPO) normaliser and the clip counters --
against finite differences, a library routine, closed forms and invariants.
The hand-worked fixtures for the same variants live in
``tests/golden/hand_worked.json``.  CPU only."""
import numpy as np
import pytest
import torch

import oracle

EPS_LO, EPS_HI = 0.2, 0.28


def _logps_case(seed, B=6, T=7, old_sd=0.3, ref_sd=0.2):
    rng = np.random.default_rng(seed)
    logp = rng.normal(-2, 0.5, (B, T))
    old = logp + rng.normal(0, old_sd, (B, T))
    ref = logp + rng.normal(0, ref_sd, (B, T))
    mask = (rng.random((B, T)) < 0.8).astype(np.uint8)
    mask[:, 0] = 1
    A = oracle.group_advantages(rng.normal(size=B).astype(np.float32), [0, 2, 4, 6])
    return logp, old, ref, mask, A


def _loss(logp, old, ref, mask, A, beta=0.04, **kw):
    return oracle.loss_from_logps(logp, ref, old, mask, A, EPS_LO, EPS_HI, beta, **kw)


def _near_kink(r, A, dual_c=None, band=1e-4):
    near = (np.abs(r - (1 + EPS_HI)) < band) | (np.abs(r - (1 - EPS_LO)) < band)
    if dual_c is not None:
        near |= np.abs(r - dual_c) < band
    return near


# ----------------------------------------------------------------------------
# finite differences: the gradient formula of each variant against its value
# ----------------------------------------------------------------------------
VARIANTS = [
    dict(kl="k1"),
    dict(kl="k2"),
    dict(dual_clip_c=1.6),
    dict(dual_clip_c=1.6, kl="k2", reduction=1),
    dict(reduction=oracle.FIXED_CONSTANT, norm_constant=17.5),
    dict(reduction=oracle.FIXED_CONSTANT, norm_constant=3.0, kl="k1", dual_clip_c=2.0),
]


@pytest.mark.parametrize("kw", VARIANTS, ids=lambda k: "-".join(f"{a}={b}" for a, b in k.items()))
def test_finite_difference_variants(kw):
    logp, old, ref, mask, A = _logps_case(7, old_sd=0.45)
    res = _loss(logp, old, ref, mask, A, **kw)
    near = _near_kink(res["ratio"], A, kw.get("dual_clip_c"))
    checked = 0
    for b in range(logp.shape[0]):
        for t in range(logp.shape[1]):
            if not mask[b, t] or near[b, t]:
                continue
            h = 1e-6
            lpp = logp.copy(); lpp[b, t] += h
            lpm = logp.copy(); lpm[b, t] -= h
            fd = (_loss(lpp, old, ref, mask, A, **kw)["loss"]
                  - _loss(lpm, old, ref, mask, A, **kw)["loss"]) / (2 * h)
            assert fd == pytest.approx(res["w"][b, t], rel=1e-6, abs=1e-10), (b, t)
            checked += 1
    assert checked > 25


def test_dual_clip_is_active_in_the_fd_case():
    # the FD case above must actually reach the dual-clip branch
    logp, old, ref, mask, A = _logps_case(7, old_sd=0.45)
    res = _loss(logp, old, ref, mask, A, dual_clip_c=1.6)
    assert res["clip_counts"][2] > 0


# ----------------------------------------------------------------------------
# CISPO
# ----------------------------------------------------------------------------
def test_cispo_special_case_is_cross_entropy_gradient():
    # A = +1, r = 1 (old = logp), one active token, beta = 0: the CISPO loss
    # is -logp, i.e. cross-entropy, and its logits gradient is torch's.
    rng = np.random.default_rng(3)
    V = 29
    x = rng.normal(size=(2, 1, V))
    lp = torch.log_softmax(torch.from_numpy(x[0, 0]), -1)[7].item()
    res = oracle.fused(x, x, "f64", np.array([[7], [0]]), np.array([[lp], [0.0]]),
                       np.array([[1], [0]], np.uint8), np.array([1, 0], np.float32),
                       np.array([0, 2]), 0.2, 0.2, 0.0, surrogate="cispo")
    xt = torch.from_numpy(x[0, 0]).clone().requires_grad_(True)
    ce = torch.nn.functional.cross_entropy(xt[None], torch.tensor([7]), reduction="sum")
    ce.backward()
    assert res["loss"] == pytest.approx(ce.item(), rel=1e-14)
    assert np.allclose(res["grad_f64"][0, 0], xt.grad.numpy(), rtol=0, atol=1e-14)


def test_cispo_gradient_equals_clip_surrogate_inside_the_clip_range():
    # inside [1 - eps_lo, 1 + eps_hi] both surrogates give -A r; outside,
    # CISPO keeps -A clip(r) where the clipped surrogate gives 0 or -A r
    logp, old, ref, mask, A = _logps_case(11, old_sd=0.3)
    a = _loss(logp, old, ref, mask, A, beta=0.0)
    b = _loss(logp, old, ref, mask, A, beta=0.0, surrogate="cispo")
    r = a["ratio"]
    m = mask.astype(bool)
    inside = m & (r >= 1 - EPS_LO) & (r <= 1 + EPS_HI)
    outside = m & ~inside
    assert inside.sum() > 5 and outside.sum() > 5
    assert np.allclose(a["w"][inside], b["w"][inside], rtol=1e-15, atol=0)
    N = m.sum()
    Ab = np.broadcast_to(A[:, None], r.shape)
    hi = outside & (r > 1 + EPS_HI)
    lo = outside & (r < 1 - EPS_LO)
    assert np.allclose(b["w"][hi], -Ab[hi] * (1 + EPS_HI) / N, rtol=1e-14)
    assert np.allclose(b["w"][lo], -Ab[lo] * (1 - EPS_LO) / N, rtol=1e-14)
    # CISPO's counters count clipped weights whatever the sign of A
    assert list(b["clip_counts"]) == [hi.sum(), lo.sum(), 0]


def test_cispo_rejects_dual_clip():
    logp, old, ref, mask, A = _logps_case(1)
    with pytest.raises(ValueError):
        _loss(logp, old, ref, mask, A, surrogate="cispo", dual_clip_c=3.0)


# ----------------------------------------------------------------------------
# dual clip
# ----------------------------------------------------------------------------
def test_dual_clip_limits():
    logp, old, ref, mask, A = _logps_case(5, old_sd=0.6)
    base = _loss(logp, old, ref, mask, A)
    huge = _loss(logp, old, ref, mask, A, dual_clip_c=1e30)
    for k in ("loss", "policy_loss", "kl"):
        assert huge[k] == base[k]
    assert np.array_equal(huge["w"], base["w"])
    dual = _loss(logp, old, ref, mask, A, dual_clip_c=1.5, beta=0.0)
    r = dual["ratio"]
    m = mask.astype(bool)
    Ab = np.broadcast_to(A[:, None], r.shape)
    hit = m & (Ab < 0) & (r > 1.5)
    assert hit.sum() > 0
    # the bound binds: p = -c A there, and the policy gradient is 0
    assert np.all(dual["w"][hit] == 0.0)
    # positive-advantage sequences are untouched
    pos = A > 0
    assert np.array_equal(dual["per_seq_policy"][pos],
                          _loss(logp, old, ref, mask, A, beta=0.0)["per_seq_policy"][pos])


def test_dual_clip_value_on_a_single_token():
    # one token, A = -1, r = e: min(rA, clip(r)A) = min(-e, -1.28) = -e, and
    # the dual clip gives max(-e, -c): -c for c < e, -e for c > e
    logp = np.array([[-1.0], [-1.0]])
    old = np.array([[-2.0], [-1.0]])  # r = e for sequence 0
    mask = np.array([[1], [0]], np.uint8)
    A = np.array([-1.0, 1.0])
    for c, p in ((2.0, 2.0), (3.0, np.e)):
        res = oracle.loss_from_logps(logp, None, old, mask, A, EPS_LO, EPS_HI, 0.0, dual_clip_c=c)
        assert res["policy_loss"] == pytest.approx(p, rel=1e-15)


# ----------------------------------------------------------------------------
# KL estimators
# ----------------------------------------------------------------------------
def test_k1_k2_closed_forms_and_k3_agreement():
    rng = np.random.default_rng(2)
    B, T = 4, 9
    logp = rng.normal(-2, 0.5, (B, T))
    mask = np.ones((B, T), np.uint8)
    A = np.zeros(B)
    shift = 0.3
    ref = logp - shift  # log ratio logp - ref = 0.3 on every token
    k1 = _loss(logp, logp, ref, mask, A, kl="k1")
    k2 = _loss(logp, logp, ref, mask, A, kl="k2")
    k3 = _loss(logp, logp, ref, mask, A)
    assert k1["kl"] == pytest.approx(shift, rel=1e-14)
    assert k2["kl"] == pytest.approx(shift * shift / 2, rel=1e-14)
    assert k3["kl"] == pytest.approx(np.expm1(-shift) + shift, rel=1e-14)
    # k2 and k3 agree to second order: |k3 - k2| <= |d|^3 e^|d| / 6
    for s in (1e-3, 1e-2, 0.1):
        a = _loss(logp, logp, logp - s, mask, A, kl="k2")["kl"]
        b = _loss(logp, logp, logp - s, mask, A)["kl"]
        assert abs(a - b) <= s ** 3 * np.exp(s) / 6 * (1 + 1e-9)
    # ref == policy: every estimator is 0
    for kl in ("k1", "k2", "k3"):
        assert _loss(logp, logp, logp, mask, A, kl=kl)["kl"] == 0.0


def test_kl_gradients_at_zero_advantage():
    # A = 0: w is the KL part alone, c beta g_kl
    logp, old, ref, mask, _ = _logps_case(13)
    A = np.zeros(logp.shape[0])
    m = mask.astype(bool)
    N = m.sum()
    d = ref - logp
    want = {"k1": np.ones_like(d), "k2": -d, "k3": -np.expm1(d)}
    for kl, g in want.items():
        res = _loss(logp, old, ref, mask, A, beta=0.5, kl=kl)
        assert np.allclose(res["w"][m], 0.5 * g[m] / N, rtol=1e-14, atol=0)
        assert np.all(res["w"][~m] == 0.0)


# ----------------------------------------------------------------------------
# fixed-constant normaliser
# ----------------------------------------------------------------------------
def test_fixed_constant_normaliser():
    logp, old, ref, mask, A = _logps_case(17)
    N = int(mask.sum())
    tm = _loss(logp, old, ref, mask, A)
    fc = _loss(logp, old, ref, mask, A, reduction=oracle.FIXED_CONSTANT, norm_constant=float(N))
    for k in ("loss", "policy_loss", "kl"):
        assert fc[k] == tm[k]
    assert np.array_equal(fc["w"], tm["w"])
    C = 1000.0  # independent of the mask: scales as N / C
    fc2 = _loss(logp, old, ref, mask, A, reduction=oracle.FIXED_CONSTANT, norm_constant=C)
    assert fc2["loss"] == pytest.approx(tm["loss"] * N / C, rel=1e-13)
    mask2 = mask.copy()
    mask2[:, -1] = 0
    fc3 = _loss(logp, old, ref, mask2, A, reduction=oracle.FIXED_CONSTANT, norm_constant=C)
    m2 = mask2.astype(bool)
    assert np.allclose(fc3["w"][m2], fc2["w"][m2], rtol=0, atol=0)
    with pytest.raises(ValueError):
        _loss(logp, old, ref, mask, A, reduction=oracle.FIXED_CONSTANT)


# ----------------------------------------------------------------------------
# clip counters, through the gradient: at beta = 0 a token of nonzero A has
# zero gradient exactly when one of the clips removes it
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dual", [None, 1.5])
def test_clip_counters_match_zero_gradient_tokens(dual):
    logp, old, ref, mask, A = _logps_case(23, B=6, T=40, old_sd=0.5)
    assert np.all(A != 0)
    res = _loss(logp, old, ref, mask, A, beta=0.0, dual_clip_c=dual)
    m = mask.astype(bool)
    zero = m & (res["w"] == 0.0)
    assert zero.sum() == res["clip_counts"].sum() > 0
    r = res["ratio"]
    Ab = np.broadcast_to(A[:, None], r.shape)
    assert res["clip_counts"][0] == (zero & (Ab > 0)).sum()
    assert res["clip_counts"][1] + res["clip_counts"][2] == (zero & (Ab < 0)).sum()
    if dual is None:
        assert res["clip_counts"][2] == 0


# ----------------------------------------------------------------------------
# GSPO: one ratio per sequence
# ----------------------------------------------------------------------------
def test_gspo_finite_differences():
    # the gradient of token t carries the coupling through rho_i: perturbing
    # one log-prob moves every token's term of its sequence
    logp, old, ref, mask, A = _logps_case(29, old_sd=0.3)
    kw = dict(reduction=oracle.SEQUENCE_MEAN, ratio_level="sequence")
    res = _loss(logp, old, ref, mask, A, **kw)
    near = _near_kink(res["ratio"], A)
    checked = 0
    for b in range(logp.shape[0]):
        if near[b][mask[b].astype(bool)].any():
            continue
        for t in range(logp.shape[1]):
            if not mask[b, t]:
                continue
            h = 1e-6
            lpp = logp.copy(); lpp[b, t] += h
            lpm = logp.copy(); lpm[b, t] -= h
            fd = (_loss(lpp, old, ref, mask, A, **kw)["loss"]
                  - _loss(lpm, old, ref, mask, A, **kw)["loss"]) / (2 * h)
            assert fd == pytest.approx(res["w"][b, t], rel=1e-6, abs=1e-10), (b, t)
            checked += 1
    assert checked > 15


def test_gspo_reduces_to_token_ratios():
    logp, old, ref, mask, A = _logps_case(31, T=9)
    kw = dict(reduction=oracle.SEQUENCE_MEAN)
    # single-token sequences: rho_i is the token's own ratio, bit for bit
    one = np.zeros_like(mask)
    one[:, 3] = 1
    a = _loss(logp, old, ref, one, A, **kw)
    b = _loss(logp, old, ref, one, A, ratio_level="sequence", **kw)
    for k in ("loss", "policy_loss", "kl"):
        assert a[k] == b[k]
    assert np.array_equal(a["w"], b["w"])
    # equal log ratios within each sequence: the same loss up to rounding
    same = logp - (logp[:, :1] - old[:, :1])
    c = _loss(logp, same, ref, mask, A, **kw)
    d = _loss(logp, same, ref, mask, A, ratio_level="sequence", **kw)
    assert d["loss"] == pytest.approx(c["loss"], rel=1e-13)
    assert np.allclose(d["w"], c["w"], rtol=1e-12, atol=1e-18)


def test_gspo_rejects_token_level_reductions_and_cispo():
    logp, old, ref, mask, A = _logps_case(1)
    with pytest.raises(ValueError):
        _loss(logp, old, ref, mask, A, ratio_level="sequence")  # token mean
    with pytest.raises(ValueError):
        _loss(logp, old, ref, mask, A, ratio_level="sequence", reduction=oracle.SEQUENCE_MEAN,
              surrogate="cispo")
