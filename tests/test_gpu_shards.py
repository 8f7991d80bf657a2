"""Sequence-sharded determinism (RL-Kernel "GRPO Loss", "Tensor and Data
Parallel"): a batch split into K contiguous shards of whole sequences --
emulated as K "ranks" on one GPU, each with its own workspace -- gives
bit-identical gradients, per-sequence totals and loss outputs to the
unsharded call, for every K, with advantage groups straddling shards.  The
exchange is what the page describes: the active-token counts gathered as
integers, the per-sequence totals concatenated in shard order.  The same
page's claim is also that this common result is the loss: every partition's
loss outputs, per-sequence totals, clip counts and gradients are compared
with the oracle as well."""
import numpy as np
import pytest
import torch

import grad_row_online_gb300 as g
import oracle
import synth
from workload_inputs import (assert_grad_rows, assert_scalar, make_case, to_device,
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


# 12 sequences in groups of 4; ragged lengths, some empty sequences
BATCH = synth.Workload("shards", B=12, T=10, V=3001, seed=121, sigma=2.0, ref_sigma=0.2,
                       samples_per_prompt=4, reward_p=0.5, len_range=(0, 10), eps_lo=0.2,
                       eps_hi=0.28, beta=0.1, old_sigma=0.3)
PARTITIONS = {
    "1": [12],
    "2": [6, 6],
    "straddle": [5, 7],           # shard boundary inside a group
    "3-uneven": [1, 8, 3],
    "with-empty": [0, 12, 0],
    "12": [1] * 12,
}
OPTIONS = {
    "token-mean": dict(),
    "sequence-mean": dict(reduction="sequence_mean"),
    "fixed-k2-dual": dict(reduction="fixed_constant", norm_constant=40.0, kl="k2",
                          dual_clip_c=1.4),
    "gspo": dict(reduction="sequence_mean", ratio_level="sequence"),
}


_RED = {"token_mean": oracle.TOKEN_MEAN, "sequence_mean": oracle.SEQUENCE_MEAN,
        "fixed_constant": oracle.FIXED_CONSTANT}


def _oracle_kw(opts: dict) -> dict:
    kw = {k: opts[k] for k in ("kl", "dual_clip_c", "norm_constant", "ratio_level") if k in opts}
    kw["reduction"] = _RED[opts.get("reduction", "token_mean")]
    return kw


def _near_clip(exp, w, opts, band=1e-6):
    """Tokens whose oracle ratio is within `band` (relative) of a clip bound:
    either branch's gradient is a correct reading there."""
    r = exp["ratio"]
    near = np.zeros(r.shape, bool)
    for b in (1.0 - float(np.float32(w.eps_lo)), 1.0 + float(np.float32(w.eps_hi)),
              float(np.float32(opts["dual_clip_c"])) if opts.get("dual_clip_c") else None):
        if b is not None:
            near |= np.abs(r - b) <= band * b
    return near


def _check_against_oracle(got, exp, near, what, dtype=None):
    """One partition's results against the oracle: the loss outputs (1e-5
    relative), per-sequence totals, clip counts (tokens at a clip kink may
    count either way) and every gradient element (1 ulp + 1e-9; logits
    gradients of dtype `dtype`, else the f32 dL/dlogp)."""
    out = got["out3"].cpu().numpy().astype(np.float64)
    for i, k in enumerate(("loss", "policy_loss", "kl")):
        assert_scalar(out[i], exp[k], f"{what} {k}")
    if got.get("per_seq") is not None:
        ps = got["per_seq"].cpu().numpy().astype(np.float64)
        assert np.allclose(ps[0], exp["per_seq_policy"], rtol=1e-5, atol=1e-6), what
        assert np.allclose(ps[1], exp["per_seq_kl"], rtol=1e-5, atol=1e-7), what
        assert np.array_equal(ps[2], exp["per_seq_active"]), what
    if got.get("clips") is not None:
        c = got["clips"].cpu().numpy()
        assert np.all(np.abs(c - exp["clip_counts"]) <= near.sum()), (what, c, exp["clip_counts"])
    if dtype is not None:
        assert_grad_rows(torch_storage(got["grad"])[~near], exp["grad"][~near], dtype,
                         what=f"{what} grad")
    else:
        want = exp["w"].astype(np.float32)
        gw = got["grad"].cpu().numpy()
        ok = np.abs(gw.astype(np.float64) - want) <= np.spacing(np.abs(want)) + 1e-9
        assert np.all(ok | near), (what, np.argwhere(~(ok | near))[:5])


def _bounds(sizes):
    out, s = [], 0
    for n in sizes:
        out.append((s, s + n))
        s += n
    return out


def _sharded_logits(dev, w, sizes, opts):
    """Run every shard, exchange counts and totals, finalize."""
    parts = _bounds(sizes)
    counts = [g.grpo_count_active(dev["mask"][a:b]) for a, b in parts]
    global_counts = torch.stack(counts).sum(0)  # integer sums: exact in any order
    grads, per_seq, totals, clips = [], [], [], []
    for a, b in parts:
        tot = g.totals_buffer(b - a)
        res = g.grpo_loss_fwd_bwd(dev["X"][a:b], dev["Y"][a:b], dev["acts"][a:b],
                                  dev["old"][a:b], dev["mask"][a:b], dev["R"],
                                  samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                  clip_eps_hi=w.eps_hi, beta=w.beta, want_per_seq=True,
                                  want_clip_counts=True,
                                  shard=g.Shard(a, global_counts, tot), **opts)
        grads.append(res["grad"])
        per_seq.append(res["per_seq"])
        totals.append(tot)
        clips.append(res["clip_counts"])
    all_totals = torch.cat(totals)  # shard order = sequence order
    out3 = g.grpo_loss_finalize(all_totals, global_counts, beta=w.beta,
                                reduction=opts.get("reduction", "token_mean"),
                                norm_constant=opts.get("norm_constant"))
    torch.cuda.synchronize()
    return dict(out3=out3, grad=torch.cat(grads), per_seq=torch.cat(per_seq, dim=1),
                totals=all_totals, clips=torch.stack(clips).sum(0), counts=global_counts)


# V = 70001: rows long enough for the row kernel's tensor-memory slice
@pytest.mark.parametrize("V", [3001, 70001])
@pytest.mark.parametrize("opt", list(OPTIONS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_logits_shards_are_bitwise_identical(dtype, opt, V):
    w = BATCH.with_(V=V)
    case = make_case(w, dtype)
    dev = to_device(case)
    opts = OPTIONS[opt]
    whole = g.grpo_loss_fwd_bwd(dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"],
                                dev["R"], samples_per_prompt=w.samples_per_prompt,
                                clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta,
                                want_per_seq=True, want_clip_counts=True, **opts)
    torch.cuda.synchronize()
    ref = _sharded_logits(dev, w, PARTITIONS["1"], opts)
    # one shard through finalize reproduces the plain call
    assert torch.equal(ref["out3"], whole["out3"])
    assert torch.equal(ref["grad"], whole["grad"])
    assert torch.equal(ref["per_seq"], whole["per_seq"])
    assert torch.equal(ref["clips"], whole["clip_counts"])
    assert int(ref["counts"][0]) == int(case["mask"].sum())
    exp = oracle.fused(case["X"], case["Y"], dtype, case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta, **_oracle_kw(opts))
    near = _near_clip(exp, w, opts)
    for name, sizes in PARTITIONS.items():
        got = _sharded_logits(dev, w, sizes, opts)
        for k in ("out3", "grad", "per_seq", "totals", "clips", "counts"):
            assert torch.equal(got[k], ref[k]), (name, k)
        _check_against_oracle(got, exp, near, f"{dtype} {opt} V={V} {name}", dtype)


LOGPS = synth.WORKLOADS["logps"].with_(name="logps_shards", B=12, T=64, len_range=(0, 64),
                                      samples_per_prompt=4, old_sigma=0.3, ref_logp_sigma=0.1,
                                      beta=0.1)


def _sharded_logps(t, w, sizes, opts, flags=0):
    parts = _bounds(sizes)
    counts = [g.grpo_count_active(t["mask"][a:b]) for a, b in parts]
    global_counts = torch.stack(counts).sum(0)
    grads, totals, per_seq, clips = [], [], [], []
    for a, b in parts:
        tot = g.totals_buffer(b - a)
        res = g.grpo_loss_from_logps(t["lp"][a:b], t["old"][a:b], t["ref"][a:b], t["mask"][a:b],
                                     t["R"], samples_per_prompt=w.samples_per_prompt,
                                     clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta,
                                     want_per_seq=True, want_clip_counts=True,
                                     shard=g.Shard(a, global_counts, tot), extra_flags=flags,
                                     **opts)
        grads.append(res["grad"])
        totals.append(tot)
        per_seq.append(res["per_seq"])
        clips.append(res["clip_counts"])
    all_totals = torch.cat(totals)
    out3 = g.grpo_loss_finalize(all_totals, global_counts, beta=w.beta,
                                reduction=opts.get("reduction", "token_mean"),
                                norm_constant=opts.get("norm_constant"))
    torch.cuda.synchronize()
    return dict(out3=out3, grad=torch.cat(grads), totals=all_totals,
                per_seq=torch.cat(per_seq, dim=1), clips=torch.stack(clips).sum(0))


@pytest.mark.parametrize("opt", list(OPTIONS))
@pytest.mark.parametrize("T", [64, 100, 37])  # staged, register and scalar paths
def test_logps_shards_are_bitwise_identical(T, opt):
    w = LOGPS.with_(T=T, len_range=(0, T))
    lp, old, ref = w.logps_inputs()
    host = dict(lp=lp, old=old, ref=ref, mask=w.completion_mask(), R=w.rewards())
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in host.items()}
    opts = OPTIONS[opt]
    whole = g.grpo_loss_from_logps(t["lp"], t["old"], t["ref"], t["mask"], t["R"],
                                   samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                   clip_eps_hi=w.eps_hi, beta=w.beta, **opts)
    torch.cuda.synchronize()
    ref_run = _sharded_logps(t, w, PARTITIONS["1"], opts)
    assert torch.equal(ref_run["out3"], whole["out3"])
    assert torch.equal(ref_run["grad"], whole["grad"])
    A = oracle.group_advantages(host["R"], w.group_boundaries())
    exp = oracle.loss_from_logps(lp, ref, old, host["mask"], A, w.eps_lo, w.eps_hi, w.beta,
                                 **_oracle_kw(opts))
    near = _near_clip(exp, w, opts)
    for name, sizes in PARTITIONS.items():
        got = _sharded_logps(t, w, sizes, opts)
        for k in ("out3", "grad", "totals", "per_seq", "clips"):
            assert torch.equal(got[k], ref_run[k]), (name, k)
        _check_against_oracle(got, exp, near, f"logps T={T} {opt} {name}")
    # the shards' advantages and counts from the separate pass: the same bits
    got = _sharded_logps(t, w, PARTITIONS["straddle"], opts, flags=g.GRPO_FLAG_SEPARATE_PREP)
    for k in ("out3", "grad", "totals", "per_seq", "clips"):
        assert torch.equal(got[k], ref_run[k]), ("separate pass", k)


def test_count_active_matches_the_mask():
    m = torch.from_numpy(BATCH.completion_mask()).cuda()
    m[3] = 0
    c = g.grpo_count_active(m)
    torch.cuda.synchronize()
    L = m.sum(1)
    assert int(c[0]) == int(L.sum()) and int(c[1]) == int((L > 0).sum())
    empty = g.grpo_count_active(m[:0])
    assert empty.tolist() == [0, 0]


def test_dp_helper_single_rank_matches_the_plain_call():
    from grad_row_online_gb300 import dp
    w = BATCH
    case = make_case(w, "bf16")
    dev = to_device(case)
    args = dict(policy=dev["X"], ref=dev["Y"], acts=dev["acts"], old=dev["old"],
                mask=dev["mask"], R=dev["R"])
    res = dp.sequence_sharded_loss(g.grpo_loss_fwd_bwd, args, dev["mask"], 0, beta=w.beta,
                                   samples_per_prompt=w.samples_per_prompt, clip_eps=w.eps_lo,
                                   clip_eps_hi=w.eps_hi)
    whole = g.grpo_loss_fwd_bwd(dev["X"], dev["Y"], dev["acts"], dev["old"], dev["mask"],
                                dev["R"], samples_per_prompt=w.samples_per_prompt,
                                clip_eps=w.eps_lo, clip_eps_hi=w.eps_hi, beta=w.beta)
    torch.cuda.synchronize()
    assert torch.equal(res["out3"], whole["out3"])
    assert torch.equal(res["grad"], whole["grad"])
    exp = oracle.fused(case["X"], case["Y"], "bf16", case["acts"], case["old"], case["mask"],
                       case["R"], case["bounds"], w.eps_lo, w.eps_hi, w.beta)
    _check_against_oracle(res, exp, _near_clip(exp, w, {}), "dp helper", "bf16")
