"""The seeded input generator: determinism and the stated workload recipes."""
import numpy as np
import pytest

import synth
from synth import WORKLOADS


def test_normal_moments_and_determinism():
    z = synth.normal(123, synth.STREAM_POLICY, 0, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert np.array_equal(z[1000:1010], synth.normal(123, synth.STREAM_POLICY, 1000, 10))
    assert not np.array_equal(z[:10], synth.normal(124, synth.STREAM_POLICY, 0, 10))


def test_rows_are_independent_of_request_order():
    w = WORKLOADS["tiny"]
    a = w.logit_rows("policy", [5, 2, 9])
    b = w.logits_host("policy").reshape(w.rows, w.V)[[5, 2, 9]]
    assert np.array_equal(a, b)
    r = w.logit_rows("ref", [5])
    assert np.abs(r.astype(np.float64) - a[:1]).max() < 1.0


def test_bf16_rows_are_bf16_of_the_normal():
    w = WORKLOADS["large_vocab"].with_(B=1, T=2, V=4096)
    rows = w.logit_rows("policy", [0, 1])
    vals = (rows.astype(np.uint32) << 16).view(np.float32)
    assert abs(vals.std() - 3.0 * np.sqrt(1 + 0.01 * 64 / 9)) < 0.3  # N(0,3) + 1% of +8
    assert (vals > 6).mean() > 0.005


def test_tiny_recipe():
    w = WORKLOADS["tiny"]
    assert (w.B, w.T, w.V, w.samples_per_prompt) == (8, 16, 64, 4)
    L = w.lengths()
    assert L.min() >= 4 and L.max() <= 16
    assert set(np.unique(w.rewards())) <= {0.0, 1.0}
    a = w.action_ids()
    assert a.min() >= 0 and a.max() < 64


def test_large_vocab_recipe():
    w = WORKLOADS["large_vocab"]
    R = w.rewards()
    assert np.all(R[:8] == 0)  # the all-zero degenerate group
    assert 0 < R[8:].sum() < 8  # the other group is not degenerate
    L = w.lengths()
    assert L.min() >= 256 and L.max() <= 2048


def test_var_groups_recipe():
    w = WORKLOADS["var_groups"]
    gb = w.group_boundaries()
    sizes = np.diff(gb)
    assert gb[0] == 0 and gb[-1] == 64
    assert sizes.min() >= 2 and sizes[:-1].max() <= 16 and sizes[-1] <= 17
    L = w.lengths()
    assert (L == 0).sum() == 4
    assert L[L > 0].min() >= 16 and L.max() <= 512
    R = w.rewards()
    assert R.dtype == np.float32 and len(np.unique(R)) == 64


def test_logps_recipe():
    w = WORKLOADS["logps"].with_(B=16, T=64, len_range=(16, 64))
    lp, old, ref = w.logps_inputs()
    assert lp.dtype == np.float32 and lp.shape == (16, 64)
    assert abs(lp.mean() + 2) < 0.1
    assert abs((old - lp).std() - 0.05) < 0.01
    assert np.all(WORKLOADS["logps_full"].with_(B=8, T=8).completion_mask() == 1)
