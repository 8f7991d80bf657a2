"""The parity tests' gradient tolerance, one ulp of the output dtype at the
oracle's rounded value plus 1e-9, computed two ways: on the host (numpy)
and on the device (torch, used by the full-size tests).  Both must agree
with the spacing of the dtype, zero and subnormals included."""
import numpy as np
import torch

from workload_inputs import ulp, ulp_device


def _values(dtype):
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-45, 5, 4000),
                        [0.0, 2.0 ** -126, 2.0 ** -130, 2.0 ** -14, 2.0 ** -20, 1.0, -1.0, 3.0]])
    t = torch.from_numpy(x)
    t = t.to({"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype])
    return t.to(torch.float64)


def test_host_and_device_ulp_agree_with_the_dtype_spacing():
    for dtype, tdt in (("f32", torch.float32), ("bf16", torch.bfloat16), ("f16", torch.float16)):
        o = _values(dtype)
        u_host = ulp(o.numpy(), dtype)
        u_dev = ulp_device(o, dtype).numpy()
        assert np.array_equal(u_host, u_dev), dtype
        # the spacing itself: the next representable value above |o|
        a = o.abs().to(tdt)
        nxt = torch.nextafter(a.float(), torch.tensor(np.inf)).to(tdt) if tdt != torch.float32 \
            else torch.nextafter(a, torch.tensor(np.inf, dtype=torch.float32))
        if tdt != torch.float32:
            # nextafter in f32 then rounding back can stay put; step the bits instead
            bits = a.view(torch.int16).to(torch.int32) + 1
            nxt = bits.to(torch.int16).view(tdt)
        gap = nxt.to(torch.float64) - a.to(torch.float64)
        finite = torch.isfinite(nxt.to(torch.float64))
        assert np.array_equal(gap[finite].numpy(), u_host[finite.numpy()]), dtype
    # zero gets the subnormal spacing, not a normal-range one
    assert ulp(np.array([0.0]), "bf16")[0] == 2.0 ** -133
    assert ulp(np.array([0.0]), "f16")[0] == 2.0 ** -24
