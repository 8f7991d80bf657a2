"""The C ABI: the shared library loads, exports every function the headers
declare, and rejects bad arguments on the host before any CUDA call (so
these run without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

import grad_row_online_gb300 as g
from grad_row_online_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    srcs = [os.path.join(_build.CSRC, s) for s in os.listdir(_build.CSRC)]
    srcs.append(os.path.join(ROOT, "include", "grpo.h"))
    if not os.path.exists(_build.LIB) or any(os.path.getmtime(s) > os.path.getmtime(_build.LIB)
                                              for s in srcs):
        _build.build()
    return g.lib()


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(grpo_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"grpo_group_adv", "grpo_loss_fwd_bwd", "grpo_loss_from_logps",
            "grpo_workspace_size", "grpo_read_device_status", "grpo_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size(lib):
    assert g.grpo_workspace_size(8, 16) >= 256 + 2 * 8 * 16 * 8
    assert g.grpo_workspace_size(-1, 4) == 0
    assert g.grpo_workspace_size(0, 0) == 256 + 0 or g.grpo_workspace_size(0, 0) >= 256
    assert g.grpo_workspace_size(1024, 4096) % 256 == 0


def test_status_strings(lib):
    for code in (0, 1, 2, 3, 4, 5, 6, 7, 8, 16, 32, 64, 48):
        assert isinstance(g.grpo_status_string(code), str) and g.grpo_status_string(code)


# ---------------------------------------------------------------------------
# host validation (no pointer is ever dereferenced: fake addresses are fine)
# ---------------------------------------------------------------------------
FAKE = 1 << 20  # 16-byte aligned, never touched


def _groups(B=8, spp=4, bounds=None, G=0):
    gr = g._Groups()
    gr.num_seqs = B
    gr.samples_per_prompt = spp
    gr.group_boundaries = bounds
    gr.num_groups = G
    return gr


def _params(**kw):
    p = g._Params()
    p.clip_eps_lo, p.clip_eps_hi, p.beta, p.adv_eps, p.grad_scale = 0.2, 0.2, 0.04, 1e-6, 1.0
    p.reduction, p.flags = 0, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _fwd(lib, B=8, T=16, V=64, dt=0, gr=None, p=None, ws=FAKE, ws_bytes=None, **ptr):
    gr = gr or _groups(B)
    p = p or _params()
    ws_bytes = g.grpo_workspace_size(B, T) if ws_bytes is None else ws_bytes
    a = dict(policy=FAKE, ref=FAKE, act=FAKE, old=FAKE, mask=FAKE, rew=FAKE, grad=FAKE,
             out3=FAKE, per_seq=None, logps=None, adv=None)
    a.update(ptr)
    return lib.grpo_loss_fwd_bwd(a["policy"], a["ref"], dt, B, T, V, a["act"], a["old"], a["mask"],
                                 a["rew"], ctypes.byref(gr), ctypes.byref(p), a["grad"], a["out3"],
                                 a["per_seq"], a["logps"], a["adv"], ws, ws_bytes, None)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, dt=7) == 3                       # dtype
    assert _fwd(lib, V=0) == 2                        # V < 1
    assert _fwd(lib, B=-1) == 2
    assert _fwd(lib, T=(1 << 30) + 1) == 2            # positions within a sequence are 32-bit
    assert _fwd(lib, policy=None) == 1                # null input
    assert _fwd(lib, out3=None) == 1
    assert _fwd(lib, ws=None) == 1
    assert _fwd(lib, B=6, gr=_groups(B=6, spp=4)) == 2      # B % spp
    assert _fwd(lib, gr=_groups(B=9)) == 2                  # num_seqs != B
    assert _fwd(lib, gr=_groups(spp=0)) == 5                # no group spec
    assert _fwd(lib, gr=_groups(spp=4, bounds=FAKE, G=2)) == 5  # both
    assert _fwd(lib, gr=_groups(spp=0, bounds=FAKE, G=0)) == 2  # empty CSR
    assert _fwd(lib, gr=_groups(spp=0, bounds=FAKE, G=9)) == 2  # more groups than sequences
    assert _fwd(lib, gr=_groups(spp=0, bounds=FAKE + 4, G=2)) == 4  # misaligned CSR
    assert _fwd(lib, p=_params(clip_eps_lo=1.0)) == 6
    assert _fwd(lib, p=_params(clip_eps_lo=-0.1)) == 6
    assert _fwd(lib, p=_params(clip_eps_hi=-0.1)) == 6
    assert _fwd(lib, p=_params(beta=-1.0)) == 6
    assert _fwd(lib, p=_params(beta=float("nan"))) == 6
    assert _fwd(lib, p=_params(adv_eps=0.0)) == 6
    assert _fwd(lib, p=_params(grad_scale=float("inf"))) == 6
    assert _fwd(lib, p=_params(reduction=3)) == 6
    assert _fwd(lib, p=_params(flags=64)) == 6
    assert _fwd(lib, p=_params(flags=0x20000000)) == 6  # a bit the header does not define
    # loss variants
    assert _fwd(lib, p=_params(reduction=2)) == 6  # fixed constant without a constant
    assert _fwd(lib, p=_params(reduction=2, norm_constant=-1.0)) == 6
    assert _fwd(lib, p=_params(reduction=2, norm_constant=float("inf"))) == 6
    assert _fwd(lib, p=_params(kl_type=3)) == 6
    assert _fwd(lib, p=_params(kl_type=-1)) == 6
    assert _fwd(lib, p=_params(surrogate=2)) == 6
    assert _fwd(lib, p=_params(dual_clip_c=1.0)) == 6  # c must exceed 1
    assert _fwd(lib, p=_params(dual_clip_c=float("nan"))) == 6
    assert _fwd(lib, p=_params(surrogate=1, dual_clip_c=3.0)) == 6  # not with CISPO
    assert _fwd(lib, p=_params(clip_counts=FAKE + 4)) == 4  # misaligned counter array
    assert _fwd(lib, p=_params(ratio_level=2)) == 6
    assert _fwd(lib, p=_params(ratio_level=1)) == 6  # GSPO needs the sequence mean
    assert _fwd(lib, p=_params(ratio_level=1, reduction=1, surrogate=1)) == 6  # not with CISPO
    assert _fwd(lib, dt=1, policy=FAKE + 1) == 4      # bf16 pointer not 2-byte aligned
    assert _fwd(lib, act=FAKE + 4) == 4               # int64 ids
    assert _fwd(lib, ws=FAKE + 16) == 4               # workspace alignment
    assert _fwd(lib, ws_bytes=1000) == 7              # workspace size


def test_logps_and_adv_reject_bad_arguments(lib):
    gr, p = _groups(), _params()
    ws = g.grpo_workspace_size(8, 16)
    L = lib.grpo_loss_from_logps
    assert L(FAKE, FAKE, None, FAKE, 8, 16, FAKE, ctypes.byref(gr), ctypes.byref(p), None, FAKE,
             None, None, FAKE, ws, None) == 1  # beta > 0 without ref_logps
    assert L(FAKE, FAKE, FAKE, FAKE, 8, 16, FAKE, ctypes.byref(gr), ctypes.byref(p), None, FAKE,
             None, None, FAKE, 10, None) == 7
    assert L(FAKE + 2, FAKE, FAKE, FAKE, 8, 16, FAKE, ctypes.byref(gr), ctypes.byref(p), None,
             FAKE, None, None, FAKE, ws, None) == 4
    assert L(FAKE, FAKE, FAKE, FAKE, 8, (1 << 30) + 1, FAKE, ctypes.byref(gr), ctypes.byref(p),
             None, FAKE, None, None, FAKE, ws, None) == 2  # T > 2^30
    A = lib.grpo_group_adv
    assert A(FAKE, ctypes.byref(gr), ctypes.c_float(0.0), 0, FAKE, FAKE, ws, None) == 6
    assert A(FAKE, ctypes.byref(gr), ctypes.c_float(1e-6), 4, FAKE, FAKE, ws, None) == 6
    assert A(FAKE, ctypes.byref(gr), ctypes.c_float(1e-6), 0, None, FAKE, ws, None) == 1
    assert A(FAKE, ctypes.byref(_groups(B=8, spp=3)), ctypes.c_float(1e-6), 0, FAKE, FAKE, ws,
             None) == 2


def test_shard_entry_points_reject_bad_arguments(lib):
    # grpo_count_active / grpo_loss_finalize host checks
    assert lib.grpo_count_active(FAKE, -1, 4, FAKE, None) == 2
    assert lib.grpo_count_active(FAKE, 2, (1 << 30) + 1, FAKE, None) == 2
    assert lib.grpo_count_active(FAKE, 2, 4, None, None) == 1
    assert lib.grpo_count_active(None, 2, 4, FAKE, None) == 1
    assert lib.grpo_count_active(FAKE, 2, 4, FAKE + 4, None) == 4
    p = _params()
    assert lib.grpo_loss_finalize(FAKE, -1, FAKE, ctypes.byref(p), FAKE, None) == 2
    assert lib.grpo_loss_finalize(None, 4, FAKE, ctypes.byref(p), FAKE, None) == 1
    assert lib.grpo_loss_finalize(FAKE, 4, None, ctypes.byref(p), FAKE, None) == 1
    assert lib.grpo_loss_finalize(FAKE, 4, FAKE, ctypes.byref(p), None, None) == 1
    assert lib.grpo_loss_finalize(FAKE + 8, 4, FAKE, ctypes.byref(p), FAKE, None) == 4
    assert lib.grpo_loss_finalize(FAKE, 4, FAKE, ctypes.byref(_params(reduction=5)), FAKE,
                                  None) == 6


def _sharded(seq_begin, counts=FAKE, totals=FAKE):
    sh = g._Shard(seq_begin, counts, totals)
    p = _params()
    p._sh = sh
    p.shard = ctypes.pointer(sh)
    return p


def test_shard_placement_is_checked(lib):
    # a shard of 4 sequences of a batch of 8 (groups and rewards span the batch)
    gr = _groups(8)
    ws = g.grpo_workspace_size(8, 16)
    assert _fwd(lib, B=4, gr=gr, p=_sharded(5), ws_bytes=ws) == 2   # runs past the batch
    assert _fwd(lib, B=4, gr=gr, p=_sharded(-1), ws_bytes=ws) == 2
    assert _fwd(lib, B=4, gr=gr, p=_sharded(0, counts=None), ws_bytes=ws) == 1
    assert _fwd(lib, B=4, gr=gr, p=_sharded(0, totals=None), ws_bytes=ws) == 1
    assert _fwd(lib, B=4, gr=gr, p=_sharded(0, totals=FAKE + 8), ws_bytes=ws) == 4
    assert _fwd(lib, B=4, gr=gr, p=_sharded(0, counts=FAKE + 4), ws_bytes=ws) == 4
    # the workspace must cover the whole batch
    assert _fwd(lib, B=4, gr=gr, p=_sharded(0), ws_bytes=g.grpo_workspace_size(4, 16)) == 7


def test_vocab_entry_points_reject_bad_arguments(lib):
    C = lib.grpo_vocab_chunk()
    assert C > 0 and C % 64 == 0
    part = lambda **kw: lib.grpo_vocab_partials(
        kw.get("pol", FAKE), kw.get("ref", FAKE), kw.get("dt", 1), kw.get("B", 2), kw.get("T", 3),
        kw.get("Vk", 100), kw.get("v0", 0), kw.get("act", FAKE), kw.get("mask", FAKE),
        kw.get("pp", FAKE), kw.get("pr", FAKE), kw.get("al", FAKE), None)
    assert part(dt=9) == 3
    assert part(v0=C + 1) == 2        # a slice starts on a chunk boundary
    assert part(Vk=0) == 2
    assert part(pol=None) == 1
    assert part(pp=FAKE + 8) == 4
    assert part(act=FAKE + 4) == 4
    gr = _groups(8)
    p = _params()
    loss = lambda **kw: lib.grpo_vocab_loss(
        FAKE, FAKE, kw.get("nck", 1), FAKE, kw.get("V", 100), FAKE, FAKE, FAKE, 8, 16, FAKE,
        ctypes.byref(gr), ctypes.byref(kw.get("p", p)), kw.get("lse", FAKE), FAKE, None, None,
        None, FAKE, kw.get("ws_bytes", g.grpo_workspace_size(8, 16)), None)
    assert loss(nck=2) == 2           # chunk count must match V
    assert loss(lse=None) == 1
    assert loss(lse=FAKE + 4) == 4
    assert loss(p=_params(beta=-1.0)) == 6
    assert loss(ws_bytes=16) == 7
    grad = lambda **kw: lib.grpo_vocab_grad(FAKE, kw.get("dt", 1), 2, 3, 100, kw.get("v0", 0),
                                            FAKE, FAKE, kw.get("lse", FAKE), FAKE,
                                            kw.get("flags", 0), None)
    assert grad(dt=9) == 3
    assert grad(v0=-1) == 2
    assert grad(flags=1) == 6         # only GRPO_SKIP_MASKED_GRAD_ROWS
    assert grad(lse=None) == 1
