import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of host time)")


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _ensure_built():
    """Build the host-side libraries the CPU tests need if missing or stale
    (the full build, CUDA included, is __graft_entry__.build())."""
    import oracle
    import synth
    jobs = []
    if _stale(oracle._SO, [os.path.join(ROOT, "oracle", "oracle.c")]):
        jobs += oracle.build_commands()
    if _stale(synth._HOST_SO, [os.path.join(ROOT, "synth", f) for f in
                               ("synth_host.c", "synth_core.h")]):
        jobs.append(synth.build_commands()[0])
    procs = [subprocess.Popen(c) for c in jobs]
    for p, c in zip(procs, jobs):
        if p.wait() != 0:
            raise RuntimeError("build failed: " + " ".join(c))


_ensure_built()
