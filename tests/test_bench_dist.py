"""The multi-process path of bench.py on CPU: two gloo ranks rendezvous
through the environment (as torchrun sets it), time-aggregate with the
max over ranks, and form the whole-job throughput of two replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    import torch.distributed as dist
    import bench
    ws, r, local = bench.dist_setup()
    assert (ws, r) == (2, rank) and dist.get_backend() == "gloo"
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, ws, "cpu")  # per-rank step times (ms)
    bench.barrier(ws)
    q.put((rank, slowest, bench.aggregate_value(1000, 4, ws, slowest)))
    dist.destroy_process_group()


def test_two_rank_harness_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 15.0  # both ranks see the slower rank's time
        assert value == pytest.approx(1000 * 4 * 2 / 0.015)  # two replicas' tokens / max time


def test_active_runs_cover_exactly_the_active_slots():
    # the end-to-end step copies these runs of logits rows; together they must
    # be exactly the active slots, in order, without overlap
    import numpy as np
    import bench
    rng = np.random.default_rng(5)
    for B, T, p in [(4, 7, 0.5), (16, 64, 0.9), (3, 5, 0.0), (3, 5, 1.0), (1, 1, 1.0)]:
        mask = (rng.random((B, T)) < p).astype(np.uint8) * rng.integers(1, 255, (B, T))
        runs = bench.active_runs(mask.astype(np.uint8))
        cover = np.zeros(B * T, dtype=bool)
        last = -1
        for b, e in runs:
            assert last < b < e <= B * T  # ordered, nonempty, separated
            cover[b:e] = True
            last = e
        assert np.array_equal(cover, mask.reshape(-1) != 0)


def test_committed_profiles_name_their_own_key():
    # every profile bench.py may take a traffic figure from exists and names
    # the key it is filed under; masked-row and vocabulary-parallel lines never
    # borrow the fused path's figure
    import os
    import re
    import bench
    import synth
    for key, (name, files) in bench.PROFILES.items():
        text = open(os.path.join(bench.ROOT, "profiles", name)).read()
        assert re.search(r"^workload:\s*([\w/]+)", text, re.M).group(1) == key
        assert re.search(r"^traffic_bytes_per_launch:\s*[0-9.eE+]+", text, re.M)
        assert re.search(r"^kernel_source_sha:\s*\w+", text, re.M)
    w = synth.WORKLOADS["large_vocab"]
    default = bench.PROFILES[bench.profile_key(w)][0]
    for key in (bench.profile_key(w, skip_masked=True), bench.profile_key(w, tp=2),
                bench.profile_key(w, tp=4)):
        assert key != "large_vocab"
        assert key not in bench.PROFILES or bench.PROFILES[key][0] != default
    assert bench.profile_key(w, "k2") == "large_vocab"
    assert bench.profile_key(synth.WORKLOADS["logps"], "k2") not in bench.PROFILES


def test_source_hash_ignores_comments_only():
    # a profile's traffic figure outlives a comment edit but not a code edit
    import bench
    code = 'int f(int x) {  // doubles\n  /* a\n block */ return 2 * x;\n}\n\nconst char* s = "a//b";\n'
    same = 'int f(int x) {\n  return 2 * x;  // twice x\n}\nconst char* s = "a//b";\n'
    assert bench._code_only(code) == bench._code_only(same)
    for changed in (code.replace("2 * x", "3 * x"), code.replace('"a//b"', '"a/b"'),
                    code.replace('"a//b"', '"a  //b"')):
        assert bench._code_only(changed) != bench._code_only(code)
