"""Multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own batch (weak scaling, no collective on the data
path); the only collective is the max over ranks of the step times."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        wl = bench.make_workload("tiny", r)
        step, e2e, dec = [1.0 + r, 5.0 - r, 0.5 * (r + 1)]
        mx = bench.reduce_max([step, e2e, dec], w)
        q.put((r, mx, wl.q.tobytes(), wl.context_lens.tolist(), w, local))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_and_own_batches():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for r, mx, _, _, w, local in out:
        assert w == world and local == r
        assert mx == [2.0, 5.0, 1.0]          # max over ranks of each time
    # each rank generates its own batch of the same shape
    assert out[0][2] != out[1][2]
    assert len(out[0][3]) == len(out[1][3])


def test_weak_value_and_single_rank_identity():
    assert bench.reduce_max([1.0, 2.0], 1) == [1.0, 2.0]
    # two ranks each moving 1 GB in a 0.5 s (slowest) step: 4 GB/s job-wide
    assert np.isclose(bench.weak_value(1e9, 2, 500.0), 4.0)


def test_source_digest_ignores_comments_only():
    """The recorded ncu traffic stays valid across comment edits and is
    dropped as soon as the code itself changes."""
    src = ('// header\nint f(int x) { /* why */ return x + 1; }\n'
           'const char* s = "a // not a comment /* nor this */";\n'
           "char c = '\\'';  // trailing\n")
    recommented = ('int f(int x) {\n    return x + 1;  // reason\n}\n'
                   'const char* s = "a // not a comment /* nor this */";\n'
                   "char c = '\\'';\n")
    changed = src.replace("x + 1", "x + 2")
    assert bench.strip_comments(src) == bench.strip_comments(recommented)
    assert bench.strip_comments(src) != bench.strip_comments(changed)
    assert "/* nor this */" in bench.strip_comments(src)
    assert "why" not in bench.strip_comments(src)


def test_profiled_traffic_matches_current_sources():
    """The committed decode profile was taken on the decode code as it is;
    if not, the bench reports roofline.traffic as null, and this says so."""
    import pytest
    if bench.profiled_traffic("llama7b_batch64") is None:
        pytest.skip("decode code changed since the committed ncu capture: traffic reads null")
