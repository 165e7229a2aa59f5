"""The in-tree build takes turns across processes (one per rank under
torchrun): concurrent build() calls on a stale library compile it once, the
others wait on the lock and return the fresh library; forced rebuilds never
overlap.  Compilation is replaced by a fake that records when it ran."""

import multiprocessing as mp
import os
import time

import pytest


def _rank(tmp, force, barrier):
    from hierarchical_speculative_decoding_gb300 import build as B

    marker = os.path.join(tmp, "fresh")
    B.BUILD = tmp
    B.LOCK = os.path.join(tmp, ".build.lock")
    B.up_to_date = lambda debug=False: os.path.exists(marker)

    def fake_compile(verbose, extra, debug=False):
        t0 = time.time()
        time.sleep(0.5)
        with open(os.path.join(tmp, "log"), "a") as f:
            f.write(f"{os.getpid()} {t0} {time.time()}\n")
        open(marker, "w").close()
        return B.LIB

    B._compile_and_link = fake_compile
    barrier.wait()
    assert B.build(force=force) == B.LIB


@pytest.mark.parametrize("force", [False, True])
def test_concurrent_builds_take_turns(tmp_path, force):
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(2)
    procs = [ctx.Process(target=_rank, args=(str(tmp_path), force, barrier)) for _ in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs)
    runs = sorted(tuple(float(x) for x in line.split()[1:]) for line in open(tmp_path / "log"))
    if force:
        assert len(runs) == 2
        assert runs[0][1] <= runs[1][0], "two builds overlapped"
    else:
        assert len(runs) == 1, "the waiting process compiled again"
