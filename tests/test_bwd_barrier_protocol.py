"""A model of the mbarrier protocol of the D = 128 backward kernel
(fa_bwd_kernel in csrc/fa_bwd.cu): every role's waits (barrier, logical
phase) and arrivals in program order, run under random interleavings with
asynchronous completions (TMA loads, tcgen05 commits) landing in any order.
It fails on a deadlock, and on a wait that finds its barrier two or more
phases past the one it means: a parity wait cannot tell those apart. The
model must be kept in step with the kernel; the second test shows that it
catches a single hand-off barrier shared by all ring stages."""
import random

import pytest

STAGES = 4


class _Bar:
    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1  # every barrier of the model completes on one arrival


def _roles(n, single_stage_handoff=False):
    W = lambda name, k: ("wait", name, k)  # noqa: E731
    A = lambda name: ("arrive", name)      # noqa: E731
    L = lambda name: ("async", name)       # noqa: E731
    ready = (lambda st, j: ("StageReady0", j)) if single_stage_handoff else \
        (lambda st, j: (f"StageReady{st}", j // STAGES))

    def producer():
        for j in range(n):
            st, b = j % STAGES, j & 1
            if j >= STAGES:
                yield W(f"StageFree{st}", j // STAGES - 1)
            yield L(f"QFull{st}")
            if j >= 2:
                yield W(f"PFull{b}", (j - 2) >> 1)
            yield L(f"LFull{b}")

    def s_issuer():  # warp 1: S^T and dP^T
        for j in range(n):
            st, b = j % STAGES, j & 1
            yield W(f"QFull{st}", j // STAGES)
            if j >= 2:
                yield W(f"PTFree{b}", (j - 2) >> 1)
                yield W(f"BufFree{b}", (j - 2) >> 1)
            yield L(f"SFull{b}")

    def product_issuer():  # warp 3: dQ^T, dV, dK
        for j in range(n):
            st, b = j % STAGES, j & 1
            yield W(f"PFull{b}", j >> 1)
            for name in (f"DQFull{b}", f"PTFree{b}", f"QEmpty{st}", f"DSFree{b}"):
                yield L(name)

    def key_rows():  # warps 4..11
        for j in range(n):
            b = j & 1
            yield W(f"LFull{b}", j >> 1)
            yield W(f"SFull{b}", j >> 1)
            if j >= 2:
                yield W(f"DSFree{b}", (j - 2) >> 1)
            yield A(f"PFull{b}")
        if n:
            yield W(f"DSFree{(n - 1) & 1}", (n - 1) >> 1)

    def dq_warps():  # warps 12..15
        for j in range(n):
            st, b = j % STAGES, j & 1
            yield W(f"DQFull{b}", j >> 1)
            yield A(f"BufFree{b}")
            yield W(f"QEmpty{st}", j // STAGES)
            yield A(ready(st, j)[0])

    def reducer():  # warp 2
        for j in range(n):
            st = j % STAGES
            yield W(*ready(st, j))
            yield L(f"StageFree{st}")

    return [producer(), s_issuer(), product_issuer(), key_rows(), dq_warps(), reducer()]


def simulate(n, seed, **kw):
    rnd = random.Random(seed)
    bars = {}
    bar = lambda name: bars.setdefault(name, _Bar())  # noqa: E731
    roles = _roles(n, **kw)
    cur = [next(r, None) for r in roles]
    in_flight = []
    while True:
        runnable = []
        for i, op in enumerate(cur):
            if op is None:
                continue
            if op[0] == "wait":
                ph = bar(op[1]).phase
                if ph >= op[2] + 2:
                    return f"alias: {op[1]} wanted phase {op[2]}, barrier at {ph}"
                if ph >= op[2] + 1:
                    runnable.append(i)
            else:
                runnable.append(i)
        if in_flight:
            runnable.append(-1)
        if not runnable:
            return "ok" if all(op is None for op in cur) else f"deadlock: {[op for op in cur if op]}"
        i = rnd.choice(runnable)
        if i < 0:
            bar(in_flight.pop(rnd.randrange(len(in_flight)))).arrive()
            continue
        op = cur[i]
        if op[0] == "arrive":
            bar(op[1]).arrive()
        elif op[0] == "async":
            in_flight.append(op[1])
        cur[i] = next(roles[i], None)


@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 6, 9, 17, 64])
def test_protocol_has_no_deadlock_or_phase_aliasing(n):
    for seed in range(200):
        assert simulate(n, seed) == "ok", (n, seed)


def test_model_catches_a_shared_handoff_barrier():
    results = {simulate(n, seed, single_stage_handoff=True) for n in (5, 9) for seed in range(200)}
    assert any(r.startswith("alias") for r in results)
