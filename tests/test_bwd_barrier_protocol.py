"""A model of the mbarrier protocol of the D = 128 backward kernel
(fa_bwd_kernel in csrc/fa_bwd.cuh): every role's waits (barrier, logical
phase) and arrivals in program order, run under random interleavings with
asynchronous completions (TMA loads, tcgen05 commits) landing in any order.

The kernel is persistent: a CTA takes work units (key tiles) one after the
other. Warp 0 fetches each unit and publishes it in a ring of unit slots
that every role reads and releases. Ring stages and buffers keep their
phases across units through one running sub-step count J. K/V of the next
unit are loaded once the current unit's last products are done (KVEmpty).
The dV/dK accumulators in TMEM need no barrier of their own: the key-row
warps read a unit's accumulators out before they publish the next unit's
first P^T, and the next unit's first dV/dK products wait for that P^T; the
model checks that this order holds. A unit with no sub-steps (no query sees
its keys) only has its zero dK/dV written.

The model fails on a deadlock, and on a wait that finds its barrier two or
more phases past the one it means: a parity wait cannot tell those apart.
It must be kept in step with the kernel; the last tests show that it
catches a single hand-off barrier shared by all ring stages and a unit slot
rewritten before every role has read it."""
import random

import pytest

STAGES = 4
RING = 4  # unit slots


class _Bar:
    def __init__(self, count=1):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


CONSUMERS = 5  # roles that read every unit slot (the kernel: 15 warps)


def _wait(name, k):
    return ("wait", name, k)


def _arrive(name):
    return ("arrive", name)


def _async(name):
    return ("async", name)


def _roles(units, single_stage_handoff=False, no_slot_release_wait=False):
    ready = (lambda st, J: ("StageReady0", J)) if single_stage_handoff else \
        (lambda st, J: (f"StageReady{st}", J // STAGES))

    def unit_slot(i):
        s = i % RING
        return f"UnitReady{s}", f"UnitFree{s}", i // RING

    def take(i):  # a consumer reads unit slot i and releases it
        rdy, free, k = unit_slot(i)
        yield _wait(rdy, k)
        yield ("read", i % RING, i)
        yield _arrive(free)

    def producer():  # warp 0
        J = wi = 0
        for i, n in enumerate(list(units) + [None]):  # None: the stop entry
            rdy, free, k = unit_slot(i)
            if i >= RING and not no_slot_release_wait:
                yield _wait(free, k - 1)
            yield ("write", i % RING, i)
            yield _arrive(rdy)
            if not n:
                continue
            if wi >= 1:
                yield _wait("KVEmpty", wi - 1)
            yield _async("KVFull")
            for _ in range(n):
                st, b = J % STAGES, J & 1
                # Q and dO halves of the stage: each refilled once the dQ
                # boxes staged over it have been read
                if J >= STAGES:
                    yield _wait(f"StageFreeQ{st}", J // STAGES - 1)
                yield _async(f"QFull{st}")
                if J >= STAGES:
                    yield _wait(f"StageFree{st}", J // STAGES - 1)
                yield _async(f"DOFull{st}")
                if J >= 2:
                    yield _wait(f"PFull{b}", (J - 2) >> 1)
                yield _async(f"LFull{b}")
                J += 1
            wi += 1

    def s_issuer():  # warp 1: S^T and dP^T
        J = wi = 0
        for i, n in enumerate(units):
            yield from take(i)
            if not n:
                continue
            yield _wait("KVFull", wi)
            for _ in range(n):
                st, b = J % STAGES, J & 1
                yield _wait(f"QFull{st}", J // STAGES)
                if J >= 2:
                    yield _wait(f"PTFree{b}", (J - 2) >> 1)
                yield _async(f"SFull{b}")  # S^T
                yield _wait(f"DOFull{st}", J // STAGES)  # dO
                if J >= 2:
                    yield _wait(f"BufFree{b}", (J - 2) >> 1)
                yield _async(f"DPFull{b}")  # dP^T
                J += 1
            wi += 1
        yield _wait(*unit_slot(len(units))[0::2])

    def product_issuer():  # warp 3: dV once P^T is in, then dQ^T and dK once dS^T is
        J = wi = 0
        for i, n in enumerate(units):
            yield from take(i)
            if not n:
                continue
            for j in range(n):
                st, b = J % STAGES, J & 1
                yield _wait(f"PTFull{b}", J >> 1)
                yield _wait(f"DOFull{st}", J // STAGES)  # dV reads dO
                if j == 0:
                    yield ("products", wi)  # overwrite the accumulators of unit wi
                yield _async(f"PTFree{b}")
                yield _wait(f"PFull{b}", J >> 1)
                for name in (f"DQFull{b}", f"QEmpty{st}", f"DSFree{b}"):
                    yield _async(name)
                J += 1
            yield _async("KVEmpty")
            wi += 1
        yield _wait(*unit_slot(len(units))[0::2])

    def key_rows():  # warps 4..11 (one role: the StagingFree barrier orders them among themselves)
        J = wi = 0
        for i, n in enumerate(units):
            yield from take(i)
            for j in range(n):
                b = J & 1
                yield _wait(f"LFull{b}", J >> 1)
                yield _wait(f"SFull{b}", J >> 1)
                yield _arrive(f"PTFull{b}")  # P^T in TMEM: dV may start
                yield _wait(f"DPFull{b}", J >> 1)
                if J >= 2:
                    yield _wait(f"DSFree{b}", (J - 2) >> 1)
                if j == 0 and i > 0:
                    yield _wait("StagingFree", i - 1)  # dS^T overwrites the staging blocks
                yield _arrive(f"PFull{b}")
                J += 1
            if n:
                yield _wait(f"DSFree{(J - 1) & 1}", (J - 1) >> 1)
                yield ("readout", wi)  # the unit's dV and dK read out of TMEM
                wi += 1
            yield _arrive("StagingFree")  # dK and dV written out of the staging blocks
        yield _wait(*unit_slot(len(units))[0::2])

    def dq_warps():  # warps 12..15
        J = 0
        for i, n in enumerate(units):
            yield from take(i)
            for _ in range(n or 0):
                st, b = J % STAGES, J & 1
                yield _wait(f"DQFull{b}", J >> 1)
                yield _arrive(f"BufFree{b}")
                yield _wait(f"QEmpty{st}", J // STAGES)
                yield _arrive(ready(st, J)[0])
                J += 1
        yield _wait(*unit_slot(len(units))[0::2])

    def reducer():  # warp 2
        J = 0
        for i, n in enumerate(units):
            yield from take(i)
            for _ in range(n or 0):
                st = J % STAGES
                yield _wait(*ready(st, J))
                yield _async(f"StageFreeQ{st}")  # the boxes over Q read
                yield _async(f"StageFree{st}")   # the boxes over dO read
                J += 1
        yield _wait(*unit_slot(len(units))[0::2])

    return [producer(), s_issuer(), product_issuer(), key_rows(), dq_warps(), reducer()]


def simulate(units, seed, **kw):
    if isinstance(units, int):
        units = [units]
    rnd = random.Random(seed)
    bars = {}

    def bar(name):
        if name not in bars:
            bars[name] = _Bar(CONSUMERS if name.startswith("UnitFree") else 1)
        return bars[name]

    roles = _roles(units, **kw)
    cur = [next(r, None) for r in roles]
    in_flight = []
    slots = {}
    read_out = -1  # the last unit whose accumulators the key-row warps have read out
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
        if op[0] == "write":
            slots[op[1]] = op[2]
        elif op[0] == "read":
            if slots.get(op[1]) != op[2]:
                return f"overwrite: unit slot {op[1]} held {slots.get(op[1])} when unit {op[2]} was read"
        elif op[0] == "arrive":
            bar(op[1]).arrive()
        elif op[0] == "async":
            in_flight.append(op[1])
        elif op[0] == "readout":
            read_out = op[1]
        elif op[0] == "products" and op[1] >= 1 and read_out < op[1] - 1:
            return f"overwrite: unit {op[1]}'s products before unit {op[1] - 1}'s accumulators were read"
        cur[i] = next(roles[i], None)


@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 6, 9, 17, 64])
def test_one_unit_has_no_deadlock_or_phase_aliasing(n):
    for seed in range(200):
        assert simulate(n, seed) == "ok", (n, seed)


@pytest.mark.parametrize("case", range(12))
def test_unit_sequences_have_no_deadlock_aliasing_or_overwrite(case):
    rnd = random.Random(case)
    for seed in range(120):
        units = [rnd.choice([0, 1, 1, 2, 3, 5, 9, 17]) for _ in range(rnd.randrange(1, 10))]
        assert simulate(units, seed) == "ok", (units, seed)


def test_model_catches_a_shared_handoff_barrier():
    results = {simulate(n, seed, single_stage_handoff=True) for n in (5, 9) for seed in range(200)}
    assert any(r.startswith("alias") for r in results)


def test_model_catches_a_unit_slot_rewritten_before_it_was_read():
    results = {simulate([1, 0, 0, 1, 0, 0, 1, 0, 1], seed, no_slot_release_wait=True).split(":")[0]
               for seed in range(300)}
    assert results & {"overwrite", "alias"}

