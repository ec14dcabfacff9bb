"""CPU models of the mbarrier protocols of the two tensor-core kernels.

Every role of a kernel (the TMA producer, the MMA warp, the softmax warp
groups) is a Python generator that yields the barrier phase it waits for and
performs the arrivals the kernel performs, in the kernel's order.  A random
scheduler interleaves the roles and delivers the asynchronous completions
(TMA loads in any order, tcgen05 commits in issue order) at random times.
Each run must finish without a deadlock, and no wait may see its barrier two
or more phases ahead of the phase it waits for (the kernels wait on the
phase's parity, so that would be aliasing).  The models mirror
`csrc/prefill_tc.cu` (work items of two query tiles, a 4-entry item ring, a
K/V ring of 4 or 8 stages) and `csrc/decode_tc.cu` (double-buffered S, lazy
O rescale waiting on the per-PV barrier); a change to a kernel's waits or
arrivals must be made here too.  Two planted mistakes check that the models
catch what they are for.
"""
from __future__ import annotations

import random

import pytest

RING = 4  # work items in flight between the prefill kernel's roles


class Bar:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, count=1):
        self.count, self.pending, self.phase = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending, self.phase = 0, self.phase + 1


class Hazard(Exception):
    pass


def wait(bar, phase):
    """Readiness test for completed phase number `phase` (0-based)."""
    def ready():
        if bar.phase >= phase + 2:
            raise Hazard(f"barrier at phase {bar.phase} while a role waits for phase {phase}")
        return bar.phase >= phase + 1
    return ready


class Sched:
    """Random interleaving of roles plus asynchronous completions."""

    def __init__(self, seed):
        self.rnd = random.Random(seed)
        self.tma = []     # pending TMA completions: any order
        self.commit = []  # pending tcgen05 commits: issue order

    def run(self, roles, limit=200000):
        waits = {n: None for n in roles}
        done = set()
        for _ in range(limit):
            if len(done) == len(roles) and not self.tma and not self.commit:
                return None
            choices = [n for n in roles if n not in done and (waits[n] is None or waits[n]())]
            if self.tma:
                choices.append("tma")
            if self.commit:
                choices.append("commit")
            if not choices:
                return "deadlock: " + ", ".join(n for n in roles if n not in done)
            n = self.rnd.choice(choices)
            if n == "tma":
                self.tma.pop(self.rnd.randrange(len(self.tma))).arrive()
            elif n == "commit":
                self.commit.pop(0).arrive()
            else:
                try:
                    waits[n] = next(roles[n])
                except StopIteration:
                    done.add(n)
        return "step limit"


# ----------------------------------------------------------------------------- prefill

def prefill_run(items, stages, seed, mistake=None):
    """items: (n_kv0, n_kv1, N) per work item, N = max(n_kv0, n_kv1)."""
    sc = Sched(seed)
    item_full = [Bar() for _ in range(RING)]
    item_empty = [Bar(3) for _ in range(RING)]  # MMA warp + two softmax groups
    q_full, q_empty = [Bar(), Bar()], [Bar(), Bar()]
    kv_full, kv_empty = [Bar() for _ in range(stages)], [Bar() for _ in range(stages)]
    s_full, p_ready, o_full = [Bar(), Bar()], [Bar(), Bar()], [Bar(), Bar()]
    ring = [None] * RING
    stream = list(items) + [(0, 0, -1)]  # the draw past the end

    def producer():
        q_uses, issued = [0, 0], 0
        for k, it in enumerate(stream):
            slot = k % RING
            if k >= RING:
                yield wait(item_empty[slot], k // RING - 1)
            ring[slot] = it
            item_full[slot].arrive()
            if it[2] < 0:
                return

            def load_q(x):
                if it[x] == 0:
                    return
                if q_uses[x] > 0:
                    yield wait(q_empty[x], q_uses[x] - 1)
                sc.tma.append(q_full[x])
                q_uses[x] += 1

            def load_kv():
                nonlocal issued
                s = issued % stages
                if issued >= stages and mistake != "no_kv_empty_wait":
                    yield wait(kv_empty[s], issued // stages - 1)
                sc.tma.append(kv_full[s])
                issued += 1

            yield from load_q(0)
            for j in range(it[2]):
                yield from load_kv()
                if j == 0:
                    yield from load_q(1)
                yield from load_kv()

    def mma():
        consumed, q_uses, pr = 0, [0, 0], [0, 0]
        for k in range(len(stream)):
            yield wait(item_full[k % RING], k // RING)
            n0, n1, N = ring[k % RING]
            item_empty[k % RING].arrive()
            if N < 0:
                return
            if N == 0:
                continue
            kslot, have_k = 0, False
            for x, n in enumerate((n0, n1)):
                if n == 0:
                    continue
                yield wait(q_full[x], q_uses[x])
                q_uses[x] += 1
                if not have_k:
                    kslot = consumed % stages
                    yield wait(kv_full[kslot], consumed // stages)
                    consumed += 1
                    have_k = True
                sc.commit.append(s_full[x])
                if n == 1:
                    sc.commit.append(q_empty[x])
            sc.commit.append(kv_empty[kslot])
            for j in range(N):
                vslot = consumed % stages
                yield wait(kv_full[vslot], consumed // stages)
                consumed += 1
                if j < n0:
                    yield wait(p_ready[0], pr[0])
                    pr[0] += 1
                    if j == n0 - 1:
                        sc.commit.append(o_full[0])
                nxt = j + 1 < N
                nslot = 0
                if nxt:
                    nslot = consumed % stages
                    yield wait(kv_full[nslot], consumed // stages)
                    consumed += 1
                    if j + 1 < n0:
                        sc.commit.append(s_full[0])
                        if j + 2 == n0:
                            sc.commit.append(q_empty[0])
                if j < n1:
                    yield wait(p_ready[1], pr[1])
                    pr[1] += 1
                    if j == n1 - 1:
                        sc.commit.append(o_full[1])
                sc.commit.append(kv_empty[vslot])
                if nxt:
                    if j + 1 < n1:
                        sc.commit.append(s_full[1])
                        if j + 2 == n1:
                            sc.commit.append(q_empty[1])
                    sc.commit.append(kv_empty[nslot])

    def softmax(x):
        sp, o_uses = 0, 0
        for k in range(len(stream)):
            slot = k % RING
            yield wait(item_full[slot], k // RING)
            it = ring[slot]
            if it[2] < 0:
                item_empty[slot].arrive()
                return
            for _ in range(it[x]):
                yield wait(s_full[x], sp)
                sp += 1
                p_ready[x].arrive()
            if it[x] > 0:
                yield wait(o_full[x], o_uses)
                o_uses += 1
            assert ring[slot] is it, "item ring slot overwritten before it was released"
            if mistake != "no_item_release" or x == 0:
                item_empty[slot].arrive()

    return sc.run({"producer": producer(), "mma": mma(), "softmax0": softmax(0), "softmax1": softmax(1)})


def random_items(rnd, n_max=24, steps_max=9):
    out = []
    for _ in range(rnd.randint(1, n_max)):
        kind = rnd.random()
        N = rnd.randint(1, steps_max)
        if kind < 0.2:
            out.append((0, 0, 0))                        # every row padded
        elif kind < 0.55:
            out.append((N - 1, N, N) if N > 1 else (1, 1, 1))  # causal pair of consecutive tiles
        elif kind < 0.75:
            out.append((N, N, N))                        # same tile of two heads (grouped query)
        elif kind < 0.85:
            out.append((N, 0, N))                        # second tile past the end
        else:
            a = rnd.randint(1, N)                        # key padding cuts one tile short
            out.append((a, N, N) if rnd.random() < 0.5 else (N, a, N))
    if rnd.random() < 0.5:                               # a run of fully padded items
        i = rnd.randint(0, len(out))
        out[i:i] = [(0, 0, 0)] * rnd.randint(3, 9)
    return out


def _prefill_trials(stages, mistake=None, trials=150):
    rnd = random.Random(stages * 7 + (mistake is not None))
    failures = []
    for t in range(trials):
        items = random_items(rnd)
        for seed in range(2):
            try:
                r = prefill_run(items, stages, seed + 10 * t, mistake)
            except (Hazard, AssertionError) as e:
                r = f"{type(e).__name__}: {e}"
            if r:
                failures.append((t, seed, r, items))
    return failures


@pytest.mark.parametrize("stages", [4, 8])  # the K/V ring at D = 128 and D = 64
def test_prefill_protocol_has_no_deadlock_or_aliasing(stages):
    failures = _prefill_trials(stages)
    assert not failures, failures[:3]


@pytest.mark.parametrize("mistake", ["no_kv_empty_wait", "no_item_release"])
def test_prefill_model_catches_planted_mistakes(mistake):
    assert _prefill_trials(4, mistake, trials=60), f"the model missed '{mistake}'"


# ----------------------------------------------------------------------------- decode (tensor cores)

def decode_run(n, stages, seed, p_rescale, mistake=None):
    """One chunk of n 64-key tiles: S double-buffered, O rescaled lazily."""
    sc = Sched(seed)
    q_full = Bar()
    kv_full, kv_empty = [Bar() for _ in range(stages)], [Bar() for _ in range(stages)]
    s_full, p_ready = [Bar(), Bar()], [Bar(), Bar()]
    o_done, o_full = Bar(), Bar()

    def producer():
        sc.tma.append(q_full)
        for issued in range(2 * n):
            s = issued % stages
            if issued >= stages:
                yield wait(kv_empty[s], issued // stages - 1)
            sc.tma.append(kv_full[s])

    def mma():
        yield wait(q_full, 0)
        pr = [0, 0]
        for j in range(n + 1):
            if j < n:  # S_j into buffer j & 1, issued before PV_{j-1}
                ks = (2 * j) % stages
                yield wait(kv_full[ks], (2 * j) // stages)
                sc.commit.append(s_full[j & 1])
                sc.commit.append(kv_empty[ks])
            if j >= 1:
                t = j - 1
                x, vs = t & 1, (2 * t + 1) % stages
                yield wait(p_ready[x], pr[x])
                pr[x] += 1
                yield wait(kv_full[vs], (2 * t + 1) // stages)
                if mistake != "no_pv_signal":
                    sc.commit.append(o_done)
                sc.commit.append(kv_empty[vs])
                if t == n - 1:
                    sc.commit.append(o_full)

    def softmax():
        rnd = random.Random(seed + 1)
        sp = [0, 0]
        for j in range(n):
            x = j & 1
            yield wait(s_full[x], sp[x])
            sp[x] += 1
            if j > 0 and rnd.random() < p_rescale:  # O holds PV_0 .. PV_{j-1}
                yield wait(o_done, j - 1)
            p_ready[x].arrive()
        yield wait(o_full, 0)

    return sc.run({"producer": producer(), "mma": mma(), "softmax": softmax()})


def _decode_trials(mistake=None):
    failures = []
    for stages in (4, 6):
        for n in range(1, 24):
            for seed in range(6):
                for p in (0.0, 0.3, 1.0):
                    try:
                        r = decode_run(n, stages, seed * 31 + n, p, mistake)
                    except Hazard as e:
                        r = f"Hazard: {e}"
                    if r:
                        failures.append((stages, n, seed, p, r))
    return failures


def test_decode_tc_protocol_has_no_deadlock_or_aliasing():
    failures = _decode_trials()
    assert not failures, failures[:3]


def test_decode_tc_model_catches_a_planted_mistake():
    assert _decode_trials("no_pv_signal"), "the model missed a PV group that never signals"
