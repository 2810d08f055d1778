"""A CPU model of the tree-attention kernel's synchronisation, run over random
schedules, with and without a role giving up part-way: it must never
deadlock, every mbarrier parity wait must be sound, no named-barrier round may
take more arrivals than its count, and no load may land in a buffer that a
queued MMA has still to read.

The model mirrors the roles of one CTA of the tensor-core tree pass:
- the TMA producer (Q tiles, then K and V tiles of a ring of slots);
- the MMA warp: per key tile j and row tile t it syncs on the named barrier of
  round j of row tile t, then issues PV_t(j) and S_t(j+1) (which overwrites
  P_t(j) only after PV_t(j) read it) and the commits;
- the V-tile warp(s): each V tile is handed on (vready) once it has landed
  (and, under F8, once both warps widened their halves); each segment's
  poison mask is published on win_bar;
- warp 3, which vouches in row tile 0's round j that V(j) is ready and K(j+1)
  has landed (a blocking participant of those rounds);
- the two softmax groups, which arrive (without blocking) on their row tile's
  named barrier once P_t(j) is stored;
plus the asynchronous engines: TMA copies land after random delays and the
tensor core runs the issuer's MMAs and commits in order.

An mbarrier counts completed phases. Every arrival names the phase it belongs
to, and the model checks it against the barrier's current phase. A parity wait
passes when the current phase's parity differs from the one named; the model
checks at every evaluation that the waiter is at most one phase behind, the
condition under which the hardware's answer is the intended one.

A named barrier counts arrivals in its current round; a sync arrives and blocks
until the round it arrived in completes. Unlike an mbarrier wait it has no time
limit, so the model fails if a role is left blocked in one. Rounds j and j+1
of a row tile use different barriers.

Giving up: with ``abort_at`` set, the role so named times out at its n-th
mbarrier wait. It sets the abort flag, after which every mbarrier wait of every
role returns "gave up" instead of blocking; each role then leaves as the kernel
does (one more arrival for the round it has not joined, where it takes part in
named barriers; the MMA warp and warp 3 also look at the flag after every
round they sync).

Mutants the model has to catch: V-tile warps that wait on a barrier shared by
K and V loads (only for the V phases, or for every phase in order), a V slot
released after the first row tile's PV instead of the last, the Q tiles
released after a segment's second S instead of its last, (FP8) vready and
win_bar left at count 1 for the two V warps, one named barrier per row tile
instead of two, a softmax group or the MMA warp leaving without its last
arrival, and an MMA warp that does not look at the abort flag after a round.
"""
import collections
import random

import pytest


class ProtocolError(AssertionError):
    pass


class _Bar:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, name, count):
        self.name, self.count, self.pend, self.done = name, count, 0, 0

    def arrive(self, phase, k=1):
        if phase != self.done:
            raise ProtocolError(f"{self.name}: arrival for phase {phase} while in phase {self.done}")
        self.pend += k
        if self.pend > self.count:
            raise ProtocolError(f"{self.name}: too many arrivals")
        if self.pend == self.count:
            self.pend = 0
            self.done += 1

    def passes(self, phase):
        if self.done > phase + 1:
            raise ProtocolError(f"{self.name}: waiter of phase {phase} two phases behind ({self.done} done)")
        return (self.done & 1) != (phase & 1)


class _Named:
    """A named (hardware) barrier: `count` thread arrivals complete a round."""

    def __init__(self, name, count):
        self.name, self.count, self.pend, self.rounds = name, count, 0, 0

    def arrive(self, k):
        """Returns the index of the round the arrival joined."""
        r = self.rounds
        self.pend += k
        if self.pend > self.count:
            raise ProtocolError(f"{self.name}: more than {self.count} arrivals in one round")
        if self.pend == self.count:
            self.pend = 0
            self.rounds += 1
        return r


def _kind_index(use, slots):
    """Phase index of `use` on its slot's K (even uses) or V (odd uses)
    barrier: with an even ring a slot holds one kind, with an odd ring the
    kinds alternate by round."""
    rnd = use // slots
    return rnd if slots % 2 == 0 else rnd >> 1


def _simulate(segs, slots, seed, mutant=None, slow_v_warp=False, max_steps=800000, f8=False, abort_at=None):
    """segs: (key tiles, row tiles present) per segment. abort_at: (role,
    n): that role's n-th mbarrier wait times out. Returns None when every
    role finishes, else the roles left blocked; raises ProtocolError on an
    unsound step."""
    rng = random.Random(seed)
    bars, named = {}, {}
    shared = mutant in ("shared_v_only", "shared_all")
    state = {"abort": False}
    checking_reads = abort_at is None

    def bar(name, count=1):
        bars[name] = _Bar(name, count)

    for s in range(slots):
        for n in ("full", "kfull", "vfull", "empty"):
            bar(f"{n}{s}")
        bar(f"vready{s}", 2 if f8 and mutant != "f8_count1" else 1)
    for t in range(2):
        bar(f"s_full{t}"), bar(f"o_fin{t}"), bar(f"o_free{t}", 128)
    bar("q_full"), bar("q_empty"), bar("drain"), bar("win_bar", 2 if f8 and mutant != "f8_count1" else 1)
    p_count = (192, 160)
    for t in range(2):
        for k in range(2):
            named[(t, k)] = _Named(f"P{t}.{k}", p_count[t])

    def p_bar(t, r):
        return named[(t, 0 if mutant == "single_pbar" else r & 1)]

    tma = []                         # [delay, barrier, phase]
    tensor_q = []                    # the issuer's MMAs and commits, run in order
    reads = collections.Counter()    # buffers that queued MMAs have still to read
    widened = collections.Counter()  # F8: V use -> halves widened

    def mma_op(*bufs):
        for b in bufs:
            reads[b] += 1
        tensor_q.append(("op", bufs))

    def commit(name, phase):
        tensor_q.append(("commit", name, phase))

    def overwrite(buf):
        # a load may land in a buffer only once every MMA that reads its old contents has run
        if checking_reads and reads[buf]:
            raise ProtocolError(f"{buf} overwritten while an MMA still has to read it")

    def load_done(use):
        if shared:
            return f"full{use % slots}", use // slots
        return f"{'v' if use & 1 else 'k'}full{use % slots}", _kind_index(use, slots)

    def producer():
        use = 0
        for segc, (nkt, _) in enumerate(segs):
            if not (yield ("wait", "q_empty", segc - 1)):
                return
            overwrite(("q", segc - 1))
            tma.append([rng.randint(1, 30), "q_full", segc])
            for _ in range(2 * nkt):
                if not (yield ("wait", f"empty{use % slots}", use // slots - 1)):
                    return
                overwrite(("kv", use - slots))
                tma.append([rng.randint(1, 30), *load_done(use)])
                use += 1

    def mma():
        use = 0
        tcnt, scnt = [0, 0], [0, 0]
        p0_rounds = 0
        ok = True
        for segc, (nkt, nt) in enumerate(segs):
            if not ((yield ("wait", "q_full", segc)) and (yield ("wait", *load_done(use)))):
                ok = False
                break
            for t in range(nt):
                mma_op(("q", segc), ("kv", use))
                commit(f"s_full{t}", tcnt[t])
            if nkt == 1:
                commit("q_empty", segc)
            commit(f"empty{use % slots}", use // slots)
            for j in range(nkt):
                vuse, kuse, more = use + 2 * j + 1, use + 2 * j + 2, j + 1 < nkt
                for t in range(nt):
                    yield ("nsync", p_bar(t, tcnt[t] + j), 32)
                    if t == 0:
                        p0_rounds += 1
                    aborted = state["abort"] and mutant != "mma_no_flag_check"
                    mma_op(("kv", vuse))
                    if more:
                        mma_op(("q", segc), ("kv", kuse))
                    v_release_at = 0 if mutant == "early_v_release" else nt - 1
                    if t == v_release_at:
                        commit(f"empty{vuse % slots}", vuse // slots)
                    if more:
                        commit(f"s_full{t}", tcnt[t] + j + 1)
                        if t == nt - 1:
                            q_release_at = 0 if mutant == "early_q_release" else nkt - 2
                            if j == q_release_at:
                                commit("q_empty", segc)
                            commit(f"empty{kuse % slots}", kuse // slots)
                    else:
                        commit(f"o_fin{t}", scnt[t])
                    if aborted:
                        ok = False
                        break
                if not ok:
                    break
            if not ok:
                break
            use += 2 * nkt
            for t in range(nt):
                tcnt[t] += nkt
                scnt[t] += 1
        if not ok and mutant != "mma_no_abort_arrive":
            p_bar(0, p0_rounds).arrive(32)
        commit("drain", 0)
        yield ("wait", "drain", 0)

    def v_warp(widener, voucher):
        use, prev_nt, scnt, rounds = 0, 0, [0, 0], 0
        ok = True
        for segc, (nkt, nt) in enumerate(segs):
            for j in range(nkt):
                kuse, vuse = use + 2 * j, use + 2 * j + 1
                if widener:
                    if mutant == "shared_v_only":
                        r = yield ("wait", f"full{vuse % slots}", vuse // slots)
                    elif mutant == "shared_all":
                        r = (yield ("wait", f"full{kuse % slots}", kuse // slots)) and \
                            (yield ("wait", f"full{vuse % slots}", vuse // slots))
                    else:
                        r = yield ("wait", f"vfull{vuse % slots}", _kind_index(vuse, slots))
                    if not r:
                        ok = False
                        break
                    if f8:
                        yield ("step",)
                        widened[vuse] += 1
                    bars[f"vready{vuse % slots}"].arrive(_kind_index(vuse, slots))
                    yield ("step",)
                if voucher:
                    r = (yield ("wait", f"vready{vuse % slots}", _kind_index(vuse, slots))) and \
                        (j + 1 == nkt or (yield ("wait", *load_done(vuse + 1))))
                    if not r:
                        ok = False
                        break
                    yield ("nsync", p_bar(0, rounds), 32)
                    rounds += 1
                    if state["abort"]:
                        ok = False
                        break
            if not ok:
                break
            if widener:
                for t in range(2):
                    if t < prev_nt and scnt[t] > 0 and not (yield ("wait", f"o_free{t}", scnt[t] - 1)):
                        ok = False
                if not ok:
                    break
                prev_nt = nt
                for t in range(nt):
                    scnt[t] += 1
                bars["win_bar"].arrive(segc)
            use += 2 * nkt
        if not ok and voucher and mutant != "voucher_no_abort_arrive":
            p_bar(0, rounds).arrive(32)

    def softmax_warp(t):
        tcnt = scnt = arrived = 0
        ok = True
        for segc, (nkt, nt) in enumerate(segs):
            if t >= nt:
                continue
            for j in range(nkt):
                if not (yield ("wait", f"s_full{t}", tcnt + j)):
                    ok = False
                    break
                yield ("step",)
                p_bar(t, arrived).arrive(32)
                arrived += 1
            if not ok:
                break
            if not ((yield ("wait", f"o_fin{t}", scnt)) and (yield ("wait", "win_bar", segc))):
                ok = False
                break
            yield ("step",)
            bars[f"o_free{t}"].arrive(scnt, 32)
            tcnt += nkt
            scnt += 1
        if not ok and mutant != "sm_no_abort_arrive":
            p_bar(t, arrived).arrive(32)

    roles = {"prod": producer(), "mma": mma(), "vw": v_warp(True, False), "w3": v_warp(f8, True)}
    for t in range(2):
        for q in range(4):
            roles[f"sm{t}.{q}"] = softmax_warp(t)
    return _run(roles, bars, state, tma, tensor_q, reads, widened, rng, slots, f8, slow_v_warp, abort_at,
                checking_reads, max_steps)


def _run(roles, bars, state, tma, tensor_q, reads, widened, rng, slots, f8, slow_v_warp, abort_at, checking_reads,
         max_steps):
    """Runs the roles (generators yielding their next wait) and the two
    engines until every role has finished or nothing can move."""
    pending, joined, nwaits, done = {}, {}, collections.Counter(), set()

    def advance(k, value):
        try:
            req = roles[k].send(value)
        except StopIteration:
            done.add(k)
            pending[k] = None
            return
        if req[0] == "nsync":
            joined[k] = req[1].arrive(req[2])
        elif req[0] == "wait":
            nwaits[k] += 1
            if abort_at is not None and abort_at == (k, nwaits[k]):
                req = ("timeout",)
        pending[k] = req

    def ready(k):
        """(True, value to resume with) when role k can move."""
        req = pending[k]
        if req[0] == "wait":
            if bars[req[1]].passes(req[2]):
                return True, True
            return (True, False) if state["abort"] else (False, None)
        if req[0] == "timeout":
            state["abort"] = True
            return True, False
        if req[0] == "nsync":
            return req[1].rounds > joined[k], None
        return True, None

    for k in roles:
        advance(k, None)
    for _ in range(max_steps):
        for e in tma:
            e[0] -= 1
        for e in [e for e in tma if e[0] <= 0]:
            tma.remove(e)
            bars[e[1]].arrive(e[2])
        if tensor_q and rng.random() < 0.5:
            op = tensor_q.pop(0)
            if op[0] == "commit":
                bars[op[1]].arrive(op[2])
            else:
                for b in op[1]:
                    reads[b] -= 1
                    if checking_reads and f8 and b[0] == "kv" and b[1] % 2 == 1 and widened[b[1]] < 2:
                        raise ProtocolError(f"MMA read V use {b[1]} before both halves were widened")
        movable = {}
        for k in roles:
            if k in done:
                continue
            ok, value = ready(k)
            if ok:
                movable[k] = value
        if not movable:
            if not tma and not tensor_q:
                return None if len(done) == len(roles) else {k: pending[k][:2] for k in roles if k not in done}
            continue
        keys = list(movable)
        if slow_v_warp and "vw" in keys and len(keys) > 1 and rng.random() < 0.9:
            keys.remove("vw")
        k = rng.choice(keys)
        advance(k, movable[k])
    raise AssertionError("schedule did not finish")


def _cases(n, seed0):
    rng = random.Random(seed0)
    for i in range(n):
        segs = [(rng.randint(1, 12), rng.choice([1, 1, 2])) for _ in range(rng.randint(2, 8))]
        yield segs, rng.choice([5, 8]), seed0 + i, i % 2 == 0


ROLES = ["prod", "mma", "vw", "w3"] + [f"sm{t}.{q}" for t in range(2) for q in range(4)]


@pytest.mark.parametrize("f8", [False, True])
def test_pipeline_never_deadlocks_and_waits_are_sound(f8):
    stuck = [(segs, slots, seed) for segs, slots, seed, slow in _cases(120, 7000)
             if _simulate(segs, slots, seed, None, slow, f8=f8) is not None]
    assert not stuck, stuck[:3]


@pytest.mark.parametrize("f8", [False, True])
def test_every_role_leaves_when_any_role_gives_up(f8):
    """Whichever role times out, at whichever of its waits, every role ends:
    no warp is left in a named-barrier sync, and no round takes more
    arrivals than its count."""
    rng = random.Random(321 + f8)
    stuck = []
    for segs, slots, seed, slow in _cases(240, 8000):
        role = rng.choice(ROLES)
        n = rng.randint(1, 12)
        res = _simulate(segs, slots, seed, None, slow, f8=f8, abort_at=(role, n))
        if res is not None:
            stuck.append((segs, slots, seed, role, n, res))
    assert not stuck, stuck[:2]


def _caught(mutant, f8, aborts, n=800, seed0=9100):
    rng = random.Random(seed0 + 1)
    for segs, slots, seed, slow in _cases(n, seed0):
        abort_at = (rng.choice(ROLES), rng.randint(1, 12)) if aborts else None
        try:
            if _simulate(segs, slots, seed, mutant, slow, f8=f8, abort_at=abort_at) is not None:
                return True
        except ProtocolError:
            return True
    return False


@pytest.mark.parametrize("mutant, f8", [("shared_v_only", False), ("shared_all", False), ("early_v_release", False),
                                        ("early_q_release", False), ("f8_count1", True)])
def test_model_catches_protocol_mutants(mutant, f8):
    """Each flawed protocol breaks on some schedule: an arrival for a phase
    the barrier is not in, a waiter two phases behind, a load over a buffer
    still to be read, a V tile read before it is widened, or a deadlock."""
    assert _caught(mutant, f8, aborts=False)


@pytest.mark.parametrize("mutant", ["single_pbar", "sm_no_abort_arrive", "mma_no_abort_arrive",
                                    "voucher_no_abort_arrive", "mma_no_flag_check"])
def test_model_catches_give_up_mutants(mutant):
    """Each flawed way of leaving breaks once some role gives up: a warp left
    blocked in a named-barrier sync, or a round with too many arrivals."""
    assert _caught(mutant, False, aborts=True)
