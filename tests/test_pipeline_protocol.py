"""A CPU model of the tree-attention kernel's mbarrier pipeline, run over
random schedules: it must never deadlock, every parity wait must be sound, and
no load may land in a buffer that a queued MMA has still to read.

The model mirrors the roles of one CTA of the tensor-core tree pass: the TMA
producer (Q tiles, then K and V tiles of a ring of slots), the MMA issuer (per
key tile j and row tile t: PV_t(j), then S_t(j+1), which overwrites P_t(j)
only after PV_t(j) read it), the V-tile warp (hands each V tile to the MMA
issuer, publishes the segment's poison mask) and the two softmax groups, plus
the asynchronous engines: TMA copies land after random delays and the tensor
core runs the issuer's MMAs and commits in order.

A barrier counts completed phases. Every arrival names the phase it belongs
to, and the model checks it against the barrier's current phase. A parity
wait passes when the current phase's parity differs from the one named; the
model checks at every evaluation that the waiter is at most one phase behind,
the condition under which the hardware's answer is the intended one. The
model also tracks which buffers (Q tiles, ring slots) queued MMAs have still
to read, and fails if a load lands in one of them first.

With ``f8`` (an FP8 cache) two V-tile warps each widen half of every V
tile's rows in place and both arrive on vready and win_bar (count 2); the
tensor core must never read a V tile before both halves are widened.

Mutants the model has to catch: V-tile warps that wait on a barrier shared by
K and V loads (only for the V phases, or for every phase in order), a V slot
released after the first row tile's PV instead of the last, the Q tiles
released after a segment's second S instead of its last, and (FP8) vready
and win_bar left at count 1 for the two V warps.
"""
import collections
import random

import pytest


class ProtocolError(AssertionError):
    pass


class _Bar:
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


def _kind_index(use, slots):
    """Phase index of `use` on its slot's K (even uses) or V (odd uses)
    barrier: with an even ring a slot holds one kind, with an odd ring the
    kinds alternate by round."""
    rnd = use // slots
    return rnd if slots % 2 == 0 else rnd >> 1


def _simulate(segs, slots, seed, mutant=None, slow_v_warp=False, max_steps=600000, f8=False):
    """segs: (key tiles, row tiles present) per segment. Returns None when
    every role finishes, else the blocked waits; raises ProtocolError on an
    unsound step."""
    rng = random.Random(seed)
    bars = {}
    shared = mutant in ("shared_v_only", "shared_all")

    def bar(name, count=1):
        bars[name] = _Bar(name, count)

    for s in range(slots):
        for n in ("full", "kfull", "vfull", "empty"):
            bar(f"{n}{s}")
        bar(f"vready{s}", 2 if f8 and mutant != "f8_count1" else 1)
    for t in range(2):
        bar(f"s_full{t}"), bar(f"p_full{t}", 128), bar(f"o_fin{t}"), bar(f"o_free{t}", 128)
    bar("q_full"), bar("q_empty"), bar("win_bar", 2 if f8 and mutant != "f8_count1" else 1)
    tma = []                       # [delay, barrier, phase]
    tensor_q = []                  # the issuer's MMAs and commits, run in order
    reads = collections.Counter()  # buffers that queued MMAs have still to read
    widened = collections.Counter()  # F8: V use -> halves widened

    def mma_op(*bufs):
        for b in bufs:
            reads[b] += 1
        tensor_q.append(("op", bufs))

    def commit(name, phase):
        tensor_q.append(("commit", name, phase))

    def overwrite(buf):
        # a load may land in a buffer only once every MMA that reads its old contents has run
        if reads[buf]:
            raise ProtocolError(f"{buf} overwritten while an MMA still has to read it")

    def load_done(use):
        if shared:
            return f"full{use % slots}", use // slots
        return f"{'v' if use & 1 else 'k'}full{use % slots}", _kind_index(use, slots)

    def k_wait(use):
        name, ph = load_done(use)
        return ("wait", name, ph)

    def producer():
        use = 0
        for segc, (nkt, _) in enumerate(segs):
            yield ("wait", "q_empty", segc - 1)
            overwrite(("q", segc - 1))
            tma.append([rng.randint(1, 30), "q_full", segc])
            for _ in range(2 * nkt):
                yield ("wait", f"empty{use % slots}", use // slots - 1)
                overwrite(("kv", use - slots))
                tma.append([rng.randint(1, 30), *load_done(use)])
                use += 1

    def mma():
        use = 0
        tcnt, scnt = [0, 0], [0, 0]
        for segc, (nkt, nt) in enumerate(segs):
            yield ("wait", "q_full", segc)
            yield k_wait(use)
            for t in range(nt):
                mma_op(("q", segc), ("kv", use))
                commit(f"s_full{t}", tcnt[t])
            if nkt == 1:
                commit("q_empty", segc)
            commit(f"empty{use % slots}", use // slots)
            for j in range(nkt):
                vuse, kuse, more = use + 2 * j + 1, use + 2 * j + 2, j + 1 < nkt
                yield ("wait", f"vready{vuse % slots}", _kind_index(vuse, slots))
                if more:
                    yield k_wait(kuse)
                for t in range(nt):
                    yield ("wait", f"p_full{t}", tcnt[t] + j)
                    if j == 0 and scnt[t] > 0:
                        yield ("wait", f"o_free{t}", scnt[t] - 1)
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
            use += 2 * nkt
            for t in range(nt):
                tcnt[t] += nkt
                scnt[t] += 1

    def v_tile_warp():
        use, prev_nt, scnt = 0, 0, [0, 0]
        for segc, (nkt, nt) in enumerate(segs):
            for j in range(nkt):
                kuse, vuse = use + 2 * j, use + 2 * j + 1
                if mutant == "shared_v_only":
                    yield ("wait", f"full{vuse % slots}", vuse // slots)
                elif mutant == "shared_all":
                    yield ("wait", f"full{kuse % slots}", kuse // slots)
                    yield ("wait", f"full{vuse % slots}", vuse // slots)
                else:
                    yield ("wait", f"vfull{vuse % slots}", _kind_index(vuse, slots))
                if f8:
                    yield ("step",)
                    widened[vuse] += 1
                bars[f"vready{vuse % slots}"].arrive(_kind_index(vuse, slots))
                yield ("step",)
            for t in range(2):
                if t < prev_nt and scnt[t] > 0:
                    yield ("wait", f"o_free{t}", scnt[t] - 1)
            prev_nt = nt
            for t in range(nt):
                scnt[t] += 1
            bars["win_bar"].arrive(segc)
            use += 2 * nkt

    def softmax(t):
        tcnt = scnt = 0
        for segc, (nkt, nt) in enumerate(segs):
            if t >= nt:
                continue
            for j in range(nkt):
                yield ("wait", f"s_full{t}", tcnt + j)
                yield ("step",)
                bars[f"p_full{t}"].arrive(tcnt + j, 128)
            yield ("wait", f"o_fin{t}", scnt)
            yield ("wait", "win_bar", segc)
            yield ("step",)
            bars[f"o_free{t}"].arrive(scnt, 128)
            tcnt += nkt
            scnt += 1

    roles = {"prod": producer(), "mma": mma(), "vw": v_tile_warp(), "sm0": softmax(0), "sm1": softmax(1)}
    if f8:
        roles["vw1"] = v_tile_warp()
    pending = {k: None for k in roles}
    done = set()
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
                    if f8 and b[0] == "kv" and b[1] % 2 == 1 and widened[b[1]] < 2:
                        raise ProtocolError(f"MMA read V use {b[1]} before both halves were widened")
        ready = [k for k in roles if k not in done and (pending[k] is None or bars[pending[k][1]].passes(pending[k][2]))]
        if not ready:
            if not tma and not tensor_q:
                return None if len(done) == len(roles) else {k: pending[k] for k in roles if k not in done}
            continue
        if slow_v_warp and "vw" in ready and len(ready) > 1 and rng.random() < 0.9:
            ready.remove("vw")
        if f8 and slow_v_warp and "vw1" in ready and len(ready) > 1 and rng.random() < 0.5:
            ready.remove("vw1")
        k = rng.choice(ready)
        try:
            nxt = next(roles[k])
            pending[k] = nxt if nxt[0] == "wait" else None
        except StopIteration:
            done.add(k)
            pending[k] = None
    raise AssertionError("schedule did not finish")


def _cases(n, seed0):
    rng = random.Random(seed0)
    for i in range(n):
        segs = [(rng.randint(1, 12), rng.choice([1, 1, 2])) for _ in range(rng.randint(2, 8))]
        yield segs, rng.choice([5, 8]), seed0 + i, i % 2 == 0


@pytest.mark.parametrize("f8", [False, True])
def test_pipeline_never_deadlocks_and_waits_are_sound(f8):
    stuck = [(segs, slots, seed) for segs, slots, seed, slow in _cases(120, 7000)
             if _simulate(segs, slots, seed, None, slow, f8=f8) is not None]
    assert not stuck, stuck[:3]


@pytest.mark.parametrize("mutant, f8", [("shared_v_only", False), ("shared_all", False), ("early_v_release", False),
                                        ("early_q_release", False), ("f8_count1", True)])
def test_model_catches_protocol_mutants(mutant, f8):
    """Each flawed protocol breaks on some schedule: an arrival for a phase
    the barrier is not in, a waiter two phases behind, a load over a buffer
    still to be read, a K tile read before it is widened, or a deadlock."""
    caught = False
    for segs, slots, seed, slow in _cases(800, 9100):
        try:
            caught = _simulate(segs, slots, seed, mutant, slow, f8=f8) is not None
        except ProtocolError:
            caught = True
        if caught:
            break
    assert caught
