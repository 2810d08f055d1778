"""A CPU model of the tree-attention kernel's mbarrier pipeline, run over
random schedules: it must never deadlock.

The model mirrors the roles of one CTA of the tensor-core tree pass: the TMA
producer (Q tile, then K and V tiles of a ring of slots), the MMA issuer, the
V-tile warp (hands each V tile to the MMA issuer) and the two softmax groups,
plus the asynchronous engines (TMA copies complete after random delays, the
tensor core runs its queue in order). A barrier counts completed phases; a
parity wait passes when the current phase's parity differs from the one
named, which is only sound while the waiter is at most one phase behind.

Two variants of the V-tile warp that an earlier form of the kernel used are
kept as mutants: waiting on a barrier shared by K and V loads (both only for
the V phases, and for every phase in order) deadlocks on some schedules, and
the model has to catch both.
"""
import random

import pytest


class _Bar:
    def __init__(self, count):
        self.count, self.pend, self.done = count, 0, 0

    def arrive(self, k=1):
        self.pend += k
        assert self.pend <= self.count
        if self.pend == self.count:
            self.pend = 0
            self.done += 1

    def passes(self, parity):
        return (self.done & 1) != parity


def _kind_phase(use, slots):
    rnd = use // slots
    return (rnd if slots % 2 == 0 else rnd >> 1) & 1


def _simulate(segs, slots, seed, v_warp="split", slow_v_warp=False, max_steps=400000):
    """segs: (key tiles, row tiles) per segment. Returns None when every role
    finishes, else the blocked waits."""
    rng = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        bars.setdefault(name, _Bar(count))
        return bars[name]

    for s in range(slots):
        for n in ("full", "kfull", "vfull", "empty", "vready"):
            bar(f"{n}{s}")
    for t in range(2):
        bar(f"s_full{t}"), bar(f"p_full{t}", 128), bar(f"o_fin{t}"), bar(f"o_free{t}", 128)
    bar("q_full"), bar("q_empty"), bar("win_bar")
    tma, tensor_q = [], []
    split = v_warp == "split"

    def load_done(use):
        if not split:
            return f"full{use % slots}"
        return f"{'v' if use & 1 else 'k'}full{use % slots}"

    def k_wait(use):
        if split:
            return ("wait", f"kfull{use % slots}", _kind_phase(use, slots))
        return ("wait", f"full{use % slots}", (use // slots) & 1)

    def producer():
        use = segc = 0
        for nkt, _ in segs:
            yield ("wait", "q_empty", (segc & 1) ^ 1)
            tma.append([rng.randint(1, 30), "q_full"])
            segc += 1
            for _ in range(2 * nkt):
                yield ("wait", f"empty{use % slots}", ((use // slots) & 1) ^ 1)
                tma.append([rng.randint(1, 30), load_done(use)])
                use += 1

    def mma():
        use = segc = 0
        tcnt, scnt = [0, 0], [0, 0]
        for nkt, nt in segs:
            yield ("wait", "q_full", segc & 1)
            yield k_wait(use)
            for t in range(nt):
                tensor_q.append(("commit", f"s_full{t}"))
            if nkt == 1:
                tensor_q.append(("commit", "q_empty"))
            tensor_q.append(("commit", f"empty{use % slots}"))
            for j in range(nkt):
                vuse, kuse, more = use + 2 * j + 1, use + 2 * j + 2, j + 1 < nkt
                yield ("wait", f"vready{vuse % slots}", _kind_phase(vuse, slots))
                if more:
                    yield k_wait(kuse)
                for t in range(nt):
                    yield ("wait", f"p_full{t}", (tcnt[t] + j) & 1)
                    if j == 0 and scnt[t] > 0:
                        yield ("wait", f"o_free{t}", (scnt[t] - 1) & 1)
                    tensor_q.append(("op",))
                    if t == nt - 1:
                        tensor_q.append(("commit", f"empty{vuse % slots}"))
                    if more:
                        tensor_q.append(("commit", f"s_full{t}"))
                        if t == nt - 1:
                            if j + 2 == nkt:
                                tensor_q.append(("commit", "q_empty"))
                            tensor_q.append(("commit", f"empty{kuse % slots}"))
                    else:
                        tensor_q.append(("commit", f"o_fin{t}"))
            use += 2 * nkt
            for t in range(nt):
                tcnt[t] += nkt
                scnt[t] += 1
            segc += 1

    def v_tile_warp():
        use, prev_nt, scnt = 0, 0, [0, 0]
        for nkt, nt in segs:
            for j in range(nkt):
                kuse, vuse = use + 2 * j, use + 2 * j + 1
                if v_warp == "split":
                    yield ("wait", f"vfull{vuse % slots}", _kind_phase(vuse, slots))
                elif v_warp == "shared_v_only":
                    yield ("wait", f"full{vuse % slots}", (vuse // slots) & 1)
                else:  # shared, every phase in order
                    yield ("wait", f"full{kuse % slots}", (kuse // slots) & 1)
                    yield ("wait", f"full{vuse % slots}", (vuse // slots) & 1)
                bars[f"vready{vuse % slots}"].arrive()
                yield ("step",)
            for t in range(2):
                if t < prev_nt and scnt[t] > 0:
                    yield ("wait", f"o_free{t}", (scnt[t] - 1) & 1)
            prev_nt = nt
            for t in range(nt):
                scnt[t] += 1
            bars["win_bar"].arrive()
            use += 2 * nkt

    def softmax(t):
        tcnt = scnt = wcnt = 0
        for nkt, nt in segs:
            wpar = wcnt & 1
            wcnt += 1
            if t >= nt:
                continue
            for j in range(nkt):
                yield ("wait", f"s_full{t}", (tcnt + j) & 1)
                yield ("step",)
                bars[f"p_full{t}"].arrive(128)
            yield ("wait", f"o_fin{t}", scnt & 1)
            yield ("wait", "win_bar", wpar)
            yield ("step",)
            bars[f"o_free{t}"].arrive(128)
            tcnt += nkt
            scnt += 1

    roles = {"prod": producer(), "mma": mma(), "vw": v_tile_warp(), "sm0": softmax(0), "sm1": softmax(1)}
    pending = {k: None for k in roles}
    done = set()
    for _ in range(max_steps):
        for e in tma:
            e[0] -= 1
        for e in [e for e in tma if e[0] <= 0]:
            tma.remove(e)
            bars[e[1]].arrive()
        if tensor_q and rng.random() < 0.5:
            op = tensor_q.pop(0)
            if op[0] == "commit":
                bars[op[1]].arrive()
        ready = [k for k in roles if k not in done and (pending[k] is None or bars[pending[k][1]].passes(pending[k][2]))]
        if not ready:
            if not tma and not tensor_q:
                return None if len(done) == len(roles) else {k: pending[k] for k in roles if k not in done}
            continue
        if slow_v_warp and "vw" in ready and len(ready) > 1 and rng.random() < 0.9:
            ready.remove("vw")
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


def test_pipeline_never_deadlocks():
    stuck = [(segs, slots, seed) for segs, slots, seed, slow in _cases(120, 7000)
             if _simulate(segs, slots, seed, "split", slow) is not None]
    assert not stuck, stuck[:3]


@pytest.mark.parametrize("variant", ["shared_v_only", "shared_all"])
def test_model_catches_shared_barrier_variants(variant):
    """Each flawed V-tile warp deadlocks on some schedule: the model can see
    the failure the split barriers remove."""
    found = any(_simulate(segs, slots, seed, variant, slow) is not None for segs, slots, seed, slow in _cases(160, 9100))
    assert found
