"""Host model of how the tensor-core tree pass splits its work, checked on the
CPU over random shapes.

The pass lays every unit's key tiles out in one flat range, in the order
(row pair, request, KV head, key tile), and gives CTA c of G the tiles
[c T / G, (c + 1) T / G). A unit's tiles inside one CTA's range form a
segment; a unit split over several CTAs leaves one partial per segment in
slot (flat unit index + CTA index), and the merge pass finds a unit's parts as
the CTAs owning its first and last tiles. The model restates those rules and
checks what the kernels rely on: every tile is covered once, no two segments
share a partial slot (so slots = units + G suffice), a split unit's parts are
exactly the segments, and with two row pairs the two halves of the range are
mirror images (CTA c and c + G/2 walk the same (request, KV head, tile)).
"""
import random


def _units(prefix, Hkv, n_pairs, W=64):
    """Flat-order units: (pair, b, hkv, nkt)."""
    out = []
    for pair in range(n_pairs):
        for b, P in enumerate(prefix):
            nkt = (P + W + 127) // 128
            for h in range(Hkv):
                out.append((pair, b, h, nkt))
    return out


def _segments(prefix, Hkv, n_pairs, G):
    units = _units(prefix, Hkv, n_pairs)
    starts, x = [], 0
    for u in units:
        starts.append(x)
        x += u[3]
    T = x
    segs = []
    for c in range(G):
        x0, x1 = T * c // G, T * (c + 1) // G
        for ui, (u, s0) in enumerate(zip(units, starts)):
            lo, hi = max(x0, s0), min(x1, s0 + u[3])
            if lo < hi:
                segs.append(dict(cta=c, unit=ui, lt0=lo - s0, lt1=hi - s0, key=u[:3]))
    return units, starts, T, segs


def _owner(x, T, G):
    return ((x + 1) * G - 1) // T


def test_split_covers_every_tile_once_and_slots_are_distinct():
    rng = random.Random(11)
    for _ in range(300):
        B = rng.randint(1, 40)
        prefix = [rng.choice([0, 1, 127, 128, 500, 4096, 8192, rng.randint(0, 20000)]) for _ in range(B)]
        Hkv = rng.choice([1, 2, 8])
        n_pairs = rng.choice([1, 1, 2, 3])
        G = rng.choice([1, 7, 152])
        units, starts, T, segs = _segments(prefix, Hkv, n_pairs, G)
        covered = {}
        for sg in segs:
            for lt in range(sg["lt0"], sg["lt1"]):
                k = (sg["unit"], lt)
                assert k not in covered
                covered[k] = sg["cta"]
        assert len(covered) == T
        slots = [sg["unit"] + sg["cta"] for sg in segs]
        assert len(slots) == len(set(slots)), "two segments share a partial slot"
        assert all(s < len(units) + G for s in slots)
        # the merge's view: a unit's parts are the CTAs from the owner of its
        # first tile to the owner of its last, each with a segment of it
        by_unit = {}
        for sg in segs:
            by_unit.setdefault(sg["unit"], set()).add(sg["cta"])
        for ui, (u, s0) in enumerate(zip(units, starts)):
            if u[3] == 0:
                continue
            c0, c1 = _owner(s0, T, G), _owner(s0 + u[3] - 1, T, G)
            owning = {c for c in range(c0, c1 + 1) if T * c // G < T * (c + 1) // G}
            assert owning == by_unit[ui]


def test_two_row_pairs_walk_in_mirror():
    rng = random.Random(12)
    for _ in range(100):
        B = rng.randint(1, 8)
        prefix = [rng.randint(0, 140000) for _ in range(B)]
        G = 2 * rng.randint(1, 80)
        units, starts, T, segs = _segments(prefix, 8, 2, G)
        if T % 2:
            continue
        first = {(sg["cta"], sg["key"][1:], sg["lt0"], sg["lt1"]) for sg in segs if sg["key"][0] == 0}
        second = {(sg["cta"] - G // 2, sg["key"][1:], sg["lt0"], sg["lt1"]) for sg in segs if sg["key"][0] == 1}
        assert first == second


def test_split_units_merge_once_in_the_pass():
    """Without FP8 the tree pass merges a unit split over CTAs itself: every
    CTA holding a part counts it once (per-CTA counters 0 and 1 for its
    range's first and last segments, the only ones that can be parts), and
    the CTA that brings a unit's count to its number of parts (the groups
    c_first .. c_last that own tiles) merges it. The model checks that each
    split unit's parts are exactly those CTAs, that no CTA has more than two
    parts or two parts on one counter, and that in any arrival order exactly
    one CTA merges each split unit."""
    rng = random.Random(13)
    for _ in range(300):
        B = rng.randint(1, 40)
        prefix = [rng.choice([0, 1, 127, 128, 500, 4096, 8192, rng.randint(0, 20000)]) for _ in range(B)]
        Hkv = rng.choice([1, 2, 8])
        n_pairs = rng.choice([1, 1, 2, 3])
        G = rng.choice([1, 7, 152])
        units, starts, T, segs = _segments(prefix, Hkv, n_pairs, G)
        parts_of = {}
        per_cta = {}
        for sg in segs:
            u = units[sg["unit"]]
            if sg["lt0"] == 0 and sg["lt1"] == u[3]:
                continue  # a whole unit: written by its CTA, no part
            x0 = T * sg["cta"] // G
            k = 0 if starts[sg["unit"]] + sg["lt0"] == x0 else 1
            per_cta.setdefault(sg["cta"], []).append(k)
            parts_of.setdefault(sg["unit"], []).append(sg["cta"])
        for c, ks in per_cta.items():
            assert len(ks) <= 2 and len(set(ks)) == len(ks), (c, ks)
        for ui, ctas in parts_of.items():
            s0, nkt = starts[ui], units[ui][3]
            c0, c1 = _owner(s0, T, G), _owner(s0 + nkt - 1, T, G)
            parts = sum(1 for c in range(c0, c1 + 1) if T * c // G < T * (c + 1) // G)
            assert sorted(ctas) == list(range(c0, c1 + 1)) or len(ctas) == parts
            assert len(ctas) == parts >= 2
            order = ctas[:]
            rng.shuffle(order)
            cnt, mergers = 0, []
            for c in order:
                if cnt == parts - 1:
                    mergers.append(c)
                cnt += 1
            assert len(mergers) == 1
