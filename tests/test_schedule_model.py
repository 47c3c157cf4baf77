"""The weight-streaming GEMM's stream-K schedule, modelled on the CPU and
checked by brute force (no GPU).

The kernel splits the (tile, 64-wide K chunk) units of a GEMM into one
contiguous range per CTA, range_start(c) = floor(c * units / ctas).  A tile
whose chunks span several ranges is "cut": each contributor stores its
partial accumulator in a slot (2c when the tile is the first segment of CTA
c's range, 2c + 1 when it is a later one), and the fixup kernel sums the
slots of CTAs cta_of_unit(first chunk) .. cta_of_unit(last chunk), where
cta_of_unit(x) = floor(((x + 1) * ctas - 1) / units) and only the first
contributor can have started before the tile.  These are the
formulas of the kernel's header, written out here; the checks below are the
properties the schedule relies on, compared with brute force over every
unit."""
import random


def range_start(c, units, ctas):
    return c * units // ctas


def cta_of_unit(x, units, ctas):
    return ((x + 1) * ctas - 1) // units


def check(units_per_tile, tiles, ctas):
    units = units_per_tile * tiles
    starts = [range_start(c, units, ctas) for c in range(ctas + 1)]
    # 1. the ranges partition the units, each CTA at least one unit
    assert starts[0] == 0 and starts[-1] == units
    assert all(starts[c + 1] > starts[c] for c in range(ctas)), "an empty range"
    owner = {}
    for c in range(ctas):
        for u in range(starts[c], starts[c + 1]):
            owner[u] = c
    assert len(owner) == units
    # 2. cta_of_unit is the owner of every unit
    assert all(cta_of_unit(u, units, ctas) == owner[u] for u in range(units))
    slots_written = {}
    for t in range(tiles):
        lo, hi = t * units_per_tile, (t + 1) * units_per_tile
        contributors = sorted({owner[u] for u in range(lo, hi)})
        c_first, c_last = cta_of_unit(lo, units, ctas), cta_of_unit(hi - 1, units, ctas)
        # 3. the contributors are exactly c_first .. c_last, without gaps
        assert contributors == list(range(c_first, c_last + 1))
        if len(contributors) == 1:
            continue          # a whole tile: no partial slots
        for c in contributors:
            # the writer's rule: slot 2c for the first segment of its range
            first_segment = starts[c] >= lo and starts[c] < hi
            writer = 2 * c + (0 if first_segment else 1)
            # the reducer's rule: only c_first may have started before the tile
            reducer = 2 * c + (0 if (c != c_first or starts[c_first] >= lo) else 1)
            assert writer == reducer, (t, c)
            assert writer not in slots_written, f"slot {writer} reused by tiles {slots_written.get(writer)} and {t}"
            slots_written[writer] = t
    # 4. at most two slots per CTA (its first and its last segment)
    per_cta = {}
    for s in slots_written:
        per_cta.setdefault(s // 2, []).append(s)
    assert all(len(v) <= 2 for v in per_cta.values())


def test_workload_shapes():
    # (K chunks per tile, tiles, CTAs): Medusa W1 and W2 at hidden 4096, LM
    # heads at vocabularies 32000 and 128256, the EAGLE draft layer's products
    for nk, tiles in [(64, 64), (64, 500), (64, 125), (64, 501), (128, 16), (64, 56), (224, 16), (64, 24)]:
        for ctas in (152, 148, 132, 76):
            if nk * tiles >= ctas:
                check(nk, tiles, ctas)


def test_random_shapes():
    rng = random.Random(5)
    for _ in range(400):
        nk = rng.choice([1, 2, 3, 4, 16, 64, 128, 224])
        tiles = rng.randint(1, 400)
        ctas = rng.randint(1, 160)
        if nk * tiles >= ctas:      # the host never launches more CTAs than units
            check(nk, tiles, ctas)
