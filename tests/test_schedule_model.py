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


# ---------------------------------------------------------------------------
# The SM-pair tree attention's weighted split (the formulas of its kernel
# header, written out).  A row group (sequence, KV head, pair of 128-row
# query tiles) has n = nt + ceil(P / 128) tiles: nt = ceil(N / 128) tree tiles
# then its prefix tiles.  It weighs n + SEG_W; its tree tiles all start at
# weight 0 within it and prefix tile t at SEG_W + t.  Cluster c's range is
# [c W / C, (c + 1) W / C) and holds the units whose start weights fall in
# it.  A cluster locates its first unit per sequence (all row groups of a
# sequence have the same n); parts of a row group cut by range ends leave
# partial slots (2c + 1 cut at the range end, 2c cut at its start) that the
# merge reads for clusters c_lo .. c_hi.

SEG_W = 3


def attn_units(tiles_per_seq, gpb, nt):
    """Every unit in order as (sequence, row group, tile, start weight,
    start weight of its row group)."""
    out, w = [], 0
    for b, n in enumerate(tiles_per_seq):
        for gi in range(gpb):
            for t in range(n):
                out.append((b, gi, t, w + (0 if t < nt else SEG_W + t), w))
            w += n + SEG_W
    return out, w


def attn_seek(x, tiles_per_seq, gpb, nt):
    """The kernel's placement of weight x: (b, gi, t, row-group weight), or
    None past the last unit."""
    wb = 0
    for b, n in enumerate(tiles_per_seq):
        wseq = gpb * (n + SEG_W)
        if wb + wseq > x:
            gi = (x - wb) // (n + SEG_W)
            r = x - wb - gi * (n + SEG_W)
            t = 0 if r == 0 else max(nt, r - SEG_W)
            wrg = wb + gi * (n + SEG_W)
            if t >= n:
                t, wrg, gi = 0, wrg + n + SEG_W, gi + 1
                if gi == gpb:
                    gi, b = 0, b + 1
            return (b, gi, t, wrg) if b < len(tiles_per_seq) else None
        wb += wseq
    return None


def check_attn(tiles_per_seq, gpb, nt, n_clusters):
    units, W = attn_units(tiles_per_seq, gpb, nt)
    C = max(1, min(n_clusters, W // (nt + SEG_W)))
    cluster_of = lambda x: ((x + 1) * C - 1) // W
    rs = [c * W // C for c in range(C + 1)]
    # 1. the placement is the first unit whose start weight is >= x
    first_at = []
    for c in range(C + 1):
        brute = next((i for i, u in enumerate(units) if u[3] >= rs[c]), len(units))
        got = attn_seek(rs[c], tiles_per_seq, gpb, nt)
        want = None if brute == len(units) else (units[brute][0], units[brute][1], units[brute][2], units[brute][4])
        assert got == want, (c, got, want)
        first_at.append(brute)
    parts = {}
    for c in range(C):
        lo, hi = first_at[c], first_at[c + 1]
        # 2. every range holds a unit; none starts between two tree tiles
        assert hi > lo, f"cluster {c} has no unit"
        assert not 0 < units[lo][2] < nt, "a range starts inside the tree tiles"
        for i in range(lo, hi):
            b, gi, t, _, _ = units[i]
            parts.setdefault((b, gi), []).append((c, i))
    written = {}
    for (b, gi), us in parts.items():
        clusters = sorted({c for c, _ in us})
        idx = [i for _, i in us]
        if len(clusters) == 1:
            continue           # complete in one range: normalised in place
        # 3. the contributors are consecutive, and the merge's c_lo / c_hi
        #    (from the row group's first and last unit weights) name them
        assert clusters == list(range(clusters[0], clusters[-1] + 1))
        first_u, last_u = units[min(idx)], units[max(idx)]
        assert cluster_of(first_u[4]) == clusters[0]
        assert cluster_of(last_u[3]) == clusters[-1]
        for c in clusters:
            mine = [i for cc, i in us if cc == c]
            cut_at_end = max(mine) == hi_of(first_at, c) - 1 and units[max(mine)][2] != tiles_per_seq[b] - 1
            slot = 2 * c + (1 if cut_at_end else 0)
            reader = 2 * c + (1 if c < clusters[-1] else 0)
            assert slot == reader, ((b, gi), c)
            assert slot not in written, f"slot {slot} written twice"
            written[slot] = (b, gi)
        # 4. exactly one range boundary inside the row group is the first:
        #    the merge of the row group is done once
        usable = [k for k in range(1, C) if units[first_at[k]][:2] == (b, gi) and units[first_at[k]][2] != 0
                  and cluster_of(units[first_at[k]][4]) == k - 1]
        assert len(usable) == 1


def hi_of(first_at, c):
    return first_at[c + 1]


def test_attention_split_workload_shapes():
    # (prefix lengths, row groups per sequence, tree nodes): the 70B serving
    # step, long context, the 8B EAGLE step, 256-node trees
    for prefix, gpb, n in [([4096] * 64, 8, 32), ([32768] * 4, 8, 64), ([512, 8192, 3000, 700, 4096, 1, 0, 6000], 8, 60),
                           ([4096] * 4, 32, 256), ([6000, 1, 3000], 32, 256), ([700, 0], 8, 256), ([333], 4, 130)]:
        nt = (n + 127) // 128
        tiles = [nt + (p + 127) // 128 for p in prefix]
        for clusters in (76, 74, 66, 7, 1):
            check_attn(tiles, gpb, nt, clusters)


def test_attention_split_random_shapes():
    rng = random.Random(9)
    for _ in range(300):
        nt = rng.choice([1, 1, 2])
        B = rng.randint(1, 12)
        tiles = [nt + rng.choice([0, 1, 2, 5, 33, rng.randint(0, 80)]) for _ in range(B)]
        check_attn(tiles, rng.randint(1, 9), nt, rng.randint(1, 80))
