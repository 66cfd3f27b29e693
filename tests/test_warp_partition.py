"""CPU model of the warp-level attention kernel's work partition.

The kernel's producer warp (csrc/attention.cu) orders the (sequence, virtual
head) segments, gives each kSegUnits start-up units in front of its tiles,
hands CTA c the units [c*quota, (c+1)*quota), and walks its range in stages of
at most kTilesPerStage tiles of one segment.  The consumers find a split
segment's CTAs from the unit of its first tile (first = start / quota, last =
(start + tiles - 1) / quota) and keep each CTA's pieces in two partial slots,
which relies on:
  - every tile of every segment lands in exactly one stage of one CTA;
  - the CTAs first..last each hold a piece, the first piece (tile 0) in CTA
    first, as that CTA's last segment;
  - every other piece is the first segment of its CTA.
Checked over random ragged batches with the kernel's constants read from the
source; the GPU tests exercise the kernel itself."""
import os
import random
import re

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "..", "gqa_decode_attention_02_gb300", "csrc", "attention.cu")


def kernel_constant(name):
    src = open(SRC).read()
    m = re.search(r"constexpr int %s = ([^;]+);" % name, src)
    assert m, name
    expr = m.group(1)
    for other in ("kTilesPerStage",):
        if other in expr:
            expr = expr.replace(other, str(kernel_constant(other)))
    return int(eval(expr, {}))


SEG_UNITS = kernel_constant("kSegUnits")
QUOTA_MIN = kernel_constant("kQuotaMin")
TILES = kernel_constant("kTilesPerStage")


def stages_of(nblks, kc, grid):
    """Stages (b, k, first tile, tiles, seg_start) each CTA issues, as the
    producer walks them."""
    units = [kc * (nb + SEG_UNITS if nb > 0 else 0) for nb in nblks]
    total = sum(units)
    quota = max(-(-total // grid), QUOTA_MIN)
    out = {}
    for c in range(grid):
        c0, c1 = c * quota, min(total, c * quota + quota)
        out[c] = []
        if c0 >= c1:
            continue
        acc = 0
        for b, u in enumerate(units):
            if c0 < acc + u:
                break
            acc += u
        base, nb = acc, nblks[b]
        su = nb + SEG_UNITS
        rel = c0 - base
        k = rel // su
        i = max(0, rel - k * su - SEG_UNITS)
        x = base + k * su + SEG_UNITS + i
        while x < c1:
            run = min(TILES, nb - i, c1 - x)
            out[c].append((b, k, i, run, base + k * su + SEG_UNITS))
            x += run
            i += run
            if i == nb:
                i = 0
                x += SEG_UNITS
                k += 1
                if k == kc:
                    k = 0
                    base += kc * su
                    if x < c1:
                        b += 1
                        while nblks[b] == 0:
                            b += 1
                        nb = nblks[b]
                        su = nb + SEG_UNITS
    return out, quota


def check(nblks, kc, grid):
    stages, quota = stages_of(nblks, kc, grid)
    cover = {}
    pieces = {}
    for c, sts in stages.items():
        ps = []
        for (b, k, i, run, start) in sts:
            assert 1 <= run <= TILES and 0 <= i and i + run <= nblks[b]
            for t in range(i, i + run):
                assert (b, k, t) not in cover
                cover[(b, k, t)] = c
            if not ps or ps[-1][:2] != (b, k):
                ps.append((b, k, i, start))
        pieces[c] = ps
    assert set(cover) == {(b, k, t) for b, nb in enumerate(nblks) for k in range(kc)
                          for t in range(nb)}
    for c, ps in pieces.items():
        for j, (b, k, t0, start) in enumerate(ps):
            first, last = start // quota, (start + nblks[b] - 1) // quota
            assert first <= c <= last
            if first == last:
                continue
            if t0 == 0:
                assert c == first and j == len(ps) - 1
            else:
                assert c > first and j == 0
            for cc in range(first + 1, last + 1):
                assert pieces[cc][0][:2] == (b, k)


def test_partition_invariants_on_random_ragged_batches():
    rng = random.Random(3)
    for _ in range(2000):
        nblks = [rng.choice([0, 1, 2, rng.randint(1, 300)]) for _ in range(rng.randint(1, 40))]
        if not any(nblks):
            continue
        check(nblks, rng.choice([1, 2, 8, 16]), rng.choice([1, 3, 152, 304]))


def test_partition_on_the_decode_workload_shapes():
    rng = random.Random(4)
    check([(rng.randint(16, 1024) + 15) // 16 for _ in range(64)], 2, 304)   # 24-layer batch
    check([19], 2, 3)                                                          # 295 tokens
    check([512] * 32, 8, 304)                                                  # 8192 tokens each
