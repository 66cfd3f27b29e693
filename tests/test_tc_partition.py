"""CPU model of the tensor-memory attention kernel's work partition.

The kernel (csrc/attention_tc.cu, tc_plan + TcWalker) orders the (sequence,
virtual head) segments, gives each a start-up cost of kSegCost units in front
of its tiles, and hands CTA c the units [c*quota, (c+1)*quota).  Its split-
segment protocol relies on three properties, checked here over random ragged
batches with the kernel's own constants read from the source:
  - every tile of every segment lands in exactly one piece;
  - a split segment's first piece (tile 0) is the last piece of its CTA, so
    it can use the CTA's second partial slot;
  - every other piece of a split segment is the first piece of its CTA (the
    first slot), and every CTA between the first and the last holds one (the
    ticket counts exactly those pieces).
The GPU tests exercise the kernel itself; this pins the arithmetic it uses."""
import os
import random
import re

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "..", "gqa_decode_attention_02_gb300", "csrc", "attention_tc.cu")


def kernel_constant(name):
    m = re.search(r"constexpr int %s = (\d+);" % name, open(SRC).read())
    assert m, name
    return int(m.group(1))


SEG_COST = kernel_constant("kSegCost")
QUOTA_MIN = kernel_constant("kQuotaMinTc")


def pieces_of(nblks, kc, grid):
    """Pieces (b, v, nb, t0, t1, first) of each CTA, as the kernel's walker
    produces them."""
    units = [kc * (nb + SEG_COST if nb > 0 else 0) for nb in nblks]
    total = sum(units)
    quota = max(-(-total // grid), QUOTA_MIN)
    out = {}
    for c in range(grid):
        c0, c1 = c * quota, min(total, c * quota + quota)
        out[c] = []
        if c0 >= c1:
            continue
        acc, b0 = 0, 0
        for b, u in enumerate(units):  # the sequence whose units hold c0
            if c0 < acc + u:
                b0 = b
                break
            acc += u
        pos, base, b, v, nb = c0, acc, b0, 0, nblks[b0]
        while pos < c1:
            seg = nb + SEG_COST if nb > 0 else 0
            first = base + v * seg
            if nb > 0 and pos < first + seg:
                e = min(c1, first + seg)
                tile0 = first + SEG_COST
                s0 = max(pos, tile0)
                pos = e
                if e > s0:
                    out[c].append((b, v, nb, s0 - tile0, e - tile0, tile0))
                continue
            if nb > 0:
                v += 1
                if v < kc:
                    continue
            base += kc * seg
            v = 0
            b += 1
            if b >= len(nblks):
                break
            nb = nblks[b]
    return out, quota


def check(nblks, kc, grid):
    pieces, quota = pieces_of(nblks, kc, grid)
    cover = {}
    for c, ps in pieces.items():
        for i, (b, v, nb, t0, t1, first) in enumerate(ps):
            assert 0 <= t0 < t1 <= nb
            for t in range(t0, t1):
                assert (b, v, t) not in cover
                cover[(b, v, t)] = c
            fc, lc = first // quota, (first + nb - 1) // quota
            if fc == lc:
                continue
            if t0 == 0:
                assert c == fc and i == len(ps) - 1  # first piece: ends its CTA's range
                for cc in range(fc + 1, lc + 1):
                    head = pieces[cc][0]
                    assert head[:2] == (b, v) and head[3] > 0  # later piece, first in range
            else:
                assert fc < c <= lc and i == 0
    assert set(cover) == {(b, v, t) for b, nb in enumerate(nblks) for v in range(kc)
                          for t in range(nb)}


def test_partition_invariants_on_random_ragged_batches():
    rng = random.Random(1)
    for _ in range(2000):
        nblks = [rng.choice([0, 1, 2, rng.randint(1, 300)]) for _ in range(rng.randint(1, 40))]
        check(nblks, rng.choice([1, 2, 8, 16]), rng.choice([1, 3, 152]))


def test_partition_on_the_verify_and_tree_shapes():
    rng = random.Random(2)
    nb = [(rng.randint(512, 4096) + 15) // 16 for _ in range(16)]
    check(nb, 8, 152)       # 40 rows per KV head: one chunk
    check(nb, 16, 152)      # 208 rows per KV head: two chunks
