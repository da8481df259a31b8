"""The order in which the ring kernel walks a unit's key tiles, checked on the host.

A unit is a block of query rows of one query shard.  For each ring step
(key shard s = (r - t) mod cp) the kernel runs key tiles [0, nk), where nk
covers every key some row of the unit sees.  It splits them into two
phases: first, step by step, the tiles [0, km) with km = (lo + 1) // 128,
lo being the last key the unit's FIRST row sees in that step; then the
tiles [km, nk).  The softmax runs the first phase without any mask, so the
split is only correct if every row of the unit sees every first-phase tile
whole.  That holds because a row's last visible key never decreases with
the row.  These tests compute visibility by brute force from global token
positions (contiguous shards: r * Ls + a; striped shards: a * cp + r; a key
is visible iff its global position is not after the query's) and check the
split against it, ragged shard lengths included."""
import pytest

BN = 128


def global_pos(layout, cp, Ls, shard, a):
    return shard * Ls + a if layout == "contiguous" else a * cp + shard


def last_visible(layout, cp, Ls, r, a, s):
    """Largest local key index b of shard s that query (r, a) sees, or -1."""
    g = global_pos(layout, cp, Ls, r, a)
    best = -1
    for b in range(Ls):
        if global_pos(layout, cp, Ls, s, b) <= g:
            best = b
    return best


def unit_phases(layout, cp, Ls, r, q0, rows):
    """[(step, phase-0 tiles, phase-1 tiles)] for the unit, by the kernel's rule,
    plus the brute-force visibility table lim[s][row]."""
    a_max = min(q0 + rows, Ls) - 1
    out, lims = [], {}
    for t in range(cp):
        s = (r - t) % cp
        lim = [last_visible(layout, cp, Ls, r, a, s) for a in range(q0, a_max + 1)]
        lims[s] = lim
        nk = 0 if max(lim) < 0 else max(lim) // BN + 1
        lo = lim[0]
        km = 0 if lo < 0 else min(nk, (lo + 1) // BN)
        out.append((s, list(range(0, km)), list(range(km, nk)), nk))
    return out, lims


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("Ls,cp,rows", [(512, 4, 128), (300, 3, 128), (1000, 2, 256), (384, 8, 256)])
def test_first_phase_tiles_are_seen_whole_by_every_row(layout, Ls, cp, rows):
    for r in range(cp):
        for q0 in range(0, Ls, rows):
            phases, lims = unit_phases(layout, cp, Ls, r, q0, rows)
            for s, p0, p1, nk in phases:
                lim = lims[s]
                # every tile once, in the two phases
                assert p0 + p1 == list(range(nk))
                for kt in p0:  # no row of the unit needs a mask on these
                    assert all(l >= min(kt * BN + BN - 1, Ls - 1) and kt * BN + BN <= Ls for l in lim), \
                        (layout, Ls, cp, r, q0, s, kt)
                if p1:  # the split is tight: the first row does not see tile km whole
                    kt = p1[0]
                    assert lim[0] < kt * BN + BN - 1


def test_striped_units_end_with_one_masked_tile_per_step():
    """Striped shards put a causal diagonal in every shard pair: a unit of
    whole 128-row tiles ends with exactly one masked tile per key shard, the
    contiguous layout with one in all (its own shard's diagonal)."""
    cp, Ls, rows = 4, 512, 128
    for layout, want in (("striped", cp), ("contiguous", 1)):
        for r in range(cp):
            for q0 in range(0, Ls, rows):
                phases, _ = unit_phases(layout, cp, Ls, r, q0, rows)
                assert sum(len(p1) for _, _, p1, _ in phases) == want, (layout, r, q0)
