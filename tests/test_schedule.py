"""Host-side check of the decode work decomposition's arithmetic (no GPU).

The decode kernel lays all (request, kv head, query slice) units' tiles end to
end, gives CTA c the range [c*T/n, (c+1)*T/n), cuts each unit into S equal
split ranges, and stores the piece (CTA range x split range) at workspace slot
c + (unit * S + split).  combine_kernel finds a unit's pieces with part_of().
These tests restate the two formulas and check, by brute force, that ranges
tile the line, that part_of inverts part_begin, and that piece slots are
unique and cover every tile exactly once."""
import random

import pytest


def part_begin(i, total, parts):
    return i * total // parts


def part_of(x, total, parts):
    return ((x + 1) * parts - 1) // total


@pytest.mark.parametrize("total", [1, 2, 3, 7, 31, 64, 100, 1000])
@pytest.mark.parametrize("parts", [1, 2, 3, 5, 8, 152, 304, 2000])
def test_part_of_inverts_part_begin(total, parts):
    for x in range(total):
        c = part_of(x, total, parts)
        assert 0 <= c < parts
        assert part_begin(c, total, parts) <= x < part_begin(c + 1, total, parts)
    assert part_begin(parts, total, parts) == total


def pieces(tiles_per_unit, n_cta, S):
    """Enumerate (slot, unit, split, cta, tile range) the way the kernel does."""
    T = sum(tiles_per_unit)
    starts = [0]
    for n in tiles_per_unit:
        starts.append(starts[-1] + n)
    out = []
    for c in range(n_cta):
        x, c1 = part_begin(c, T, n_cta), part_begin(c + 1, T, n_cta)
        u = 0
        while x < c1:
            while x >= starts[u + 1]:
                u += 1
            n_u = tiles_per_unit[u]
            t = x - starts[u]
            s = part_of(t, n_u, S)
            n = min(part_begin(s + 1, n_u, S) - t, c1 - x)
            out.append((c + u * S + s, u, s, c, t, n))
            x += n
    return out


def test_piece_slots_unique_and_covering():
    rng = random.Random(0)
    for _ in range(300):
        units = [rng.choice([0, 1, 2, 5, 40, 300]) for _ in range(rng.randint(1, 30))]
        if sum(units) == 0:
            continue
        n_cta = rng.choice([1, 2, 7, 152, 304])
        S = rng.choice([1, 2, 3, 128])
        ps = pieces(units, n_cta, S)
        slots = [p[0] for p in ps]
        assert len(slots) == len(set(slots))
        assert max(slots) < n_cta + len(units) * S
        covered = [[0] * n for n in units]
        for slot, u, s, c, t, n in ps:
            for k in range(t, t + n):
                covered[u][k] += 1
        assert all(v == 1 for row in covered for v in row)
        # combine's view: every (split, CTA) it visits for a unit is a real piece
        T = sum(units)
        start = 0
        real = {(p[1], p[2], p[3]) for p in ps}
        for u, n_u in enumerate(units):
            for s in range(S):
                x0, x1 = start + part_begin(s, n_u, S), start + part_begin(s + 1, n_u, S)
                if x1 <= x0:
                    continue
                for c in range(part_of(x0, T, n_cta), part_of(x1 - 1, T, n_cta) + 1):
                    if part_begin(c, T, n_cta) == part_begin(c + 1, T, n_cta):
                        continue          # CTA with an empty range holds no piece
                    assert (u, s, c) in real
            start += n_u


def step_jobs(tiles_per_request, UPB, n_cta):
    """kv4_decode_step's new-token jobs, per CTA, the way the kernel lists
    them: request b's units occupy [start_b, start_b + UPB n_b) of the line
    (n_b tiles each, in unit order), unit j's last tile is start_b + (j + 1)
    n_b - 1, and CTA c writes the units whose last tile is in its range."""
    T = UPB * sum(tiles_per_request)
    jobs = {c: [] for c in range(n_cta)}
    start = 0
    for b, n_b in enumerate(tiles_per_request):
        for c in range(n_cta):
            c0, c1 = part_begin(c, T, n_cta), part_begin(c + 1, T, n_cta)
            for j in range(UPB):
                last = start + (j + 1) * n_b - 1
                if n_b > 0 and c0 <= last < c1:
                    jobs[c].append(b * UPB + j)
        start += UPB * n_b
    return jobs


def test_step_jobs_owned_by_the_cta_that_decodes_the_last_tile():
    rng = random.Random(1)
    for _ in range(300):
        reqs = [rng.choice([0, 1, 2, 3, 17, 200]) for _ in range(rng.randint(1, 40))]
        UPB = rng.choice([1, 2, 4, 8])
        n_cta = rng.choice([1, 3, 7, 152, 456])
        jobs = step_jobs(reqs, UPB, n_cta)
        owner = {}
        for c, us in jobs.items():
            for u in us:
                assert u not in owner, "a new token written by two CTAs"
                owner[u] = c
        units = [n for n in reqs for _ in range(UPB)]
        for u, n_u in enumerate(units):
            if n_u == 0:
                assert u not in owner            # an empty request writes nothing
                continue
            assert u in owner                    # every other unit's token is written
        # the writer is the CTA whose piece holds the unit's last tile, so no
        # other CTA loads that tile
        for slot, u, s, c, t, n in pieces(units, n_cta, 1):
            if t + n == units[u]:
                assert owner[u] == c
