"""CPU model of the kernel's work decomposition (no GPU needed).

The decode kernel hands each CTA a list of unit pieces: in balanced mode the
visible 16-key tiles of all (sequence, KV head) units are laid end to end and
cut into equal contiguous ranges; with a fixed split count each unit is cut
into that many chunks, dealt round robin. This model restates those index
rules and checks the properties the kernel relies on: every visible tile is
processed exactly once, the piece count and slots that the split combine
derives for a unit from the prefix alone (all_slots) are those of the pieces
the walk cuts, in key order, partial slots are distinct and inside the
workspace the host sizes, and each empty unit gets exactly one zero-fill
piece.
"""
import itertools
import random

import pytest

TILE = 16


def seq_span(L, qlen, window, cap):
    L = min(max(L, 0), cap)
    if L == 0:
        return L, 0, 0
    lo = max(0, L - qlen - window + 1) if window > 0 else 0
    t0 = lo // TILE
    return L, t0, (L - 1) // TILE - t0 + 1


def chunk_plan(T, grid):
    """The balanced mode's cut: Ce = min(grid, T) contiguous ranges of equal
    size (to one tile), range k belonging to CTA k."""
    return dict(T=T, Ce=min(T, grid) if T > 0 else 0)


def chunk_start(cp, k):
    return cp["T"] * k // cp["Ce"]


def chunk_end(cp, k):
    return cp["T"] * (k + 1) // cp["Ce"]


def owner(cp, x):
    return ((x + 1) * cp["Ce"] - 1) // cp["T"]


def all_pieces(grid, B, Hkv, lens, qlen, window, cap, S, rng, cost=0):
    """Every CTA's pieces. In balanced mode each unit with visible tiles is
    preceded by `cost` virtual tiles (a piece's fixed cost), which count when
    the ranges are cut but are not processed."""
    spans = [seq_span(L, qlen, window, cap) for L in lens]
    per_cta = {c: [] for c in range(grid)}
    if S == 0:
        pre = [0]
        for _, _, n in spans:
            pre.append(pre[-1] + ((n + cost) * Hkv if n > 0 else 0))
        cp = chunk_plan(pre[B], grid)
        for k in range(cp["Ce"]):
            cta = k
            g, ge = chunk_start(cp, k), chunk_end(cp, k)
            while g < ge:
                b = max(i for i in range(B) if pre[i] <= g)
                span = (pre[b + 1] - pre[b]) // Hkv
                kh = (g - pre[b]) // span
                us = pre[b] + kh * span
                rs = us + cost  # first real tile of the unit
                ue = us + span
                if g < rs:
                    g = rs
                    if g >= ge:
                        break
                pe = min(ue, ge)
                L, t0, _ = spans[b]
                cf, cl = owner(cp, rs), owner(cp, ue - 1)
                npieces = cl - cf + 1
                slots = [2 * cf + (1 if chunk_start(cp, cf) < rs else 0)] + \
                        [2 * (cf + q) for q in range(1, npieces)]
                per_cta[cta].append(dict(unit=b * Hkv + kh, tiles=list(range(t0 + g - rs, t0 + pe - rs)),
                                         npieces=npieces, slot=2 * k + (1 if chunk_start(cp, k) < rs else 0),
                                         all_slots=slots))
                g = pe
        for c in range(grid):
            for b in range(c, B, grid):
                if pre[b + 1] == pre[b]:
                    for kh in range(Hkv):
                        per_cta[c].append(dict(unit=b * Hkv + kh, tiles=[], npieces=1, slot=None,
                                               all_slots=[]))
        return per_cta, 2 * grid
    total = B * Hkv * S
    for p in range(total):
        c = p % grid
        u, s = divmod(p, S)
        b, kh = divmod(u, Hkv)
        L, t0, n = spans[b]
        chunk = (n + S - 1) // S
        c0, c1 = s * chunk, min(s * chunk + chunk, n)
        if n == 0:
            if s == 0:
                per_cta[c].append(dict(unit=u, tiles=[], npieces=1, slot=None, all_slots=[]))
            continue
        if c0 >= c1:
            continue
        npieces = (n + chunk - 1) // chunk
        per_cta[c].append(dict(unit=u, tiles=list(range(t0 + c0, t0 + c1)), npieces=npieces,
                               slot=u * S + s, all_slots=[u * S + k for k in range(npieces)]))
    return per_cta, (B * Hkv * S if S > 1 else 0)


def check(B, Hkv, lens, qlen, window, cap, S, grid, seed=0, cost=0):
    seen = {}
    slots_used = []
    units_pieces = {}
    per_cta, nslots = all_pieces(grid, B, Hkv, lens, qlen, window, cap, S, random.Random(seed), cost)
    for c in range(grid):
        for pc in per_cta[c]:
            u = pc["unit"]
            units_pieces.setdefault(u, []).append(pc)
            for t in pc["tiles"]:
                assert (u, t) not in seen, "tile processed twice"
                seen[(u, t)] = c
            if pc["npieces"] > 1:
                assert 0 <= pc["slot"] < nslots
                slots_used.append(pc["slot"])
    assert len(slots_used) == len(set(slots_used)), "two pieces share a slot"
    for b, L in enumerate(lens):
        _, t0, n = seq_span(L, qlen, window, cap)
        for kh in range(Hkv):
            u = b * Hkv + kh
            pcs = units_pieces.get(u, [])
            got = sorted(t for pc in pcs for t in pc["tiles"])
            assert got == list(range(t0, t0 + n)), "tiles missing"
            if n == 0:
                assert len(pcs) == 1 and pcs[0]["tiles"] == [], "empty unit needs one zero piece"
                continue
            assert all(pc["npieces"] == len(pcs) for pc in pcs), "piece count mismatch"
            if len(pcs) > 1:
                assert sorted(pcs[0]["all_slots"]) == sorted(pc["slot"] for pc in pcs)
                # the combiner visits partials in key order
                order = [pc["slot"] for pc in sorted(pcs, key=lambda p: p["tiles"][0])]
                assert pcs[0]["all_slots"] == order


CASES = [
    (1, 4, [4096], 1, 0), (2, 4, [4096, 4096], 1, 0), (32, 4, [4096] * 32, 1, 0),
    (2, 2, [100, 0], 1, 0), (3, 2, [0, 0, 0], 1, 0), (4, 2, [1, 15, 17, 333], 1, 0),
    (3, 2, [1, 2, 40], 3, 0), (2, 1, [100, 16], 1, 1), (2, 2, [97, 300], 2, 5),
    (2, 4, [32768, 32768], 1, 4096), (8, 4, [8192] * 8, 3, 0),
]


@pytest.mark.parametrize("grid", [1, 3, 7, 152])
@pytest.mark.parametrize("S", [0, 1, 3, 8, 17])
@pytest.mark.parametrize("case", CASES)
def test_schedule_covers_each_tile_once(case, S, grid):
    B, Hkv, lens, qlen, window = case
    cap = 1 << 20
    check(B, Hkv, lens, qlen, window, cap, S, grid)


@pytest.mark.parametrize("grid", [1, 3, 7, 152])
@pytest.mark.parametrize("cost", [1, 16, 1000])
@pytest.mark.parametrize("case", CASES)
def test_balanced_schedule_with_unit_cost(case, cost, grid):
    """The tensor-memory kernel's split: every unit start charged `cost`
    virtual tiles (ranges that fall inside them do nothing)."""
    B, Hkv, lens, qlen, window = case
    check(B, Hkv, lens, qlen, window, 1 << 20, 0, grid, cost=cost)


def test_unit_cost_unloads_ranges_that_take_a_second_unit():
    # 32 units of 512 tiles over 152 ranges: without a cost every range gets
    # 107-108 real tiles whether it spans one unit or two; with a cost, a range
    # holding a unit's start gets up to `cost` fewer, and a range that takes on
    # a second unit always holds one
    B, Hkv, lens = 8, 4, [8192] * 8
    for cost in (0, 16):
        per_cta, _ = all_pieces(152, B, Hkv, lens, 3, 0, 1 << 20, 0, random.Random(0), cost=cost)
        real = [sum(len(pc["tiles"]) for pc in per_cta[c]) for c in range(152)]
        two = [r for c, r in enumerate(real) if len(per_cta[c]) == 2]
        one = [r for c, r in enumerate(real) if len(per_cta[c]) == 1]
        assert sum(real) == B * Hkv * 512 and two and one
        assert max(real) - min(real) <= cost + 1
        if cost:
            assert max(two) <= max(one) - cost


def test_schedule_random():
    rng = random.Random(0)
    for _ in range(200):
        B = rng.randint(1, 40)
        Hkv = rng.randint(1, 8)
        lens = [rng.choice([0, rng.randint(1, 20), rng.randint(1, 3000)]) for _ in range(B)]
        qlen = rng.randint(1, 4)
        window = rng.choice([0, 0, rng.randint(1, 500)])
        S = rng.choice([0, 0, 1, 2, 5, 9])
        grid = rng.choice([1, 2, 5, 16, 152])
        cost = rng.choice([0, 0, 16, rng.randint(1, 200)]) if S == 0 else 0
        check(B, Hkv, lens, qlen, window, 1 << 20, S, grid, seed=rng.randrange(1 << 30), cost=cost)


def chunk_start_qr(T, Ce, k):
    """The kernel's start(k): floor(T k / Ce) as q k + floor(r k / Ce)."""
    q, r = divmod(T, Ce)
    return q * k + (r * k) // Ce


def chunk_owner_stepped(T, Ce, x):
    """The kernel's owner(x): a single-precision estimate of x Ce / T, then
    steps along start() to the largest k with start(k) <= x."""
    import numpy as np
    k = int(np.float32(x) * (np.float32(Ce) / np.float32(T)))
    k = min(max(k, 0), Ce - 1)
    while k > 0 and chunk_start_qr(T, Ce, k) > x:
        k -= 1
    while k < Ce - 1 and chunk_start_qr(T, Ce, k + 1) <= x:
        k += 1
    return k


def test_chunk_plan_arithmetic_matches_the_division_form():
    rng = random.Random(5)
    cases = [(1, 1), (7, 7), (152, 152), (153, 152), (2 ** 31 - 1, 152), (2 ** 31 - 1, 304),
             (4112, 152), (4176, 152), (67_000_000, 304)]
    cases += [(rng.randint(1, 2 ** 31 - 1), rng.randint(1, 304)) for _ in range(300)]
    for T, grid in cases:
        Ce = min(T, grid)
        for k in set([0, 1, Ce - 1, Ce] + [rng.randint(0, Ce) for _ in range(20)]):
            assert chunk_start_qr(T, Ce, k) == T * k // Ce
        xs = [0, T - 1] + [rng.randint(0, T - 1) for _ in range(40)]
        xs += [T * k // Ce + d for k in range(min(Ce, 8)) for d in (-1, 0, 1) if 0 <= T * k // Ce + d < T]
        for x in xs:
            assert chunk_owner_stepped(T, Ce, x) == ((x + 1) * Ce - 1) // T, (T, Ce, x)
