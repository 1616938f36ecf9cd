"""Host-side model of the length-balanced decode partition.

Cost space: unit (sequence b, kv head g) with pb > 0 pages occupies W + pb
positions (W for the fixed work of a unit piece, then its pages); n parts
(at most one per warp, fewer when the total cost T is small) own
[v*T/n, (v+1)*T/n).  A part walks the units its share meets and processes the
pages whose positions fall inside it.  The combine locates a unit's pieces
as the parts between owner(first page) and owner(last page) whose share is
not empty, owner(x) = ((x + 1) * n - 1) // T.  These are the properties the
partial and combine kernels rely on."""
from __future__ import annotations

import numpy as np
import pytest

MIN_PART_COST = 4


def parts_in_use(T, n_parts):
    return max(1, min(n_parts, (T + MIN_PART_COST - 1) // MIN_PART_COST))


def owner(x, T, n):
    return ((x + 1) * n - 1) // T


def walk(share, units, W):
    """Pieces (unit index, first page, end page) of a share, walking the units
    like the kernel: start at the unit holding position share[0]."""
    s, e = share
    pieces = []
    for u, (start, pb) in enumerate(units):
        if pb == 0:
            continue
        pf = max(0, s - start - W)
        pe = min(pb, e - start - W)
        if pe > pf:
            pieces.append((u, pf, pe))
    return pieces


@pytest.mark.parametrize("seed", range(60))
def test_cost_partition(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 24))
    Hkv = int(rng.integers(1, 9))
    W = 2
    n_parts = int(rng.choice([8, 56, 1216]))
    pages = [int(x) for x in rng.integers(0, 60, size=B)]
    pages = [p if rng.random() > 0.1 else 0 for p in pages]  # some invalid lengths
    units, start = [], 0
    for b in range(B):
        for g in range(Hkv):
            units.append((start, pages[b]))
            if pages[b]:
                start += W + pages[b]
    T = start
    if T == 0:
        return
    n = parts_in_use(T, n_parts)
    assert 1 <= n <= n_parts
    shares = [(v * T // n, (v + 1) * T // n) for v in range(n)]
    covered = {}
    slots = set()
    per_unit = {}
    for v, sh in enumerate(shares):
        for (u, pf, pe) in walk(sh, units, W):
            for i in range(pf, pe):
                assert (u, i) not in covered, "page processed twice"
                covered[(u, i)] = v
            per_unit.setdefault(u, []).append((v, pf, pe))
            assert v + u < n_parts + len(units) and (v + u) not in slots
            slots.add(v + u)
    for u, (ustart, pb) in enumerate(units):
        if pb == 0:
            assert u not in per_unit
            continue
        assert all((u, i) in covered for i in range(pb)), "page never processed"
        p0 = ustart + W
        c0, c1 = owner(p0, T, n), owner(p0 + pb - 1, T, n)
        want = [v for v in range(c0, c1 + 1) if shares[v][0] < shares[v][1]]
        got = [v for v, _, _ in per_unit[u]]
        assert got == want
        whole = [(pf == 0 and pe == pb) for _, pf, pe in per_unit[u]]
        assert any(whole) == (c0 == c1) == (len(got) == 1)


# The kernels' own part count: CTAs in use = min(grid, ceil(T / 3)); eight
# warp parts a CTA with the in-CTA merge compiled in, else
# clamp(ceil(T / n_cta), 1, 8).  Both can exceed T (empty parts), which the
# combine must skip.  Row blocks are extra units: (b, kv head, block).
MIN_CTA_COST, CW = 3, 8


def kernel_parts(T, grid, cta_merge_variant):
    n_cta = max(1, min(grid, (T + MIN_CTA_COST - 1) // MIN_CTA_COST))
    wpc = CW if cta_merge_variant else max(1, min(CW, (T + n_cta - 1) // n_cta))
    return n_cta, n_cta * wpc


@pytest.mark.parametrize("seed", range(80))
def test_kernel_part_counts_locate_every_piece(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 20))
    Hkv = int(rng.integers(1, 9))
    NB = int(rng.choice([1, 1, 2, 3]))  # row blocks as units
    grid = int(rng.choice([4, 37, 152]))
    merge = bool(rng.integers(0, 2))
    W = 2
    pages = [int(x) for x in rng.integers(0, 40, size=B)]
    pages = [p if rng.random() > 0.1 else 0 for p in pages]
    units, start = [], 0
    for b in range(B):
        for g in range(Hkv * NB):
            units.append((start, pages[b]))
            if pages[b]:
                start += W + pages[b]
    T = start
    if T == 0:
        return
    n_cta, n = kernel_parts(T, grid, merge)
    assert n_cta <= grid and n <= n_cta * CW
    shares = [(v * T // n, (v + 1) * T // n) for v in range(n)]
    # CTA c's share is the union of its warps' shares
    for c in range(n_cta):
        w = n // n_cta
        assert shares[c * w][0] == c * T // n_cta and shares[c * w + w - 1][1] == (c + 1) * T // n_cta
    covered, per_unit = {}, {}
    for v, sh in enumerate(shares):
        for (u, pf, pe) in walk(sh, units, W):
            for i in range(pf, pe):
                assert (u, i) not in covered
                covered[(u, i)] = v
            per_unit.setdefault(u, []).append(v)
            assert v + u < n_cta * CW + len(units)  # workspace slot
    for u, (ustart, pb) in enumerate(units):
        if pb == 0:
            continue
        assert all((u, i) in covered for i in range(pb))
        p0 = ustart + W
        c0, c1 = owner(p0, T, n), owner(p0 + pb - 1, T, n)
        nonempty = [v for v in range(c0, c1 + 1) if (v * T // n) != ((v + 1) * T // n)]
        assert per_unit[u] == nonempty
        if T >= n:  # the combine's shortcut: no share is empty
            assert nonempty == list(range(c0, c1 + 1))
