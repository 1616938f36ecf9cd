"""Host-side model of the length-balanced decode partition.

CTA c of n owns positions [c*T/n, (c+1)*T/n) of the ordered (sequence, kv
head, page) list; the combine finds a unit's owners as
c(x) = ((x + 1) * n - 1) // T and skips CTAs whose share is empty.  These
properties are what the partial and combine kernels rely on."""
from __future__ import annotations

import numpy as np
import pytest


def share(c, T, n):
    return c * T // n, (c + 1) * T // n


def owner(x, T, n):
    return ((x + 1) * n - 1) // T


@pytest.mark.parametrize("seed", range(40))
def test_owners_and_pieces(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 20))
    Hkv = int(rng.integers(1, 9))
    n = int(rng.choice([1, 7, 148, 152, 160]))
    pages = [int(x) for x in rng.integers(0, 40, size=B)]
    T = Hkv * sum(pages)
    if T == 0:
        return
    # every position has exactly one owner, and owner() finds it
    own = np.full(T, -1)
    for c in range(n):
        a, b = share(c, T, n)
        assert a <= b
        own[a:b] = c
    assert (own >= 0).all()
    assert all(owner(x, T, n) == own[x] for x in range(T))
    # pieces of each unit: the non-empty CTAs between its first and last owner
    start = 0
    slots = set()
    for b in range(B):
        for g in range(Hkv):
            s_u, e_u = start, start + pages[b]
            start = e_u
            if pages[b] == 0:
                continue
            c0, c1 = owner(s_u, T, n), owner(e_u - 1, T, n)
            pieces = [c for c in range(c0, c1 + 1) if share(c, T, n)[0] < share(c, T, n)[1]]
            touching = sorted({own[x] for x in range(s_u, e_u)})
            assert pieces == touching
            u = b * Hkv + g
            for c in pieces:  # workspace slot c + u is unique
                assert (c + u) not in slots
                slots.add(c + u)
                assert c + u < n + B * Hkv
