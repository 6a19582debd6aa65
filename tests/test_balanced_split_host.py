"""Host check of the balanced decode split's arithmetic (CPU, no GPU).

The prepare kernel lays the decode groups' keys end to end on one line (each group
padded to whole 16-key stages and followed by a gap of kDecPieceCost keys that no CTA
processes, the cost of starting a piece) and gives CTA c the line's keys [c * share,
(c + 1) * share); it counts a group's pieces as one plus the share boundaries inside
the group and records, per CTA, the group its share starts in.  The decode kernel cuts
its pieces from those records.  This test restates both rules in Python and checks, for
random batches, that every key of every group is covered exactly once and that a group's
split indices are exactly 0 .. pieces - 1 (so every partial slot is written once).
"""
import os
import random
import re

import pytest

_HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "paged_variable_length_gb300",
                    "csrc", "pva_internal.h")
_CONST = lambda name: int(re.search(name + r"\s*=\s*(\d+)", open(_HDR).read()).group(1))
STAGE, MIN_SHARE, PIECE_COST = _CONST("kDecKeysPerStage"), _CONST("kMinDecShare"), _CONST("kDecPieceCost")


def _plan(exts, n_ctas, min_share=MIN_SHARE, cost=PIECE_COST):
    r16 = lambda x: (x + STAGE - 1) // STAGE * STAGE
    line = sum(r16(e) + cost for e in exts)
    share = max(min_share, r16((line + n_ctas - 1) // n_ctas))
    g0s, x = [], 0
    for e in exts:
        g0s.append(x)
        x += r16(e) + cost
    pieces = [1 + (g0 + e - 1) // share - g0 // share for g0, e in zip(g0s, exts)]
    first = [None] * (n_ctas + 1)
    for c in range((line + share - 1) // share, n_ctas + 1):
        first[c] = len(exts)
    for g, (g0, e) in enumerate(zip(g0s, exts)):
        end, c = g0 + r16(e) + cost, (g0 + share - 1) // share
        while c * share < end and c <= n_ctas:
            assert first[c] is None, "two groups claim one CTA"
            first[c] = g
            c += 1
    return share, g0s, pieces, first


def _cut(exts, n_ctas, share, g0s, first):
    """Every CTA's pieces, as the decode kernel's producer cuts them."""
    out = []
    for b in range(n_ctas):
        lo, hi = b * share, (b + 1) * share

        def piece(g):
            a, e = max(g0s[g], lo), min(g0s[g] + exts[g], hi)
            if a >= e:
                return None
            return g, a - g0s[g], e - g0s[g], 0 if a == g0s[g] else b - g0s[g] // share

        g, p = first[b], None
        if g < len(exts):
            p = piece(g)
            if p is None and g + 1 < len(exts):  # the share starts in the group's padding
                p = piece(g + 1)
        while p is not None:
            out.append(p)
            p = piece(p[0] + 1) if p[0] + 1 < len(exts) else None
    return out


@pytest.mark.parametrize("seed", range(6))
def test_pieces_cover_every_key_once(seed):
    rng = random.Random(seed)
    for _ in range(400):
        n = rng.randint(1, 80)
        exts = [rng.choice([rng.randint(1, 40), rng.randint(1, 5000), rng.randint(500, 9000)]) for _ in range(n)]
        n_ctas = rng.choice([1, 2, 7, 152, 304])
        share, g0s, pieces, first = _plan(exts, n_ctas, rng.choice([STAGE, MIN_SHARE]))
        assert all(v is not None for v in first[:n_ctas])
        cover = [[0] * e for e in exts]
        splits = [set() for _ in exts]
        for g, k0, k1, sp in _cut(exts, n_ctas, share, g0s, first):
            assert 0 <= sp < pieces[g] and sp not in splits[g]
            splits[g].add(sp)
            for k in range(k0, k1):
                cover[g][k] += 1
        for g in range(n):
            assert all(c == 1 for c in cover[g])
            assert splits[g] == set(range(pieces[g]))


def test_decode_workload_shape():
    """64 requests of 512..4096 keys on 152 CTAs: about 976 keys a CTA, ~214 pieces."""
    rng = random.Random(0)
    exts = [rng.randint(512, 4096) for _ in range(64)]
    share, g0s, pieces, first = _plan(exts, 152)
    line = sum((e + STAGE - 1) // STAGE * STAGE + PIECE_COST for e in exts)
    assert share * 152 >= line > share * 151 - share
    assert sum(pieces) <= len(exts) + 152
