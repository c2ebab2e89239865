"""The split schedule's partition, restated on the host and checked exhaustively.

`Schedule` in csrc/attention.cuh cuts the stream-K tail into equal-cost
ranges: every unit counts as kSegCost "segment start" slots followed by its
n_kv key tiles, and the virtual space is cut evenly among the G CTAs.  The
kernel's merge of a cut unit relies on these properties, checked here for
many unit counts, grids and tile counts:
  * every tail key tile belongs to exactly one CTA;
  * every CTA range holds at least n_kv key tiles;
  * a unit is cut into at most two pieces, the last segment of CTA c and the
    first segment of CTA c + 1, and the first piece starts at key tile 0;
  * cta_of(first tile of a unit) is the CTA holding it, and that CTA's
    piece is its first segment exactly when its range starts at the unit.
"""
import re
from pathlib import Path

import pytest

SRC = Path(__file__).resolve().parents[1] / "relative_position_bias_gb300" / "csrc" / "attention.cuh"


def seg_cost() -> int:
    m = re.search(r"static constexpr int kSegCost = (\d+);", SRC.read_text())
    assert m, "kSegCost not found"
    return int(m.group(1))


def partition(U: int, G: int, n_kv: int, seg: int):
    dp = max(U // G - 1, 0)
    sk = dp * G * n_kv
    per = n_kv + seg
    V = (U - dp * G) * per

    def real_of(v):
        u, o = divmod(v, per)
        return u * n_kv + max(0, o - seg)

    def begin(c):
        return sk + real_of(c * V // G)

    def cta_of(t):
        tr = t - sk
        u = tr // n_kv
        v = u * per + seg + (tr - u * n_kv)
        c = min(G - 1, v * G // V)
        while c + 1 < G and begin(c + 1) <= t:
            c += 1
        while c > 0 and begin(c) > t:
            c -= 1
        return c

    return dp, sk, begin, cta_of


@pytest.mark.parametrize("n_kv", [1, 2, 3, 5, 8, 14, 16, 20, 22, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 3, 7, 148, 152])
def test_tail_partition(n_kv, G):
    seg = seg_cost()
    for U in list(range(G + 1, 3 * G + 3)) + [10 * G + 7]:
        if U % G == 0:
            continue  # whole waves are not split
        dp, sk, begin, cta_of = partition(U, G, n_kv, seg)
        owner, pieces = {}, {}
        for c in range(G):
            it, end, tail = begin(c), begin(c + 1), 0
            assert end - it >= n_kv
            while it < end:
                u = it // n_kv
                j0 = it - u * n_kv
                j1 = min(n_kv, j0 + (end - it))
                for t in range(it, u * n_kv + j1):
                    assert t not in owner
                    owner[t] = c
                pieces.setdefault(u, []).append((c, j0, j1, tail))
                tail += 1
                it += j1 - j0
        assert set(owner) == set(range(sk, U * n_kv))
        for u in range(dp * G, U):
            ps, u0 = pieces[u], u * n_kv
            assert len(ps) <= 2
            assert cta_of(u0) == ps[0][0]
            if len(ps) == 2:
                (c0, a0, b0, t0), (c1, a1, b1, t1) = ps
                assert c1 == c0 + 1 and t1 == 0 and a0 == 0 and b1 == n_kv and b0 == a1
                assert (t0 == 0) == (begin(c0) == u0)


@pytest.mark.parametrize("G", [1, 2, 3, 7, 148, 152])
def test_round_robin_without_cuts(G):
    """Without cuts (no workspace, or units shorter than 4 key tiles) CTA c of G runs the whole
    units c, c + G, c + 2G, ... below U: every unit exactly once, in ceil(U / G) rounds."""
    for U in list(range(1, 3 * G + 3)) + [10 * G + 7]:
        rounds = -(-U // G)
        seen = []
        for c in range(G):
            mine = [r * G + c for r in range(rounds) if r * G + c < U]
            assert len(mine) in (rounds - 1, rounds) or U < G
            seen.extend(mine)
        assert sorted(seen) == list(range(U))
