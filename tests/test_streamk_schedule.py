"""Host-side model of the stream-K work split of the CTA-pair GEMM kernel.

The launch uses G groups of MB pairs (MB = number of 256-row M blocks,
G = min(floor(pairs / MB), V)); pair m of group g works on M block m.  The
V = N-tiles x K-blocks column iterations are split evenly over the groups
(group g: [V*g/G, V*(g+1)/G), cut at N-tile boundaries), so the pairs of a
group read the same W slices at the same time.  The pair holding a tile's
first K block finishes the tile after adding the fp32 partials that the same
M block's pairs in the following groups (those whose shares start before the
N-tile ends) write from their first segments.  These checks pin what the
device code relies on: every (tile, K block) is computed exactly once, no pair
has an empty share, only a pair's first segment can start inside a tile, and a
tile's owner waits exactly on the pairs holding the rest of it, each of which
reaches that work first, before any wait of its own.
"""
import pytest


def plan(MB, NB, KB, pairs):
    V = NB * KB
    G = min(pairs // MB, V) if MB <= pairs else 0
    return G


def segments(MB, NB, KB, G):
    V = NB * KB
    out = {}
    for g in range(G):
        for m in range(MB):
            v, ve = V * g // G, V * (g + 1) // G
            ss = []
            while v < ve:
                nb, k0 = v // KB, v % KB
                k1 = min(KB, k0 + (ve - v))
                ss.append((m + nb * MB, k0, k1))
                v += k1 - k0
            out[g * MB + m] = ss
    return out


def contributors(MB, NB, KB, G, pair, tile):
    V, te, n = NB * KB, (tile // MB + 1) * KB, 0
    g = pair // MB + 1
    while g < G and V * g // G < te:
        n += 1
        g += 1
    return n


@pytest.mark.parametrize("MB", [1, 2, 3, 4, 16])
@pytest.mark.parametrize("NB", [1, 2, 5, 20, 77])
@pytest.mark.parametrize("KB", [1, 2, 8, 13, 216])
@pytest.mark.parametrize("pairs", [1, 3, 7, 76])
def test_stream_k_schedule(MB, NB, KB, pairs):
    G = plan(MB, NB, KB, pairs)
    if G == 0:
        return
    S = segments(MB, NB, KB, G)
    cover = {}
    for pair, ss in S.items():
        assert ss, "empty share"
        m = pair % MB
        for i, (t, k0, k1) in enumerate(ss):
            assert t % MB == m
            if k0 != 0:
                assert i == 0
            if k1 != KB:
                assert i == len(ss) - 1
            for k in range(k0, k1):
                cover[(t, k)] = cover.get((t, k), 0) + 1
            if k0 == 0 and k1 < KB:
                first = (pair // MB + 1) * MB + m
                got = set()
                for e in range(contributors(MB, NB, KB, G, pair, t)):
                    t2, a2, b2 = S[first + e * MB][0]
                    assert t2 == t and a2 != 0
                    got.update(range(a2, b2))
                assert got == set(range(k1, KB))
    assert all(cover.get((t, k)) == 1 for t in range(MB * NB) for k in range(KB))
