"""Host-side model of the stream-K work split of the CTA-pair GEMM kernel.

The kernel gives pair c the K iterations [U*c/P, U*(c+1)/P) of the
U = tiles x K-blocks total, cut at tile boundaries; the pair holding a tile's
first K block finishes it after adding the fp32 partials that the following
pairs (those whose shares start before the tile ends) write from their first
segments.  These checks pin the properties the device code relies on: every
K iteration is computed exactly once, no pair has an empty share (the host
launches min(P, U) pairs), only a pair's first segment can start inside a
tile, and a tile's owner waits exactly on the pairs that hold the rest of it,
each of which reaches that work first, before any wait of its own.
"""
import pytest


def segments(T, KB, P):
    U = T * KB
    out = []
    for c in range(P):
        u, ue = U * c // P, U * (c + 1) // P
        ss = []
        while u < ue:
            t, k0 = u // KB, u % KB
            k1 = min(KB, k0 + (ue - u))
            ss.append((t, k0, k1))
            u += k1 - k0
        out.append(ss)
    return out


def contributors(T, KB, P, pair, tile):
    U, te, n, c = T * KB, (tile + 1) * KB, 0, pair + 1
    while c < P and U * c // P < te:
        n += 1
        c += 1
    return n


@pytest.mark.parametrize("T", [1, 2, 3, 5, 60, 75, 76, 77, 150, 1000])
@pytest.mark.parametrize("KB", [1, 2, 3, 8, 13, 64, 216])
@pytest.mark.parametrize("pairs", [1, 2, 7, 76])
def test_stream_k_schedule(T, KB, pairs):
    P = min(pairs, T * KB)
    S = segments(T, KB, P)
    cover = {}
    for c, ss in enumerate(S):
        assert ss, "empty share"
        for i, (t, k0, k1) in enumerate(ss):
            if k0 != 0:
                assert i == 0
            if k1 != KB:
                assert i == len(ss) - 1
            for k in range(k0, k1):
                cover[(t, k)] = cover.get((t, k), 0) + 1
            if k0 == 0 and k1 < KB:
                got = set()
                for e in range(contributors(T, KB, P, c, t)):
                    t2, a2, b2 = S[c + 1 + e][0]
                    assert t2 == t and a2 != 0
                    got.update(range(a2, b2))
                assert got == set(range(k1, KB))
    assert all(cover.get((t, k)) == 1 for t in range(T) for k in range(KB))
