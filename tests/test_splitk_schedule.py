"""Host-side model of the decode path's stream-K split (no GPU needed).

The split-K GEMM deals the (m-tile, K-block) units of a call out to G CTAs
in contiguous ranges [c*U/G, (c+1)*U/G); each CTA writes one fp32 partial
tile per m-tile it touches, into slot (its index - the index of the m-tile's
first CTA); the reducer sums an m-tile's slots in slot order.  The kernels
find "which CTA owns unit u" with a closed form in 32-bit arithmetic, which
the host allows only while (U + 1) * G + U < 2^32.  This model checks the
closed form against the ranges, that the ranges cover every unit once, and
that the slot indices of each m-tile are 0..n-1 without gaps (so the
reducer's fixed-order sum reads exactly the slots that were written).
"""
import random


def owner_closed_form(u, U, G):
    assert (U + 1) * G + U < 2 ** 32
    return ((u + 1) * G + U - 1) // U - 1


def owner_by_ranges(U, G):
    own = [None] * U
    for c in range(G):
        for u in range(c * U // G, (c + 1) * U // G):
            assert own[u] is None
            own[u] = c
    assert None not in own
    return own


def test_closed_form_matches_the_ranges():
    rng = random.Random(7)
    cases = [(U, G) for U in range(1, 200) for G in range(1, min(U, 160) + 1)]
    cases += [(rng.randint(1000, 200000), rng.randint(1, 152)) for _ in range(60)]
    for U, G in cases:
        own = owner_by_ranges(U, G)
        for u in (range(U) if U <= 5000 else rng.sample(range(U), 3000)):
            assert owner_closed_form(u, U, G) == own[u], (u, U, G)


def slots_per_m_tile(m_tiles, kb, G):
    U = m_tiles * kb
    out = []
    for m in range(m_tiles):
        first = owner_closed_form(m * kb, U, G)
        ctas = sorted({owner_closed_form(u, U, G) for u in range(m * kb, (m + 1) * kb)})
        out.append([c - first for c in ctas])
    return out


def test_slots_are_dense_from_zero():
    # 70B o_proj (64 m-tiles x 128 K-blocks) and down_proj (64 x 448) on 152 CTAs, and small shapes
    for m_tiles, kb, G in [(64, 128, 152), (64, 448, 152), (32, 224, 152), (1, 300, 16), (3, 7, 20), (65, 128, 152)]:
        G = min(G, m_tiles * kb)
        for slots in slots_per_m_tile(m_tiles, kb, G):
            assert slots == list(range(len(slots)))
        assert max(len(s) for s in slots_per_m_tile(m_tiles, kb, G)) <= 16
