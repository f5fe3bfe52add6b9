"""The balanced schedule's split tiles, recomputed from its definition (test
infrastructure only): whole waves run whole; the key blocks of the tiles % G
leftover tiles are cut into C = min(G, rem*n // 8) equal ranges (range i starts
at iteration rem*n*i // C), used only if C > rem and a range is shorter than a
tile by at least max(16, n // 8) blocks."""

MIN_PIECE = 8   # key blocks per CTA range, at least
MIN_GAIN = 16   # key blocks a split must save per CTA, at least


def split_tiles(tiles, n, G):
    """{tile index: [key blocks where the tile is cut]} ({} when nothing is split)."""
    rem = tiles % G
    if rem == 0:
        return {}
    sk = rem * n
    ctas = min(G, sk // MIN_PIECE)
    if ctas <= rem or n - (sk + ctas - 1) // ctas < max(MIN_GAIN, n // 8):
        return {}
    dp = tiles - rem
    out = {}
    for i in range(1, ctas):
        start = sk * i // ctas
        if start % n:
            out.setdefault(dp + start // n, []).append(start % n)
    return out


def tile_rows(tile, B, H, S):
    """(b, first row, last row) of query tile `tile` (tiles numbered b, h, query tile)."""
    n = (S + 127) // 128
    qt = tile % n
    b = tile // (n * H)
    return b, qt * 128, min(qt * 128 + 127, S - 1)
