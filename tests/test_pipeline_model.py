"""CPU checks of the attention kernel's work schedule and of its per-CTA mbarrier
protocol, on host models (`_pipeline_model.py`) of what every role walks.

Schedule: for the shapes the benchmark and the tests launch (and the SM counts
of other parts), every (tile, key block) is covered exactly once, the balanced
schedule splits the tiles its definition says it splits, and every TMA row and
destination row lies inside its tensor.  This includes the single-launch
packed causal schedule whose launch faulted the GPU (75,776 tokens as four
sequences, 40 heads; the library now runs that form as one causal launch per
sequence): its schedule is in range on every CTA.

Protocol: one CTA's producer, S issuer, PV issuer and eight softmax warps run
against phase-counting mbarriers with random timing over the per-CTA piece
sequences of those schedules: no parity alias, no buffer hazard, no deadlock,
for both configurations (D = 128: one Q buffer, 4 ring stages; D = 64: two Q
buffers, 10 stages).  Each planted protocol error (a wait left out, a parity
for the wrong buffer count, P signalled before it is written) is caught.
"""
import random

import pytest

import _pipeline_model as pm
from _schedule import split_tiles

DENSE = [  # B, H, S
    (1, 24, 4608), (1, 12, 32768), (1, 40, 75776), (2, 16, 8192), (2, 16, 131072), (3, 4, 1000), (1, 2, 129),
]
VARLEN = [
    [27916, 12272, 30881, 4707],          # the large video shape's tokens as four sequences
    [500, 12, 700, 300],
    [1, 127, 128, 129, 300, 1000, 3],
    [0, 640, 0, 0, 384],
]


@pytest.mark.parametrize("G", [152, 148, 132])
@pytest.mark.parametrize("B,H,S", DENSE)
def test_dense_schedule_covers_every_block_once(B, H, S, G):
    n = (S + 127) // 128
    tiles = B * H * n
    ranges = {}
    for ps in pm.dense_pieces(tiles, n, G):
        for t, k0, nb in ps:
            assert 0 <= t < tiles and nb >= 1 and 0 <= k0 and k0 + nb <= n
            ranges.setdefault(t, []).append((k0, nb))
            qt = t % n
            assert qt * 128 < S and (k0 + nb - 1) * 128 < S   # first rows of the Q and last K/V boxes
    assert len(ranges) == tiles
    splits = {}
    for t, rs in ranges.items():
        rs.sort()
        pos = 0
        for k0, nb in rs:                                    # the ranges tile [0, n) without overlap
            assert k0 == pos, f"tile {t}: block {pos} missing or covered twice"
            pos = k0 + nb
        assert pos == n
        if len(rs) > 1:
            splits[t] = [k0 for k0, _ in rs[1:]]
    assert splits == {t: sorted(v) for t, v in split_tiles(tiles, n, G).items()}


@pytest.mark.parametrize("head_major", [False, True])
@pytest.mark.parametrize("BH,S", [(24, 4608), (12, 32768), (40, 75776), (4, 1000)])
def test_causal_schedule_longest_first_covers_every_tile_once(BH, S, head_major):
    n_qt = (S + 127) // 128
    G = 152
    seen = set()
    for i, ps in enumerate(pm.causal_pieces(BH, n_qt, G, head_major)):
        for (bh, qt), k0, nb in ps:
            assert (bh, qt) not in seen and 0 <= bh < BH and 0 <= qt < n_qt and k0 == 0 and nb == qt + 1
            seen.add((bh, qt))
    assert len(seen) == BH * n_qt
    if not head_major:
        # each wave holds the longest remaining tiles
        firsts = [ps[0][2] for ps in pm.causal_pieces(BH, n_qt, G, False) if ps]
        assert min(firsts) >= n_qt - (G + BH - 1) // BH


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seqlens", VARLEN, ids=["video_large_tokens", "mix1", "around_tile", "empty_seqs"])
@pytest.mark.parametrize("H,P", [(40, 8), (4, 4)])
def test_varlen_schedule_in_range(seqlens, H, P, causal):
    T = sum(seqlens)
    if T % P:
        pytest.skip("token count not divisible by the shard count")
    G = 152
    Tl = T // P
    seen = set()
    for ps in pm.varlen_pieces(seqlens, H, G, causal):
        for (seq, h, qt), row0, L, nb in ps:
            assert (seq, h, qt) not in seen
            seen.add((seq, h, qt))
            assert 0 <= h < H and L >= 1 and qt * 128 < L and row0 + L <= T
            assert nb == (qt + 1 if causal else (L + 127) // 128)
            assert row0 + qt * 128 < T                      # Q box start
            assert row0 + (nb - 1) * 128 < T                # last K/V box start
            last_row = row0 + min(L, qt * 128 + 128) - 1     # last stored row of the tile
            assert last_row < T and last_row // Tl < P       # destination shard in range
    assert len(seen) == sum((L + 127) // 128 for L in seqlens) * H


def _capped(blocks, cap=7):
    # the protocol does not depend on how long a piece runs past a few blocks
    return [min(n, cap) for n in blocks]


def test_protocol_random_piece_sequences():
    for seed in range(24):
        r = random.Random(seed)
        blocks = [r.choice([1, 1, 2, 3, 4, 5, 9]) for _ in range(r.randint(1, 40))]
        for D in (128, 64):
            pm.run_cta(blocks, D, seed)


@pytest.mark.parametrize("D", [128, 64])
def test_protocol_on_scheduled_pieces(D):
    cases = []
    # the balanced schedule of the large video shape (whole tiles, then parts and heads)
    n = (75776 + 127) // 128
    dense = pm.dense_pieces(40 * n, n, 152)
    cases += [[nb for _, _, nb in dense[i]] for i in (0, 47, 151)]
    # causal image, longest first
    causal = pm.causal_pieces(24, 36, 152, False)
    cases += [[nb for _, _, nb in causal[i]] for i in (0, 100)]
    # the packed causal call that faulted, and its bidirectional form
    for c in (True, False):
        v = pm.varlen_pieces(VARLEN[0], 40, 152, c)
        cases += [[nb for _, _, _, nb in v[i]] for i in (0, 75, 151)]
    for k, blocks in enumerate(cases):
        assert blocks
        pm.run_cta(_capped(blocks), D, seed=k)


@pytest.mark.parametrize("mutation", pm.MUTATIONS)
@pytest.mark.parametrize("D", [128, 64])
def test_protocol_model_catches_planted_errors(mutation, D):
    r = random.Random(1)
    blocks = [r.choice([1, 1, 2, 3, 4, 5, 9]) for _ in range(30)]
    with pytest.raises(pm.ProtocolError):
        for seed in range(4):
            pm.run_cta(blocks, D, seed, mutate=mutation)
