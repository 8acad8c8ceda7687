"""Pins of the index-map oracle (partitions, ring schedule, tile classes) against
the counts and orders the pages print, and against brute force (no GPU)."""
import numpy as np
import pytest

import oracle
from tests.conftest import golden


def causal_pairs(tokens):
    # causal: token t sees keys 0..t, i.e. t + 1 pairs
    return int(sum(t + 1 for t in tokens))


def test_pair_counts_printed_on_the_page():
    g = golden("causal_pair_counts.json")
    for kind in ("contiguous", "zigzag"):
        tok = oracle.partition(g["T"], g["P"], kind)
        owned = [sorted(r.tolist()) for r in tok]
        assert owned == g[kind]["owned"]
        pairs = []
        for r in range(g["P"]):
            n = 0
            for i in tok[r]:
                for j in range(g["T"]):
                    n += oracle.is_visible(0, int(i), j, True, None, None)
            pairs.append(n)
        assert pairs == g[kind]["pairs"]
        assert pairs == [causal_pairs(r) for r in tok]


def test_ring_order_printed_on_the_page():
    g = golden("ring_order.json")
    src = oracle.schedule(g["P"])
    assert src[0].tolist() == g["gpu0_block_order"]
    tok = oracle.partition(g["T"], g["P"], "contiguous")
    assert [tok[s].tolist() for s in src[0]] == g["gpu0_tokens_per_step"]
    assert src.shape[1] == g["steps"]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_schedule_every_rank_sees_every_block_once_and_passes_to_next(P):
    src = oracle.schedule(P)
    for r in range(P):
        assert sorted(src[r].tolist()) == list(range(P))
        assert src[r, 0] == r  # local block first
    # the block rank r holds at step s+1 is the one rank r-1 held at step s
    for s in range(P - 1):
        for r in range(P):
            assert src[r, s + 1] == src[(r - 1) % P, s]


@pytest.mark.parametrize("T,P,kind", [(8, 4, "contiguous"), (1024, 4, "contiguous"), (8192, 8, "zigzag"),
                                      (65536, 16, "zigzag"), (512, 2, "contiguous"), (96, 3, "zigzag")])
def test_partitions_are_permutations(T, P, kind):
    tok = oracle.partition(T, P, kind)
    assert tok.shape == (P, T // P)
    assert np.array_equal(np.sort(tok.reshape(-1)), np.arange(T))
    if kind == "zigzag":
        c = T // (2 * P)
        pairs = [causal_pairs(r) for r in tok]
        assert len(set(pairs)) == 1  # exactly balanced causal work
        assert tok[0, 0] == 0 and tok[0, -1] == T - 1 and tok[P - 1, 0] == (P - 1) * c


def test_zigzag_balance_at_8k():
    tok = oracle.partition(8192, 8, "zigzag")
    assert [causal_pairs(r) for r in tok] == [4194816] * 8
    cont = oracle.partition(8192, 8, "contiguous")
    cp = [causal_pairs(r) for r in cont]
    assert cp[0] == 524800 and cp[-1] == 7864832


def test_tile_classes_hand_worked():
    # causal over 256 tokens in 128-tiles: diagonal tiles partial, upper empty, lower full
    cls = oracle.tile_classes(1, 256, 256, causal=True)
    P_, E, F = oracle.PARTIAL, oracle.EMPTY, oracle.FULL
    assert cls[0].tolist() == [[P_, E], [F, P_]]
    # keys padded from 100 on: the second key tile is empty, the first partial
    kpm = np.zeros((1, 256), np.uint8)
    kpm[0, 100:] = 1
    cls = oracle.tile_classes(1, 256, 256, kpm=kpm)
    assert cls[0].tolist() == [[P_, E], [P_, E]]
    # a block at an offset: rows 128..255 against keys 0..127 under causal is full
    cls = oracle.tile_classes(1, 128, 128, q_off=128, k_off=0, causal=True)
    assert cls[0].tolist() == [[F]]
    cls = oracle.tile_classes(1, 128, 128, q_off=0, k_off=128, causal=True)
    assert cls[0].tolist() == [[E]]


def test_tile_classes_match_vectorised_recount():
    rng = np.random.default_rng(0)
    B, L, S, tile = 2, 70, 90, 16
    kpm = (rng.random((B, S + 5)) < 0.2).astype(np.uint8)
    am = (rng.random((L + 3, S + 5)) < 0.5).astype(np.uint8)
    am[:, 40:56] = 1   # a fully forbidden key band -> EMPTY tiles
    am[0:16, 0:16] = 0
    for causal in (False, True):
        cls = oracle.tile_classes(B, L, S, q_off=3, k_off=5, causal=causal, kpm=kpm, am=am, tile=tile)
        i = np.arange(L)[:, None] + 3
        j = np.arange(S)[None, :] + 5
        for b in range(B):
            excl = am[i, j].astype(bool) | kpm[b, j].astype(bool)
            if causal:
                excl |= j > i
            vis = ~excl
            for qt in range(cls.shape[1]):
                for kt in range(cls.shape[2]):
                    blk = vis[qt * tile:(qt + 1) * tile, kt * tile:(kt + 1) * tile]
                    want = oracle.EMPTY if not blk.any() else (oracle.FULL if blk.all() else oracle.PARTIAL)
                    assert cls[b, qt, kt] == want


def test_striped_partition_brute_force_counts():
    """Striped (round-robin) partition of T=8 over P=2: rank 0 holds the even
    tokens, rank 1 the odd ones; causal pair counts by brute force are 16 / 20,
    between contiguous (10 / 26) and zigzag (18 / 18)."""
    tok = oracle.partition(8, 2, "striped")
    assert tok.tolist() == [[0, 2, 4, 6], [1, 3, 5, 7]]
    pairs = [sum(oracle.is_visible(0, int(i), j, True, None, None) for i in r for j in range(8)) for r in tok]
    assert pairs == [16, 20]
    # at 8K over 8 ranks the spread is one row's worth per rank step: max/min < 1.002
    tok = oracle.partition(8192, 8, "striped")
    p = [causal_pairs(r) for r in tok]
    assert sorted(np.concatenate(tok).tolist()) == list(range(8192))
    assert max(p) / min(p) < 1.002
